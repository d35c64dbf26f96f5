// moe.cu -- the routed-expert block.
//
// Per routed (row s, slot k) with expert e = ids[s][k] >= 0 and weight w[s][k]
// (colibri-strix commit log, "metal: batched moe_block": gate/up -> silu ->
// down for a whole expert block, per-row ragged routing, weighted
// scatter-add of the expert outputs):
//   h = silu(G_e x[s]) * (U_e x[s]);   y[s] += w[s][k] * D_e h.
//
// Decode (S*K <= 64): ONE cooperative launch.
//   phase 0  every CTA reads ids/w and forms the same routing inversion in
//            shared memory (stable sort of the slots by expert id);
//   phase A  warps stream gate/up row pairs (j of expert e) once each and
//            compute h for every slot routed to e, into a scratch buffer;
//   wait     one grid-wide barrier, bounded in time (on expiry the kernel
//            records DEV_ERR_TIMEOUT and returns);
//   phase B  each CTA owns a block of output rows; its warps stream the down
//            rows of every routed expert for those rows against h (staged in
//            shared memory) and the CTA sums the weighted slot results in
//            ascending slot order, so y is written once, without atomics, and
//            the result does not depend on timing.
//
// Prefill (larger S*K): routing inversion on the device, then the grouped
// GEMMs (tiled-gemm kernels) and a deterministic combine.
#include "coli_internal.cuh"

namespace coli {

namespace {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ bool grid_barrier(unsigned *bar, int *err, long long timeout_ns) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        const unsigned gen = ld_acquire(bar + 1);
        __threadfence();
        const unsigned prev = atomicAdd(bar, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = global_ns();
            while (ld_acquire(bar + 1) == gen) {
                if ((long long)(global_ns() - t0) > timeout_ns) {
                    atomicCAS(err, 0, DEV_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
                __nanosleep(100);
            }
        }
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

template <int FMT, int NS>
__device__ __forceinline__ void phase_a_item(const MatDesc &G, const MatDesc &U, int j, const float *xs,
                                             int xlen, const int *s_order, int p0, int K, int cpr, int lane,
                                             float *hbuf, int F) {
    const uint8_t *rows[2] = {G.q + (size_t)j * G.rs, U.q + (size_t)j * U.rs};
    const float *scl[2] = {row_scales(FMT, G, j), row_scales(FMT, U, j)};
    const int gpc[2] = {chunks_per_group(FMT, G.gs), chunks_per_group(FMT, U.gs)};
    const float *xsv[NS];
#pragma unroll
    for (int n = 0; n < NS; n++) xsv[n] = xs + (size_t)(s_order[p0 + n] / K) * xlen;
    float out[2][NS];
    dot_rows<FMT, 2, NS>(rows, scl, gpc, xsv, cpr, lane, out);
#pragma unroll
    for (int n = 0; n < NS; n++)
        if (lane == n) hbuf[(size_t)(p0 + n) * F + j] = silu_f(out[0][n]) * out[1][n];
}

template <int FMT, int NS, int RB>
__device__ __forceinline__ void phase_b_item(const MatDesc &D, int o0, int H, const float *hs, int xlen,
                                             int prel, const float *s_w, const int *s_order, int p0, int cpr,
                                             int lane, float *ypart, int rpc, int orel) {
    const uint8_t *rows[RB];
    const float *scl[RB];
    int gpc[RB];
#pragma unroll
    for (int r = 0; r < RB; r++) {
        const int o = min(o0 + r, H - 1);
        rows[r] = D.q + (size_t)o * D.rs;
        scl[r] = row_scales(FMT, D, o);
        gpc[r] = chunks_per_group(FMT, D.gs);
    }
    const float *xsv[NS];
#pragma unroll
    for (int n = 0; n < NS; n++) xsv[n] = hs + (size_t)(prel + n) * xlen;
    float out[RB][NS];
    dot_rows<FMT, RB, NS>(rows, scl, gpc, xsv, cpr, lane, out);
    if (lane == 0) {
#pragma unroll
        for (int n = 0; n < NS; n++) {
            const float wk = s_w[s_order[p0 + n]];
#pragma unroll
            for (int r = 0; r < RB; r++)
                if (o0 + r < H && orel + r < rpc) ypart[(size_t)(prel + n) * rpc + orel + r] = wk * out[r][n];
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kDecodeThreads, 2) moe_decode_kernel(const MoeDecodeArgs a) {
    extern __shared__ float4 smem4[];
    float *stage = reinterpret_cast<float *>(smem4);
    __shared__ int s_ids[kMaxDecodeSlots];
    __shared__ float s_w[kMaxDecodeSlots];
    __shared__ int s_order[kMaxDecodeSlots];
    __shared__ int s_seg[kMaxDecodeSlots + 1];
    __shared__ int s_exp[kMaxDecodeSlots];
    __shared__ int s_nact, s_nvalid, s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int n = a.S * a.K;

    // ---- phase 0: routing inversion (identical in every CTA)
    if (tid == 0) s_bad = 0;
    __syncthreads();
    if (tid < n) {
        const int e = a.ids[tid];
        s_ids[tid] = e;
        s_w[tid] = a.w[tid];
        if (e < -1 || e >= a.n_experts) atomicOr(&s_bad, 1);
    }
    __syncthreads();
    if (s_bad) {
        if (blockIdx.x == 0 && tid == 0) atomicCAS(a.err, 0, DEV_ERR_BAD_ID);
        return;
    }
    if (tid < n) {
        const int e = s_ids[tid];
        if (e >= 0) {
            int r = 0;
            for (int t = 0; t < n; t++) {
                const int f = s_ids[t];
                r += (f >= 0) && (f < e || (f == e && t < tid));
            }
            s_order[r] = tid;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int nv = 0;
        for (int t = 0; t < n; t++) nv += s_ids[t] >= 0;
        int na = 0;
        for (int p = 0; p < nv; p++) {
            const int e = s_ids[s_order[p]];
            if (p == 0 || e != s_ids[s_order[p - 1]]) {
                s_exp[na] = e;
                s_seg[na] = p;
                na++;
            }
        }
        s_seg[na] = nv;
        s_nact = na;
        s_nvalid = nv;
    }
    __syncthreads();
    const int nact = s_nact, nvalid = s_nvalid;

    // ---- phase A: h = silu(G x) * (U x) for every routed slot
    const int xlen_gu = staged_len(FMT, a.cpr_gu);
    for (int s = 0; s < a.S; s++)
        stage_vec<FMT>(stage + (size_t)s * xlen_gu, a.x + (size_t)s * a.H, a.H, xlen_gu, tid, blockDim.x);
    __syncthreads();
    {
        const long long items = (long long)nact * a.F;
        for (long long it = (long long)blockIdx.x * nwarps + warp; it < items;
             it += (long long)gridDim.x * nwarps) {
            const int ai = (int)(it / a.F), j = (int)(it - (long long)ai * a.F);
            const ExpertDesc &E = a.table[s_exp[ai]];
            for (int p0 = s_seg[ai]; p0 < s_seg[ai + 1]; p0 += 2) {
                if (s_seg[ai + 1] - p0 == 1)
                    phase_a_item<FMT, 1>(E.m[0], E.m[1], j, stage, xlen_gu, s_order, p0, a.K, a.cpr_gu, lane, a.hbuf, a.F);
                else
                    phase_a_item<FMT, 2>(E.m[0], E.m[1], j, stage, xlen_gu, s_order, p0, a.K, a.cpr_gu, lane, a.hbuf, a.F);
            }
        }
    }

    // ---- grid-wide wait: every h must be written before phase B reads it
    if (!grid_barrier(a.bar, a.err, a.timeout_ns)) return;

    // ---- phase B: y rows [oc0, oc1) of this CTA
    const int xlen_d = staged_len(FMT, a.cpr_d);
    const int rpc = a.rpc;
    const int oc0 = blockIdx.x * rpc;
    const int oc1 = min(a.H, oc0 + rpc);
    float *ypart = stage + (size_t)a.sb * xlen_d;   // [sb][rpc]
    float *yacc = ypart + (size_t)a.sb * rpc;       // [S][rpc]
    for (int t = tid; t < a.S * rpc; t += blockDim.x) yacc[t] = 0.f;
    if (oc0 < oc1) {
        const int nrb = (oc1 - oc0 + 1) / 2;
        for (int b0 = 0; b0 < nvalid; b0 += a.sb) {
            const int b1 = min(nvalid, b0 + a.sb);
            __syncthreads();
            if (xlen_d == a.F) {   // contiguous unpadded rows: one staging pass for the batch
                stage_vec<FMT>(stage, a.hbuf + (size_t)b0 * a.F, (b1 - b0) * a.F, (b1 - b0) * xlen_d, tid, blockDim.x);
            } else {
                for (int p = b0; p < b1; p++)
                    stage_vec<FMT>(stage + (size_t)(p - b0) * xlen_d, a.hbuf + (size_t)p * a.F, a.F, xlen_d, tid,
                                   blockDim.x);
            }
            __syncthreads();
            // experts intersecting [b0, b1)
            int a_lo = 0;
            while (a_lo < nact && s_seg[a_lo + 1] <= b0) a_lo++;
            int a_hi = a_lo;
            while (a_hi < nact && s_seg[a_hi] < b1) a_hi++;
            const int items = (a_hi - a_lo) * nrb;
            for (int it = warp; it < items; it += nwarps) {
                const int ai = a_lo + it / nrb;
                const int rb = it - (it / nrb) * nrb;
                const MatDesc &D = a.table[s_exp[ai]].m[2];
                const int q0 = max(s_seg[ai], b0), q1 = min(s_seg[ai + 1], b1);
                const int o0 = oc0 + rb * 2;
                for (int p0 = q0; p0 < q1; p0 += 2) {
                    if (q1 - p0 == 1)
                        phase_b_item<FMT, 1, 2>(D, o0, a.H, stage, xlen_d, p0 - b0, s_w, s_order, p0, a.cpr_d, lane, ypart, rpc, o0 - oc0);
                    else
                        phase_b_item<FMT, 2, 2>(D, o0, a.H, stage, xlen_d, p0 - b0, s_w, s_order, p0, a.cpr_d, lane, ypart, rpc, o0 - oc0);
                }
            }
            __syncthreads();
            // ordered sum of this batch's slot results into yacc
            for (int t = tid; t < a.S * rpc; t += blockDim.x) {
                const int s = t / rpc, rr = t - s * rpc;
                if (oc0 + rr >= oc1) continue;
                float acc = yacc[t];
                for (int p = b0; p < b1; p++)
                    if (s_order[p] / a.K == s) acc += ypart[(size_t)(p - b0) * rpc + rr];
                yacc[t] = acc;
            }
        }
        __syncthreads();
        for (int t = tid; t < a.S * rpc; t += blockDim.x) {
            const int s = t / rpc, rr = t - s * rpc;
            if (oc0 + rr < oc1) a.y[(size_t)s * a.H + oc0 + rr] = yacc[t];
        }
    }
}

// ------------------------------------------------------------ routing
constexpr int kRouteThreads = 1024;
constexpr int kRouteWarpHistE = 256;   // up to this many experts: placement by all warps (per-warp histograms)

// Block-wide exclusive scan of one value per thread (blockDim.x = kRouteThreads);
// *total: the sum over the block.  Contains __syncthreads.
__device__ __forceinline__ int route_block_excl(int v, int *s_part, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x / 32) ? s_part[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        s_part[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int ex = incl - v + (warp > 0 ? s_part[warp - 1] : 0);
    *total = s_part[blockDim.x / 32 - 1];
    __syncthreads();   // s_part may be reused
    return ex;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteArgs a) {
    extern __shared__ int rsm[];
    int *cnt = rsm;                // [E]
    int *base = rsm + a.E;         // [E+1]
    int *fill = base + a.E + 1;    // [E]
    int *hist = fill + a.E;        // [32][E] when E <= kRouteWarpHistE
    __shared__ int s_bad;
    __shared__ int s_part[kRouteThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.S * a.K;
    if (tid == 0) s_bad = 0;
    for (int e = tid; e < a.E; e += blockDim.x) cnt[e] = 0, fill[e] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += blockDim.x) {
        const int e = a.ids[t];
        if (e < -1 || e >= a.E) atomicOr(&s_bad, 1);
        else if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            atomicCAS(a.err, 0, DEV_ERR_BAD_ID);
            if (a.n_tiles) *a.n_tiles = 0;
            if (a.n_sg) *a.n_sg = 0;
        }
        for (int e = tid; e <= a.E; e += blockDim.x) a.offsets[e] = 0;
        for (int t = tid; t < n && a.inv; t += blockDim.x) a.inv[t] = -1;
        return;
    }
    // exclusive scan of cnt -> base (block-wide, chunked per thread)
    const int per = (a.E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(a.E, tid * per), e1 = min(a.E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; e++) local += cnt[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < (int)(blockDim.x / 32) ? s_part[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        s_part[lane] = v;   // inclusive over warps
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? s_part[warp - 1] : 0);
    for (int e = e0; e < e1; e++) {
        base[e] = run;
        run += cnt[e];
    }
    if (tid == blockDim.x - 1) base[a.E] = run;
    __syncthreads();
    for (int e = tid; e <= a.E; e += blockDim.x) a.offsets[e] = base[e];
    // stable placement (rows of an expert in slot order).  Up to
    // kRouteWarpHistE experts: warp w takes the w-th of 32 equal slot ranges,
    // counts its slots per expert, and places them after the earlier warps'
    // ones; else warp 0 alone, 32 slots at a time.
    const bool par = a.E <= kRouteWarpHistE;
    const int span = par ? ((n + 31) / 32 + 31) / 32 * 32 : n;
    const int t_lo = par ? min(n, warp * span) : 0, t_hi = par ? min(n, t_lo + span) : n;
    int *wfill = par ? hist + warp * a.E : fill;
    if (par) {
        for (int i = tid; i < 32 * a.E; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
            const int t = t0 + lane;
            const int e = t < t_hi ? a.ids[t] : -2;
            const unsigned grp = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && __popc(grp & ((1u << lane) - 1u)) == 0) wfill[e] += __popc(grp);
            __syncwarp();
        }
        __syncthreads();
        for (int e = tid; e < a.E; e += blockDim.x) {
            int run = base[e];
            for (int w = 0; w < 32; w++) {
                const int c = hist[w * a.E + e];
                hist[w * a.E + e] = run;
                run += c;
            }
        }
        __syncthreads();
    }
    if (par || warp == 0) {
        for (int t0 = t_lo; t0 < t_hi; t0 += 32) {
            const int t = t0 + lane;
            const int e = t < t_hi ? a.ids[t] : -2;
            const unsigned grp = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(grp & ((1u << lane) - 1u));
            int pos = -1;
            if (e >= 0) pos = (par ? wfill[e] : base[e] + wfill[e]) + rank;
            __syncwarp();
            if (e >= 0) {
                a.order[pos] = t;
                if (rank == 0) wfill[e] += __popc(grp);
            }
            if (t < t_hi && a.inv) a.inv[t] = pos;
            __syncwarp();
        }
    }
    // tile list: ceil(count / tile_rows) tiles per expert, in expert order;
    // experts of at most small_rows rows: groups of up to 4 rows instead.  Each
    // thread writes the entries of its own range of experts.
    if (a.n_tiles) {
        __syncthreads();
        int lt = 0, lg = 0;
        for (int e = e0; e < e1; e++) {
            const int c = base[e + 1] - base[e];
            const bool sm = c > 0 && c <= a.small_rows;
            lt += sm ? 0 : (c + a.tile_rows - 1) / a.tile_rows;
            lg += sm ? (c + 3) / 4 : 0;
        }
        int tot_t = 0, tot_g = 0;
        int nt = route_block_excl(lt, s_part, &tot_t);
        int ng = route_block_excl(lg, s_part, &tot_g);
        for (int e = e0; e < e1; e++) {
            const int c = base[e + 1] - base[e];
            if (c > 0 && c <= a.small_rows) {
                for (int p = base[e]; p < base[e + 1]; p += 4) {
                    a.sg_e[ng] = e;
                    a.sg_p0[ng] = p;
                    a.sg_n[ng] = min(4, base[e + 1] - p);
                    ng++;
                }
                continue;
            }
            for (int p = base[e]; p < base[e + 1]; p += a.tile_rows) {
                a.tile_e[nt] = e;
                a.tile_p0[nt] = p;
                a.tile_p1[nt] = min(base[e + 1], p + a.tile_rows);
                nt++;
            }
        }
        if (tid == 0) {
            *a.n_tiles = tot_t;
            if (a.n_sg) *a.n_sg = tot_g;
        }
        if (a.row_small)
            for (int e = tid; e < a.E; e += blockDim.x) {
                const int c = base[e + 1] - base[e];
                const uint8_t f = (c > 0 && c <= a.small_rows) ? 1 : 0;
                for (int p = base[e]; p < base[e + 1]; p++) a.row_small[p] = f;
            }
    }
}

// ------------------------------------------------------------ combine
// y[s][o] = sum_k w[s][k] * slot_out[inv[s*K+k]][o], k ascending.
__global__ void combine_kernel(const float *slot_out, const int32_t *inv, const float *w, int S, int K, int H,
                               float *y) {
    const int s = blockIdx.y;
    for (int o = blockIdx.x * blockDim.x + threadIdx.x; o < H; o += gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int k = 0; k < K; k++) {
            const int p = inv[s * K + k];
            if (p >= 0) acc = fmaf(w[s * K + k], slot_out[(size_t)p * H + o], acc);
        }
        y[(size_t)s * H + o] = acc;
    }
}

__global__ void fmt1_encode_kernel(uint8_t *q, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        q[i] ^= 0x80;
}

template <int FMT>
cudaError_t launch_decode_t(const MoeDecodeArgs &a, int grid, size_t smem, cudaStream_t st) {
    auto kern = moe_decode_kernel<FMT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT>
cudaError_t occ_t(size_t smem, int *per_sm) {
    auto kern = moe_decode_kernel<FMT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, kDecodeThreads, smem);
}

}  // namespace

cudaError_t moe_decode_occupancy(int fmt, size_t smem, int *per_sm) {
    switch (fmt) {
    case 0: return occ_t<0>(smem, per_sm);
    case 1: return occ_t<1>(smem, per_sm);
    case 2: return occ_t<2>(smem, per_sm);
    case 3: return occ_t<3>(smem, per_sm);
    case 4: return occ_t<4>(smem, per_sm);
    case 7: return occ_t<7>(smem, per_sm);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_moe_decode(const MoeDecodeArgs &a, int fmt, int grid, size_t smem, cudaStream_t st) {
    switch (fmt) {
    case 0: return launch_decode_t<0>(a, grid, smem, st);
    case 1: return launch_decode_t<1>(a, grid, smem, st);
    case 2: return launch_decode_t<2>(a, grid, smem, st);
    case 3: return launch_decode_t<3>(a, grid, smem, st);
    case 4: return launch_decode_t<4>(a, grid, smem, st);
    case 7: return launch_decode_t<7>(a, grid, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_route(const RouteArgs &a, cudaStream_t st) {
    const size_t smem = (size_t)(3 * a.E + 1 + (a.E <= kRouteWarpHistE ? 32 * a.E : 0)) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    route_kernel<<<1, kRouteThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *slot_out, const int32_t *inv, const float *w, int S, int K, int H,
                           float *y, cudaStream_t st) {
    dim3 grid((H + 255) / 256, S);
    combine_kernel<<<grid, 256, 0, st>>>(slot_out, inv, w, S, K, H, y);
    return cudaGetLastError();
}

cudaError_t launch_fmt1_encode(uint8_t *q, long long n, cudaStream_t st) {
    const long long g = (n + 255) / 256;
    const int grid = (int)(g < 4096 ? g : 4096);
    fmt1_encode_kernel<<<grid, 256, 0, st>>>(q, n);
    return cudaGetLastError();
}

}  // namespace coli
