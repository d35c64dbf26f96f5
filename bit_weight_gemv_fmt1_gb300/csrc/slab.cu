// slab.cu -- S = 1 matvec and S = 1 decode expert block, "activation slab in
// registers" form.
//
// A row of W is cut into slabs of 32 chunks of 16 bytes (512 bytes: 1024 int4,
// 512 int8 or 128 f32 inputs).  A warp owns one slab at a time: each lane keeps
// the activations of its own 16-byte chunk in registers (read once from the
// swizzled shared-memory copy) and the warp streams rows of that slab -- one
// coalesced 512-byte load per row -- through a software prefetch ring of P
// rows, so the loads of the next P rows are in flight while the current one is
// decoded and multiplied.  Each row's slab partial is reduced across the warp
// and stored per (slab, row) in shared memory; the CTA then adds the slabs of
// a row in ascending order, so results do not depend on timing.
//
// Formats 0, 1, 2 and 4 (fmt=4 with gs = 32 * 2^k, one scale per chunk).
//
// The arithmetic per chunk is that of dot_rows: exact decode of each code into
// the mantissa of 1.0 (or 2^23 for int8), exact offset removal, packed f32x2
// FMA into bit-position classes that are rescaled by powers of two.
#include <type_traits>

#include "coli_internal.cuh"
#include "mbarrier.cuh"

namespace coli {

namespace {

constexpr int kSlabThreads = 256;

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    F2U A{a}, B{b}, D;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(D.u) : "l"(A.u), "l"(B.u));
    return D.f;
}

__host__ __device__ inline size_t staged_words(int fmt, int cpr) { return (size_t)staged_len(fmt, cpr); }

// Activations of one lane's chunk, in registers, and the chunk dot product.
template <int FMT> struct XReg;

template <> struct XReg<4> {
    float4 v[8];
    __device__ __forceinline__ void load(const uint32_t *stage, int c) {
        const float4 *s4 = reinterpret_cast<const float4 *>(stage + (size_t)c * 32);
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = s4[j ^ (c & 7)];
    }
    __device__ __forceinline__ float dot(uint4 q) const {
        Acc4 a;
        Dec4 d = decode4(q.x);
        a.a01 = fmul2(d.v01, make_float2(v[0].x, v[0].y));
        a.a25 = fmul2(d.v25, make_float2(v[0].z, v[0].w));
        a.a36 = fmul2(d.v36, make_float2(v[1].x, v[1].y));
        a.a47 = fmul2(d.v47, make_float2(v[1].z, v[1].w));
        fma4(a, decode4(q.y), v[2], v[3]);
        fma4(a, decode4(q.z), v[4], v[5]);
        fma4(a, decode4(q.w), v[6], v[7]);
        return acc_combine(a);
    }
};
template <> struct XReg<2> : XReg<4> {};

template <> struct XReg<1> {
    float4 v[4];
    __device__ __forceinline__ void load(const uint32_t *stage, int c) {
        const float4 *s4 = reinterpret_cast<const float4 *>(stage + (size_t)c * 16);
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = s4[j ^ ((c >> 1) & 3)];
    }
    __device__ __forceinline__ float dot(uint4 q) const {
        Acc1 a;
        Dec1 d = decode1(q.x);
        a.a = fmul2(d.v01, make_float2(v[0].x, v[0].y));
        a.b = fmul2(d.v23, make_float2(v[0].z, v[0].w));
        fma1(a, decode1(q.y), v[1]);
        fma1(a, decode1(q.z), v[2]);
        fma1(a, decode1(q.w), v[3]);
        return acc_combine(a);
    }
};

template <> struct XReg<0> {
    float4 v;
    __device__ __forceinline__ void load(const uint32_t *stage, int c) {
        v = reinterpret_cast<const float4 *>(stage)[c];
    }
    __device__ __forceinline__ float dot(uint4 q) const {
        float2 a = fmul2(make_float2(__uint_as_float(q.x), __uint_as_float(q.y)), make_float2(v.x, v.y));
        ffma2(a, make_float2(__uint_as_float(q.z), __uint_as_float(q.w)), make_float2(v.z, v.w));
        return a.x + a.y;
    }
};

// Unit walker: units u = w, w+NW, ... over a slab-major index space
// u = s * n_rows + rr, kept incrementally (no division per unit).
struct Walk {
    int s, rr;
    __device__ __forceinline__ void init(int u, int n_rows) {
        s = u / n_rows;
        rr = u - s * n_rows;
    }
    __device__ __forceinline__ void step(int nw, int n_rows) {
        rr += nw;
        while (rr >= n_rows) {
            rr -= n_rows;
            s++;
        }
    }
};

// Stage activations in the swizzled order XReg<FMT> reads.
template <int FMT>
__device__ __forceinline__ void stage_x(uint32_t *dst, const float *src, int n, int cpr) {
    stage_vec<FMT>(reinterpret_cast<float *>(dst), src, n, staged_len(FMT, cpr), threadIdx.x, blockDim.x);
}

__device__ __forceinline__ uint4 ld_or_zero(const uint8_t *p, bool ok) {
    return ok ? ld_stream(p) : make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ matvec
// Rows of all matrices of the job form one index space (row_start prefix);
// CTA b owns rows [b*rpc, (b+1)*rpc).
template <int FMT, int P>
__global__ void __launch_bounds__(kSlabThreads, 2) slab_gemv_kernel(const GemvJob job, int rpc, int gshift) {
    extern __shared__ float4 smem4[];
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem4);
    const size_t xwords = staged_words(FMT, job.cpr);
    float *red = reinterpret_cast<float *>(xs + xwords);   // [n_slab][rpc]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int n_slab = (job.cpr + 31) >> 5;
    const int total_rows = job.row_start[job.n];
    const int r0 = blockIdx.x * rpc;
    const int n_rows = min(rpc, total_rows - r0);
    if (n_rows <= 0) return;

    const int n_units = n_slab * n_rows;
    auto row_of = [&](int rr, int &m, int &o) {
        const int r = r0 + rr;
        m = 0;
        while (r >= job.row_start[m + 1]) m++;
        o = r - job.row_start[m];
    };
    uint4 qb[P];
    float sb[P];
    Walk wl, wc;
    wl.init(warp < n_units ? warp : 0, n_rows);
    wc = wl;
#pragma unroll
    for (int i = 0; i < P; i++) {
        const int u = warp + i * nw;
        const bool ok = u < n_units;
        int m = 0, o = 0;
        if (ok) row_of(wl.rr, m, o);
        const int c = wl.s * 32 + lane;
        const bool okc = ok && c < job.cpr;
        qb[i] = ld_or_zero(job.q[m] + (size_t)o * job.rs[m] + (size_t)c * 16, okc);
        if constexpr (FMT == 4) sb[i] = okc ? __ldg(job.s[m] + (size_t)o * job.ng[m] + (c >> gshift)) : 0.f;
        else if constexpr (FMT != 0) sb[i] = ok ? __ldg(job.s[m] + o) : 0.f;
        else sb[i] = 1.f;
        if (ok) wl.step(nw, n_rows);
    }
    // the first weight loads are in flight; the activations may come from the previous kernel
    pdl_wait();
    stage_x<FMT>(xs, job.x, job.I, job.cpr);
    __syncthreads();
    XReg<FMT> xr;
    int cur_s = -1;
    for (int k0 = 0; warp + k0 * nw < n_units; k0 += P) {
#pragma unroll
        for (int i = 0; i < P; i++) {
            const int u = warp + (k0 + i) * nw;
            if (u >= n_units) break;
            if (wc.s != cur_s) {
                cur_s = wc.s;
                const int c = cur_s * 32 + lane;
                xr.load(xs, c < n_slab * 32 ? c : 0);
            }
            float p = xr.dot(qb[i]) * sb[i];
            // refill slot i with unit u + P*nw
            const int un = u + P * nw;
            const bool ok = un < n_units;
            int m = 0, o = 0;
            if (ok) row_of(wl.rr, m, o);
            const int cn = wl.s * 32 + lane;
            const bool okc = ok && cn < job.cpr;
            qb[i] = ld_or_zero(job.q[m] + (size_t)o * job.rs[m] + (size_t)cn * 16, okc);
            if constexpr (FMT == 4) sb[i] = okc ? __ldg(job.s[m] + (size_t)o * job.ng[m] + (cn >> gshift)) : 0.f;
            else if constexpr (FMT != 0) sb[i] = ok ? __ldg(job.s[m] + o) : 0.f;
            if (ok) wl.step(nw, n_rows);
            p = warp_sum(p);
            if (lane == 0) red[cur_s * rpc + wc.rr] = p;
            wc.step(nw, n_rows);
        }
    }
    pdl_trigger();
    __syncthreads();
    for (int rr = threadIdx.x; rr < n_rows; rr += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < n_slab; s++) acc += red[s * rpc + rr];
        int m, o;
        row_of(rr, m, o);
        job.y[m][o] = acc;
    }
}

// ------------------------------------------------------------------ decode block, S = 1
__device__ bool slab_grid_barrier(unsigned *bar, int *err, long long timeout_ns) {
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

__device__ __forceinline__ const float *srow(int fmt, const MatDesc &m, int row) {
    return fmt == 4 ? m.s + (size_t)row * m.ng : m.s + row;
}

template <int FMT>
__device__ __forceinline__ float unit_scale(const MatDesc &m, int row, int c, int gshift, bool ok) {
    if constexpr (FMT == 4) return ok ? __ldg(m.s + (size_t)row * m.ng + (c >> gshift)) : 0.f;
    else if constexpr (FMT == 0) return 1.f;
    else return ok ? __ldg(m.s + row) : 0.f;
}

// Phase A unit = (slab s, pair index pr) -> expert a = pr / F, row j = pr % F,
// two rows (gate j, up j) of expert a; all against the token's activations.
// Phase B unit = (expert-in-batch a, slab s, row rr of the CTA's output rows).
template <int FMT, int P>
__global__ void __launch_bounds__(kSlabThreads, 2) moe_decode_slab_kernel(const MoeDecodeArgs a, int gshift_gu,
                                                                           int gshift_d) {
    extern __shared__ float4 smem4[];
    uint32_t *stage = reinterpret_cast<uint32_t *>(smem4);
    __shared__ int s_ids[kMaxDecodeSlots];
    __shared__ float s_w[kMaxDecodeSlots];
    __shared__ int s_exp[kMaxDecodeSlots];
    __shared__ float s_ew[kMaxDecodeSlots];
    __shared__ int s_nact, s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int n = a.K;   // S = 1

    // ---- phase 0: distinct routed experts in ascending id order, weights summed
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
    if (tid == 0) {
        int na = 0;
        int last = -1;
        for (;;) {   // next larger id
            int best = 0x7fffffff;
            for (int t = 0; t < n; t++)
                if (s_ids[t] > last && s_ids[t] < best) best = s_ids[t];
            if (best == 0x7fffffff) break;
            float wsum = 0.f;
            for (int t = 0; t < n; t++)
                if (s_ids[t] == best) wsum += s_w[t];
            s_exp[na] = best;
            s_ew[na] = wsum;
            na++;
            last = best;
        }
        s_nact = na;
    }
    __syncthreads();
    const int nact = s_nact;

    // ---- phase A: h[a][j] = silu(G_a[j] x) * (U_a[j] x)
    const size_t xw_gu = staged_words(FMT, a.cpr_gu);
    const int n_slab_gu = (a.cpr_gu + 31) >> 5;
    const long long pairs = (long long)nact * a.F;
    const int ppc = (int)((pairs + gridDim.x - 1) / gridDim.x);       // pairs per CTA
    const long long pr0 = (long long)blockIdx.x * ppc;
    const int n_pr = (int)max(0LL, min((long long)ppc, pairs - pr0));
    float *redA = reinterpret_cast<float *>(stage + xw_gu);           // [n_slab][ppc][2]
    if (n_pr > 0) {
        stage_x<FMT>(stage, a.x, a.H, a.cpr_gu);
        __syncthreads();
        const int n_units = n_slab_gu * n_pr;
        uint4 qg[P], qu[P];
        float sg[P], su[P];
        Walk wl, wc;
        wl.init(warp < n_units ? warp : 0, n_pr);
        wc = wl;
        // (expert index, row) of the prefetch walker, kept incrementally; the
        // expert's gate/up descriptors are cached and reloaded on change
        int lai, lj;
        {
            const long long pr = pr0 + wl.rr;
            lai = (int)(pr / a.F);
            lj = (int)(pr - (long long)lai * a.F);
        }
        int cur_ai = -1;
        MatDesc Gd = {}, Ud = {};
        auto load = [&](int i, bool ok) {
            if (ok && lai != cur_ai) {
                cur_ai = lai;
                const ExpertDesc &E = a.table[s_exp[lai]];
                Gd = E.m[0];
                Ud = E.m[1];
            }
            const int j = lj;
            const int c = wl.s * 32 + lane;
            const bool okc = ok && c < a.cpr_gu;
            qg[i] = ld_or_zero(Gd.q + (size_t)j * Gd.rs + (size_t)c * 16, okc);
            qu[i] = ld_or_zero(Ud.q + (size_t)j * Ud.rs + (size_t)c * 16, okc);
            sg[i] = unit_scale<FMT>(Gd, j, c, gshift_gu, okc);
            su[i] = unit_scale<FMT>(Ud, j, c, gshift_gu, okc);
            if (ok) {
                const int rr_before = wl.rr;
                wl.step(nw, n_pr);
                // advance (lai, lj) by the same pair-index step (rr moved by nw, minus n_pr per slab wrap)
                lj += wl.rr - rr_before;
                while (lj >= a.F) { lj -= a.F; lai++; }
                while (lj < 0) { lj += a.F; lai--; }
            }
        };
#pragma unroll
        for (int i = 0; i < P; i++) load(i, warp + i * nw < n_units);
        XReg<FMT> xr;
        int cur_s = -1;
        for (int k0 = 0; warp + k0 * nw < n_units; k0 += P) {
#pragma unroll
            for (int i = 0; i < P; i++) {
                const int u = warp + (k0 + i) * nw;
                if (u >= n_units) break;
                if (wc.s != cur_s) {
                    cur_s = wc.s;
                    const int c = cur_s * 32 + lane;
                    xr.load(stage, c);
                }
                float pg = xr.dot(qg[i]) * sg[i];
                float pu = xr.dot(qu[i]) * su[i];
                load(i, u + P * nw < n_units);
                pg = warp_sum(pg);
                pu = warp_sum(pu);
                if (lane == 0) {
                    redA[(cur_s * ppc + wc.rr) * 2] = pg;
                    redA[(cur_s * ppc + wc.rr) * 2 + 1] = pu;
                }
                wc.step(nw, n_pr);
            }
        }
        __syncthreads();
        for (int rr = tid; rr < n_pr; rr += blockDim.x) {
            float g = 0.f, u = 0.f;
            for (int s = 0; s < n_slab_gu; s++) {
                g += redA[(s * ppc + rr) * 2];
                u += redA[(s * ppc + rr) * 2 + 1];
            }
            a.hbuf[pr0 + rr] = g / (1.0f + expf(-g)) * u;   // hbuf[a][j] = hbuf[pr]
        }
    }

    if (!slab_grid_barrier(a.bar, a.err, a.timeout_ns)) return;

    // ---- phase B: y[o] = sum_a w_a * D_a[o] h_a over this CTA's rows
    const size_t xw_d = staged_words(FMT, a.cpr_d);
    const int n_slab_d = (a.cpr_d + 31) >> 5;
    const int rpc = a.rpc;
    const int oc0 = blockIdx.x * rpc;
    const int n_o = min(rpc, a.H - oc0);
    if (n_o <= 0) return;
    float *redB = reinterpret_cast<float *>(stage + (size_t)a.sb * xw_d);   // [sb][n_slab][rpc]
    float *yacc = redB + (size_t)a.sb * n_slab_d * rpc;
    for (int t = tid; t < n_o; t += blockDim.x) yacc[t] = 0.f;
    for (int b0 = 0; b0 < nact; b0 += a.sb) {
        const int nb = min(a.sb, nact - b0);
        __syncthreads();
        if (xw_d == (size_t)a.F) {   // contiguous unpadded rows of h: one staging pass
            stage_vec<FMT>(reinterpret_cast<float *>(stage), a.hbuf + (size_t)b0 * a.F, nb * a.F, nb * (int)xw_d, tid,
                           blockDim.x);
        } else {
            for (int bi = 0; bi < nb; bi++)
                stage_x<FMT>(stage + (size_t)bi * xw_d, a.hbuf + (size_t)(b0 + bi) * a.F, a.F, a.cpr_d);
        }
        __syncthreads();
        const int per_e = n_slab_d * n_o;
        const int n_units = nb * per_e;
        uint4 qb[2 * P];
        float sb[2 * P];
        // unit u -> (bi, s, rr) with u = (bi * n_slab_d + s) * n_o + rr; walker over (bs, rr)
        Walk wl, wc;
        wl.init(warp < n_units ? warp : 0, n_o);
        wc = wl;
        int lbi = wl.s / n_slab_d, lsl = wl.s - lbi * n_slab_d;   // (expert in batch, slab) of the prefetch walker
        int cur_bi = -1;
        MatDesc Dd = {};
        auto load = [&](int i, bool ok) {
            if (ok && lbi != cur_bi) {
                cur_bi = lbi;
                Dd = a.table[s_exp[b0 + lbi]].m[2];
            }
            const int o = oc0 + wl.rr;
            const int c = lsl * 32 + lane;
            const bool okc = ok && c < a.cpr_d;
            qb[i] = ld_or_zero(Dd.q + (size_t)o * Dd.rs + (size_t)c * 16, okc);
            sb[i] = unit_scale<FMT>(Dd, o, c, gshift_d, okc);
            if (ok) {
                const int s_before = wl.s;
                wl.step(nw, n_o);
                for (int k = s_before; k < wl.s; k++)
                    if (++lsl == n_slab_d) { lsl = 0; lbi++; }
            }
        };
#pragma unroll
        for (int i = 0; i < 2 * P; i++) load(i, warp + i * nw < n_units);
        XReg<FMT> xr;
        int cur = -1;
        for (int k0 = 0; warp + k0 * nw < n_units; k0 += 2 * P) {
#pragma unroll
            for (int i = 0; i < 2 * P; i++) {
                const int u = warp + (k0 + i) * nw;
                if (u >= n_units) break;
                if (wc.s != cur) {
                    cur = wc.s;
                    const int bi = cur / n_slab_d, s = cur - bi * n_slab_d;
                    xr.load(stage + (size_t)bi * xw_d, s * 32 + lane);
                }
                float p = xr.dot(qb[i]) * sb[i];
                load(i, u + 2 * P * nw < n_units);
                p = warp_sum(p);
                if (lane == 0) redB[(size_t)cur * rpc + wc.rr] = p;
                wc.step(nw, n_o);
            }
        }
        __syncthreads();
        for (int rr = tid; rr < n_o; rr += blockDim.x) {
            float acc = yacc[rr];
            for (int bi = 0; bi < nb; bi++) {
                float d = 0.f;
                for (int s = 0; s < n_slab_d; s++) d += redB[(size_t)(bi * n_slab_d + s) * rpc + rr];
                acc = fmaf(s_ew[b0 + bi], d, acc);
            }
            yacc[rr] = acc;
        }
    }
    __syncthreads();
    for (int rr = tid; rr < n_o; rr += blockDim.x) a.y[oc0 + rr] = yacc[rr];
}


// ------------------------------------------------------------------ lane decoders of the streamed matvec
// int4 chunk dot product without the offset-removal adds.
// A code n at bit position p of a word, AND-ed out with no exponent bits, is
// the f32 subnormal n * 2^(p-149), exactly.  Each lane holds its chunk's
// activations multiplied by 2^(k-p), p the bit position its code will sit at
// and k chosen from the chunk's largest |x| so that |x * 2^k| < 2^27 (exact:
// powers of two).  Every product is then n * x * 2^(k-149), the same scale for
// all positions, a normal f32 formed with the usual single rounding of the FMA,
// so two accumulators per chunk suffice; the sum is rescaled by 2^(149-k) and
// the code offset 8 comes off as 8 * sum(x).  The FMAs must keep subnormal
// inputs: plain fma.rn.f32x2, no flush to zero.
__device__ __forceinline__ float exp2i(int e) {   // 2^e for -126 <= e <= 127
    return __int_as_float((e + 127) << 23);
}
__device__ __forceinline__ float mul_exp2(float x, int e) {   // x * 2^e, -252 <= e <= 254, exact unless it under/overflows
    return (x * exp2i(e / 2)) * exp2i(e - e / 2);
}
struct XRegS4 {
    static constexpr int LB = 16, NIN = 32;   // code bytes and inputs per lane
    using Q = uint4;
    float4 v[8];        // x * 2^(k-p), pairs in the order of dot()
    float xsum;         // sum of the chunk's 32 activations
    float f1, f2, f3;   // 2^(149-k) = f1 * f2 * f3
    // raw[2k], raw[2k+1]: inputs 8k..8k+3, 8k+4..8k+7 of the chunk in natural order
    __device__ __forceinline__ void set(const float4 (&raw)[8]) {
        float t = 0.f, mx = 0.f;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float4 a = raw[2 * k], b = raw[2 * k + 1];
            t += ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                 fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w)))));
        }
        xsum = t;
        // biased exponent eb of mx: mx < 2^(eb-126); k = 153 - eb, kept in [-126, 127]
        const int eb = (__float_as_int(mx) >> 23) & 0xFF;
        const int ks = min(127, max(-126, 153 - eb));
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float4 a = raw[2 * k], b = raw[2 * k + 1];
            // x0 x1 x2 x5 at bit positions 0 4 8 8 | x3 x6 x4 x7 at 12 12 16 16
            v[2 * k] = make_float4(mul_exp2(a.x, ks), mul_exp2(a.y, ks - 4), mul_exp2(a.z, ks - 8), mul_exp2(b.y, ks - 8));
            v[2 * k + 1] = make_float4(mul_exp2(a.w, ks - 12), mul_exp2(b.z, ks - 12), mul_exp2(b.x, ks - 16),
                                       mul_exp2(b.w, ks - 16));
        }
        const int r = 149 - ks;   // in [22, 275]
        f1 = exp2i(r / 3);
        f2 = exp2i(r / 3);
        f3 = exp2i(r - 2 * (r / 3));
    }
    // chunk c of a vector staged by stage_vec<4> (permuted, swizzled, zero padded)
    __device__ __forceinline__ void load_staged(const uint32_t *stage, int c) {
        const float4 *s4 = reinterpret_cast<const float4 *>(stage + (size_t)c * 32);
        float4 raw[8];
#pragma unroll
        for (int j = 0; j < 8; j++) raw[j] = s4[j ^ (c & 7)];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float4 p0 = raw[2 * k], p1 = raw[2 * k + 1];   // staged: x0 x1 x2 x5 | x3 x6 x4 x7
            raw[2 * k] = make_float4(p0.x, p0.y, p0.z, p1.x);
            raw[2 * k + 1] = make_float4(p1.z, p0.w, p1.y, p1.w);
        }
        set(raw);
    }
    __device__ __forceinline__ static float2 sub2(uint32_t a, uint32_t b) {
        return make_float2(__uint_as_float(a), __uint_as_float(b));
    }
    __device__ __forceinline__ float finish(float2 a, float2 b) const {
        const float s = (a.x + a.y) + (b.x + b.y);
        return fmaf(-8.0f, xsum, ((s * f1) * f2) * f3);
    }
    // N chunks against the same activations, interleaved word by word
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        float2 a[N], b[N];
#pragma unroll
        for (int d = 0; d < N; d++) a[d] = b[d] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; k++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t w = k == 0 ? q[d].x : k == 1 ? q[d].y : k == 2 ? q[d].z : q[d].w;
                const uint32_t hi = w >> 12;
                ffma2(a[d], sub2(w & 0xFu, w & 0xF0u), make_float2(v[2 * k].x, v[2 * k].y));
                ffma2(b[d], sub2(w & 0xF00u, hi & 0xF00u), make_float2(v[2 * k].z, v[2 * k].w));
                ffma2(a[d], sub2(w & 0xF000u, hi & 0xF000u), make_float2(v[2 * k + 1].x, v[2 * k + 1].y));
                ffma2(b[d], sub2(w & 0xF0000u, hi & 0xF0000u), make_float2(v[2 * k + 1].z, v[2 * k + 1].w));
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = finish(a[d], b[d]);
    }
    __device__ __forceinline__ void dot4(const uint4 (&q)[4], float (&out)[4]) const { dotn<4>(q, out); }
};


// int8 (stored offset binary u = code + 128), 16 inputs per lane: bytes 0, 1 of
// a word at bit positions 0 and 8, bytes 2, 3 the same after a 16-bit shift;
// the offset comes off as 128 * sum(x).  Same scaling as XRegS4.
struct XRegS1 {
    static constexpr int LB = 16, NIN = 16;
    using Q = uint4;
    float4 v[4];
    float xsum, f1, f2, f3;
    __device__ __forceinline__ void set(const float4 (&raw)[4]) {
        float t = 0.f, mx = 0.f;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float4 a = raw[j];
            t += (a.x + a.y) + (a.z + a.w);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
        xsum = t;
        const int eb = (__float_as_int(mx) >> 23) & 0xFF;
        const int ks = min(127, max(-126, 153 - eb));
#pragma unroll
        for (int j = 0; j < 4; j++)
            v[j] = make_float4(mul_exp2(raw[j].x, ks), mul_exp2(raw[j].y, ks - 8), mul_exp2(raw[j].z, ks),
                               mul_exp2(raw[j].w, ks - 8));
        const int r = 149 - ks;
        f1 = exp2i(r / 3);
        f2 = exp2i(r / 3);
        f3 = exp2i(r - 2 * (r / 3));
    }
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        float2 a[N], b[N];
#pragma unroll
        for (int d = 0; d < N; d++) a[d] = b[d] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; k++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t w = k == 0 ? q[d].x : k == 1 ? q[d].y : k == 2 ? q[d].z : q[d].w;
                const uint32_t hi = w >> 16;
                ffma2(a[d], XRegS4::sub2(w & 0xFFu, w & 0xFF00u), make_float2(v[k].x, v[k].y));
                ffma2(b[d], XRegS4::sub2(hi & 0xFFu, hi & 0xFF00u), make_float2(v[k].z, v[k].w));
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) {
            const float sm = (a[d].x + a[d].y) + (b[d].x + b[d].y);
            out[d] = fmaf(-128.0f, xsum, ((sm * f1) * f2) * f3);
        }
    }
};

// int2 (crumb - 2), 32 inputs per lane = 8 code bytes: crumbs 0..10 of a word at
// their own bit positions, 11..15 after a 12-bit shift; the offset comes off as
// 2 * sum(x).  Same scaling as XRegS4.
struct XRegS3 {
    static constexpr int LB = 8, NIN = 32;
    using Q = uint2;
    float2 v[16];       // pair j of word k: v[8k + j]
    float xsum, f1, f2, f3;
    __device__ __forceinline__ static int pos(int t) { return t <= 10 ? 2 * t : 2 * t - 12; }
    __device__ __forceinline__ void set(const float4 (&raw)[8]) {
        float xs[32];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            xs[4 * j] = raw[j].x;
            xs[4 * j + 1] = raw[j].y;
            xs[4 * j + 2] = raw[j].z;
            xs[4 * j + 3] = raw[j].w;
        }
        float t = 0.f, mx = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i++) {
            t += xs[i];
            mx = fmaxf(mx, fabsf(xs[i]));
        }
        xsum = t;
        const int eb = (__float_as_int(mx) >> 23) & 0xFF;
        const int ks = min(127, max(-126, 153 - eb));
#pragma unroll
        for (int k = 0; k < 2; k++)
#pragma unroll
            for (int j = 0; j < 8; j++)
                v[8 * k + j] = make_float2(mul_exp2(xs[16 * k + 2 * j], ks - pos(2 * j)),
                                           mul_exp2(xs[16 * k + 2 * j + 1], ks - pos(2 * j + 1)));
        const int r = 149 - ks;
        f1 = exp2i(r / 3);
        f2 = exp2i(r / 3);
        f3 = exp2i(r - 2 * (r / 3));
    }
    template <int N>
    __device__ __forceinline__ void dotn(const uint2 (&q)[N], float (&out)[N]) const {
        float2 a[N], b[N];
#pragma unroll
        for (int d = 0; d < N; d++) a[d] = b[d] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 2; k++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t w = k == 0 ? q[d].x : q[d].y, hi = w >> 12;
                const float2 *vk = v + 8 * k;
                ffma2(a[d], XRegS4::sub2(w & 0x3u, w & 0xCu), vk[0]);
                ffma2(b[d], XRegS4::sub2(w & 0x30u, w & 0xC0u), vk[1]);
                ffma2(a[d], XRegS4::sub2(w & 0x300u, w & 0xC00u), vk[2]);
                ffma2(b[d], XRegS4::sub2(w & 0x3000u, w & 0xC000u), vk[3]);
                ffma2(a[d], XRegS4::sub2(w & 0x30000u, w & 0xC0000u), vk[4]);
                ffma2(b[d], XRegS4::sub2(w & 0x300000u, hi & 0xC00u), vk[5]);
                ffma2(a[d], XRegS4::sub2(hi & 0x3000u, hi & 0xC000u), vk[6]);
                ffma2(b[d], XRegS4::sub2(hi & 0x30000u, hi & 0xC0000u), vk[7]);
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) {
            const float sm = (a[d].x + a[d].y) + (b[d].x + b[d].y);
            out[d] = fmaf(-2.0f, xsum, ((sm * f1) * f2) * f3);
        }
    }
};


// f32 weights, 16 inputs per lane (64 contiguous bytes): plain f32x2 FMAs.
struct Q4 {
    uint4 v[4];
};
struct XRegF32 {
    static constexpr int LB = 64, NIN = 16;
    using Q = Q4;
    float4 x[4];
    __device__ __forceinline__ void set(const float4 (&raw)[4]) {
#pragma unroll
        for (int j = 0; j < 4; j++) x[j] = raw[j];
    }
    template <int N>
    __device__ __forceinline__ void dotn(const Q4 (&q)[N], float (&out)[N]) const {
#pragma unroll
        for (int d = 0; d < N; d++) {
            float2 a = make_float2(0.f, 0.f), b = a;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                ffma2(a, make_float2(__uint_as_float(q[d].v[j].x), __uint_as_float(q[d].v[j].y)),
                      make_float2(x[j].x, x[j].y));
                ffma2(b, make_float2(__uint_as_float(q[d].v[j].z), __uint_as_float(q[d].v[j].w)),
                      make_float2(x[j].z, x[j].w));
            }
            out[d] = (a.x + a.y) + (b.x + b.y);
        }
    }
};

// FP8 E4M3 (fmt=7), 16 inputs per lane: each byte pair converts exactly to an
// f16 pair and then to f32 (no offset, no scaling); the 128 x 128 block scale
// is applied per lane chunk by the caller (BlockScaled).
struct XRegF8 {
    static constexpr int LB = 16, NIN = 16;
    using Q = uint4;
    float4 v[4];   // inputs 4k..4k+3 of the lane's 16, natural order
    __device__ __forceinline__ void set(const float4 (&raw)[4]) {
#pragma unroll
        for (int k = 0; k < 4; k++) v[k] = raw[k];
    }
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        float2 a[N], b[N];
#pragma unroll
        for (int d = 0; d < N; d++) a[d] = b[d] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; k++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t w = k == 0 ? q[d].x : k == 1 ? q[d].y : k == 2 ? q[d].z : q[d].w;
                ffma2(a[d], e4m3x2_to_f32x2(w & 0xFFFFu), make_float2(v[k].x, v[k].y));
                ffma2(b[d], e4m3x2_to_f32x2(w >> 16), make_float2(v[k].z, v[k].w));
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = (a[d].x + a[d].y) + (b[d].x + b[d].y);
    }
};

// Decoders whose lane unit is several 16-byte chunks (f32: four): chunk j of
// lane l of a slab sits at (32 j + l) * 16 bytes, so each 16-byte load of a
// warp reads 512 contiguous bytes (no bank conflicts), and the lane's inputs
// follow the same interleave.
template <class XR> struct Interleaved { static constexpr bool value = false; };
template <> struct Interleaved<XRegF32> { static constexpr bool value = true; };

// Decoders whose scale is per 128 x 128 block (read from global memory by the
// consumer) instead of per row or per row group (copied with the rows).
template <class XR> struct BlockScaled { static constexpr bool value = false; };
template <> struct BlockScaled<XRegF8> { static constexpr bool value = true; };

// Sums of four per-lane values over the warp with 6 shuffles: afterwards lane
// 8k (k = 0..3) holds the total of value k.
__device__ __forceinline__ float warp_sum4(float v0, float v1, float v2, float v3, int lane) {
    const bool h16 = lane & 16, h8 = lane & 8;
    float a0 = h16 ? v2 : v0, a1 = h16 ? v3 : v1;
    const float b0 = h16 ? v0 : v2, b1 = h16 ? v1 : v3;
    a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
    float k = h8 ? a1 : a0;
    const float sd = h8 ? a0 : a1;
    k += __shfl_xor_sync(0xffffffffu, sd, 8);
    k += __shfl_xor_sync(0xffffffffu, k, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    return k;
}

// ------------------------------------------------------------------ matvec, S = 1, streamed
// The same streaming scheme as the decode block's phase A for coli_matmul at
// S = 1: rows of all matrices of the call form one index space, CTA b owns a
// contiguous block of rpc rows, warp 12 copies stages of RG rows (codes and
// scales) into the ring, warps 0-11 own one 512-byte slab each with the
// activations in registers and form four row dot products per stage.  fmt=4
// reads the group scale of each 32-input chunk, fmt 1-3 the row scale (both
// copied with the rows), fmt=7 the scale of the chunk's 128 x 128 block (from
// global memory, where the whole scale grid stays cached).
// NR (1, 2 or 4): rows of a stage each consumer warp multiplies, the stage's
// rows per slab group rounded up (RG <= NR * G).
template <int NWC, class XR, int NR>
__global__ void __launch_bounds__((NWC + 1) * 32, 1) stream_gemv_kernel(const GemvJob job, int rpc, int RG,
                                                                         int gshift, long long timeout_ns) {
    constexpr int NCT = NWC * 32, NS = kStreamStages, SB = kStreamStageBytes;
    extern __shared__ uint8_t sraw[];
    uint8_t *ring = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    float *red = reinterpret_cast<float *>(ring + NS * SB);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + NS * SB + kStreamRedBytes);
    uint64_t *empty = full + NS;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = job.row_start[job.n];
    const int r0 = blockIdx.x * rpc, r1 = min(total, r0 + rpc);
    if (r0 >= r1) return;
    uint64_t deadline = global_ns() + (uint64_t)timeout_ns;
    // lane units: XR::LB code bytes = XR::NIN inputs; a row has lpr of them
    const int lpr = (job.I + XR::NIN - 1) / XR::NIN;
    const int ns = (lpr + 31) >> 5, sl = warp % ns, sub = warp / ns, G = NWC / ns;
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NWC);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // one CTA fills an SM (its ring takes most of the shared memory): the next
    // kernel may launch now; its CTAs start as this kernel frees SMs
    pdl_trigger();
    // scales copied with each row: none for f32 and for block-scaled FP8
    const int ng = job.fmt == 4 ? job.ng[0] : (job.fmt == 0 || BlockScaled<XR>::value) ? 0 : 1;
    const long long rs = job.rs[0];
    // stage cursor: next row r, its matrix m
    int r = r0, m = 0;
    while (r >= job.row_start[m + 1]) m++;
    auto next = [&](int &st_m, int &st_o, int &st_n) -> bool {
        if (r >= r1) return false;
        while (r >= job.row_start[m + 1]) m++;
        st_m = m;
        st_o = r - job.row_start[m];
        st_n = min(RG, min(r1, job.row_start[m + 1]) - r);
        r += st_n;
        return true;
    };
    int sm_, so, sn;
    if (warp == NWC) {
        if (lane == 0) {
            int s = 0, it = 0;
            uint32_t ph = 0;
            while (next(sm_, so, sn)) {
                if (it == NS) {
                    // the ring is full of weights; from here on the consumers, which
                    // waited for the previous kernel, pace the copies
                    pdl_wait();
                    deadline = global_ns() + (uint64_t)timeout_ns;
                }
                if (it >= NS && !mbar_wait(&empty[s], ph ^ 1, deadline, &abort_flag)) {
                    if (!abort_flag) {
                        abort_flag = 1;
                        atomicCAS(job.err, 0, DEV_ERR_TIMEOUT);
                    }
                    break;
                }
                uint8_t *dst = ring + s * SB;
                const uint32_t cb = (uint32_t)(sn * rs), sbytes = (uint32_t)(sn * ng * 4);
                mbar_expect_tx(&full[s], cb + sbytes);
                bulk_load(dst, job.q[sm_] + (size_t)so * rs, cb, &full[s]);
                if (sbytes) bulk_load(dst + RG * rs, job.s[sm_] + (size_t)so * ng, sbytes, &full[s]);
                it++;
                if (++s == NS) {
                    s = 0;
                    ph ^= 1;
                }
            }
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int k = max(0, it - NS); k < it; k++) mbar_wait(&full[k % NS], (k / NS) & 1, dl2, &no_abort);
        }
        return;
    }
    pdl_wait();
    deadline = global_ns() + (uint64_t)timeout_ns;
    constexpr bool IL = Interleaved<XR>::value;
    constexpr int NCH = XR::LB / 16;   // 16-byte chunks of a lane unit (interleaved decoders)
    float4 xraw[XR::NIN / 4];
#pragma unroll
    for (int j = 0; j < XR::NIN / 4; j++) xraw[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (IL) {
        // chunk j of this lane: inputs sl * 32 * NIN + (32 j + lane) * 4 .. + 3 (I is a multiple of 128)
#pragma unroll
        for (int j = 0; j < NCH; j++) {
            const int i0 = sl * 32 * XR::NIN + (32 * j + lane) * 4;
            if (i0 < job.I) xraw[j] = __ldg(reinterpret_cast<const float4 *>(job.x + i0));
        }
    } else if (sl * 32 + lane < lpr) {
        const float4 *p = reinterpret_cast<const float4 *>(job.x + (size_t)(sl * 32 + lane) * XR::NIN);
#pragma unroll
        for (int j = 0; j < XR::NIN / 4; j++) xraw[j] = __ldg(p + j);
    }
    XR xr;
    xr.set(xraw);
    int s = 0;
    uint32_t ph = 0;
    const int c = sl * 32 + lane;
    const bool okc = c < lpr;
    using Q = typename XR::Q;
    while (next(sm_, so, sn)) {
        if (warp_wait(&full[s], ph, deadline, &abort_flag, lane)) {
            const uint8_t *src = ring + s * SB;
            Q qq[NR];
            float sc[NR], dd[NR];
#pragma unroll
            for (int k = 0; k < NR; k++) {
                const int rr = sub + k * G;
                const bool ok = okc && rr < sn;
                if constexpr (IL) {
                    const uint8_t *rb = src + rr * rs + sl * 32 * XR::LB + lane * 16;
#pragma unroll
                    for (int j = 0; j < NCH; j++)
                        reinterpret_cast<uint4 *>(&qq[k])[j] =
                            (rr < sn && sl * 32 * XR::NIN + (32 * j + lane) * 4 < job.I)
                                ? *reinterpret_cast<const uint4 *>(rb + j * 512)
                                : make_uint4(0u, 0u, 0u, 0u);
                } else {
                    qq[k] = ok ? *reinterpret_cast<const Q *>(src + rr * rs + c * XR::LB) : Q{};
                }
                if constexpr (IL)
                    sc[k] = rr < sn ? 1.f : 0.f;   // (f32: no scales; chunk validity is in the loads)
                else if constexpr (BlockScaled<XR>::value)
                    sc[k] = ok ? __ldg(job.s[sm_] + (size_t)((so + rr) / kFp8Block) * job.ng[sm_] + (c >> gshift)) : 0.f;
                else
                    sc[k] = !ok ? 0.f : ng == 0 ? 1.f : *reinterpret_cast<const float *>(src + RG * rs + (rr * ng + (c >> gshift)) * 4);
            }
            xr.template dotn<NR>(qq, dd);
            if constexpr (NR == 1) {
                float t = dd[0] * sc[0];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0 && sub < sn) red[(job.row_start[sm_] + so + sub - r0) * ns + sl] = t;
            } else {
                float v[4];
#pragma unroll
                for (int k = 0; k < 4; k++) v[k] = k < NR ? dd[k] * sc[k] : 0.f;
                const float t = warp_sum4(v[0], v[1], v[2], v[3], lane);
                if ((lane & 7) == 0 && (lane >> 3) < NR) {
                    const int rr = sub + (lane >> 3) * G;
                    if (rr < sn) red[(job.row_start[sm_] + so + rr - r0) * ns + sl] = t;
                }
            }
        } else if (!abort_flag && lane == 0) {
            abort_flag = 1;
            atomicCAS(job.err, 0, DEV_ERR_TIMEOUT);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == NS) {
            s = 0;
            ph ^= 1;
        }
    }
    named_sync(1, NCT);
    for (int rr = tid; rr < r1 - r0; rr += NCT) {
        float acc = 0.f;
        for (int k = 0; k < ns; k++) acc += red[rr * ns + k];
        const int rg = r0 + rr;
        int mm = 0;
        while (rg >= job.row_start[mm + 1]) mm++;
        job.y[mm][rg - job.row_start[mm]] = acc;
    }
}


// ------------------------------------------------------------------ matvec, S = 2..4, int4, streamed
// As stream_gemv_kernel, but every lane covers half a chunk (8 bytes = 16
// inputs) so that the activations of all S rows fit in registers: a warp owns a
// 256-byte half slab of every row, decodes each code once and multiplies it
// into S accumulators.  Activations are pre-scaled per lane and per code
// position exactly as in XRegS4.
template <int S>
struct XRegHalf {
    float4 v[S][4];     // per row: x * 2^(k-p), pairs in the order of the dot product
    float xsum[S], f1[S], f2[S], f3[S];
    __device__ __forceinline__ void set(int row, const float4 (&raw)[4]) {
        float t = 0.f, mx = 0.f;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float4 a = raw[j];
            t += (a.x + a.y) + (a.z + a.w);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
        xsum[row] = t;
        const int eb = (__float_as_int(mx) >> 23) & 0xFF;
        const int ks = min(127, max(-126, 153 - eb));
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const float4 a = raw[2 * k], b = raw[2 * k + 1];
            v[row][2 * k] =
                make_float4(mul_exp2(a.x, ks), mul_exp2(a.y, ks - 4), mul_exp2(a.z, ks - 8), mul_exp2(b.y, ks - 8));
            v[row][2 * k + 1] = make_float4(mul_exp2(a.w, ks - 12), mul_exp2(b.z, ks - 12), mul_exp2(b.x, ks - 16),
                                            mul_exp2(b.w, ks - 16));
        }
        const int r = 149 - ks;
        f1[row] = exp2i(r / 3);
        f2[row] = exp2i(r / 3);
        f3[row] = exp2i(r - 2 * (r / 3));
    }
    // dot products of N code half-chunks with the S rows: out[d][s]
    template <int N>
    __device__ __forceinline__ void dots(const uint2 (&q)[N], float (&out)[N][S]) const {
        float2 acc[N][S];
#pragma unroll
        for (int d = 0; d < N; d++)
#pragma unroll
            for (int r = 0; r < S; r++) acc[d][r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 2; k++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t w = k == 0 ? q[d].x : q[d].y, hi = w >> 12;
                const float2 c01 = XRegS4::sub2(w & 0xFu, w & 0xF0u), c25 = XRegS4::sub2(w & 0xF00u, hi & 0xF00u);
                const float2 c36 = XRegS4::sub2(w & 0xF000u, hi & 0xF000u);
                const float2 c47 = XRegS4::sub2(w & 0xF0000u, hi & 0xF0000u);
#pragma unroll
                for (int r = 0; r < S; r++) {
                    ffma2(acc[d][r], c01, make_float2(v[r][2 * k].x, v[r][2 * k].y));
                    ffma2(acc[d][r], c25, make_float2(v[r][2 * k].z, v[r][2 * k].w));
                    ffma2(acc[d][r], c36, make_float2(v[r][2 * k + 1].x, v[r][2 * k + 1].y));
                    ffma2(acc[d][r], c47, make_float2(v[r][2 * k + 1].z, v[r][2 * k + 1].w));
                }
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++)
#pragma unroll
            for (int r = 0; r < S; r++)
                out[d][r] = fmaf(-8.0f, xsum[r], (((acc[d][r].x + acc[d][r].y) * f1[r]) * f2[r]) * f3[r]);
    }
};

template <int NWC, int S>
__global__ void __launch_bounds__((NWC + 1) * 32, 1) stream_gemv_s_kernel(const GemvJob job, int rpc, int RG,
                                                                           int gshift, long long timeout_ns) {
    constexpr int NCT = NWC * 32, NS = kStreamStages, SB = kStreamStageBytes;
    extern __shared__ uint8_t sraw[];
    uint8_t *ring = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    float *red = reinterpret_cast<float *>(ring + NS * SB);   // [rpc][S][nh]
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + NS * SB + kStreamGemvRedBytes);
    uint64_t *empty = full + NS;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = job.row_start[job.n];
    const int r0 = blockIdx.x * rpc, r1 = min(total, r0 + rpc);
    if (r0 >= r1) return;
    uint64_t deadline = global_ns() + (uint64_t)timeout_ns;
    const int hcpr = job.cpr * 2;                        // 8-byte half chunks per row
    const int nh = (hcpr + 31) >> 5, sl = warp % nh, sub = warp / nh, G = NWC / nh;
    const int hc = sl * 32 + lane;                       // this lane's half chunk
    const bool okc = hc < hcpr;
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NWC);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int ng = job.fmt == 4 ? job.ng[0] : 1;
    const long long rs = job.rs[0];
    int r = r0, m = 0;
    while (r >= job.row_start[m + 1]) m++;
    auto next = [&](int &st_m, int &st_o, int &st_n) -> bool {
        if (r >= r1) return false;
        while (r >= job.row_start[m + 1]) m++;
        st_m = m;
        st_o = r - job.row_start[m];
        st_n = min(RG, min(r1, job.row_start[m + 1]) - r);
        r += st_n;
        return true;
    };
    int sm_, so, sn;
    if (warp == NWC) {
        if (lane == 0) {
            int s = 0, it = 0;
            uint32_t ph = 0;
            while (next(sm_, so, sn)) {
                if (it == NS) {
                    pdl_wait();
                    deadline = global_ns() + (uint64_t)timeout_ns;
                }
                if (it >= NS && !mbar_wait(&empty[s], ph ^ 1, deadline, &abort_flag)) {
                    if (!abort_flag) {
                        abort_flag = 1;
                        atomicCAS(job.err, 0, DEV_ERR_TIMEOUT);
                    }
                    break;
                }
                uint8_t *dst = ring + s * SB;
                const uint32_t cb = (uint32_t)(sn * rs), sbytes = (uint32_t)(sn * ng * 4);
                mbar_expect_tx(&full[s], cb + sbytes);
                bulk_load(dst, job.q[sm_] + (size_t)so * rs, cb, &full[s]);
                bulk_load(dst + RG * rs, job.s[sm_] + (size_t)so * ng, sbytes, &full[s]);
                it++;
                if (++s == NS) {
                    s = 0;
                    ph ^= 1;
                }
            }
            pdl_trigger();
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int k = max(0, it - NS); k < it; k++) mbar_wait(&full[k % NS], (k / NS) & 1, dl2, &no_abort);
        }
        return;
    }
    pdl_wait();
    deadline = global_ns() + (uint64_t)timeout_ns;
    XRegHalf<S> xr;
#pragma unroll
    for (int r = 0; r < S; r++) {
        float4 raw[4];
#pragma unroll
        for (int j = 0; j < 4; j++)
            raw[j] = okc ? __ldg(reinterpret_cast<const float4 *>(job.x + (size_t)r * job.I + (size_t)hc * 16) + j)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        xr.set(r, raw);
    }
    int s = 0;
    uint32_t ph = 0;
    while (next(sm_, so, sn)) {
        if (warp_wait(&full[s], ph, deadline, &abort_flag, lane)) {
            const uint8_t *src = ring + s * SB;
            // this warp's rows of the stage, two at a time
            for (int rr0 = sub; rr0 < sn; rr0 += 2 * G) {
                uint2 qq[2];
                float sc[2];
#pragma unroll
                for (int d = 0; d < 2; d++) {
                    const int rr = rr0 + d * G;
                    const bool ok = okc && rr < sn;
                    qq[d] = ok ? *reinterpret_cast<const uint2 *>(src + rr * rs + hc * 8) : make_uint2(0, 0);
                    sc[d] = ok ? *reinterpret_cast<const float *>(src + RG * rs + (rr * ng + (hc >> gshift)) * 4) : 0.f;
                }
                float dd[2][S];
                xr.template dots<2>(qq, dd);
                // reduce the 2*S values in groups of four
#pragma unroll
                for (int g4 = 0; g4 < (2 * S + 3) / 4; g4++) {
                    float v4[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int idx = g4 * 4 + k;   // idx = d * S + row
                        v4[k] = idx < 2 * S ? dd[idx / S][idx % S] * sc[idx / S] : 0.f;
                    }
                    const float t = warp_sum4(v4[0], v4[1], v4[2], v4[3], lane);
                    const int idx = g4 * 4 + (lane >> 3);
                    if ((lane & 7) == 0 && idx < 2 * S) {
                        const int rr = rr0 + (idx / S) * G;
                        if (rr < sn) red[((job.row_start[sm_] + so + rr - r0) * S + idx % S) * nh + sl] = t;
                    }
                }
            }
        } else if (!abort_flag && lane == 0) {
            abort_flag = 1;
            atomicCAS(job.err, 0, DEV_ERR_TIMEOUT);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == NS) {
            s = 0;
            ph ^= 1;
        }
    }
    pdl_trigger();
    named_sync(1, NCT);
    for (int t = tid; t < (r1 - r0) * S; t += NCT) {
        const int rr = t / S, row = t - rr * S;
        float acc = 0.f;
        for (int k = 0; k < nh; k++) acc += red[(rr * S + row) * nh + k];
        const int rg = r0 + rr;
        int mm = 0;
        while (rg >= job.row_start[mm + 1]) mm++;
        job.y[mm][(size_t)row * job.O[mm] + rg - job.row_start[mm]] = acc;
    }
}

template <int FMT>
cudaError_t slab_gemv_t(const GemvJob &job, int n_sm, int gshift, cudaStream_t st) {
    const int total = job.row_start[job.n];
    const int n_slab = (job.cpr + 31) / 32;
    // CTAs: two per SM, each owning a contiguous block of rows
    int grid = 2 * n_sm;
    int rpc = (total + grid - 1) / grid;
    grid = (total + rpc - 1) / rpc;
    const size_t smem = (staged_words(FMT, job.cpr) + (size_t)n_slab * rpc) * sizeof(float);
    auto kern = slab_gemv_kernel<FMT, 4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kSlabThreads), smem, st, job, rpc, gshift);
}

template <int FMT>
cudaError_t slab_decode_t(const MoeDecodeArgs &a, int grid, size_t smem, int gs_gu, int gs_d, cudaStream_t st) {
    auto kern = moe_decode_slab_kernel<FMT, 4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSlabThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, gs_gu, gs_d);
}

template <int FMT>
cudaError_t slab_decode_occ_t(size_t smem, int *per_sm) {
    auto kern = moe_decode_slab_kernel<FMT, 4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, kSlabThreads, smem);
}

int log2_exact(int v) {
    int k = 0;
    while ((1 << k) < v) k++;
    return (1 << k) == v ? k : -1;
}

}  // namespace

size_t stream_gemv_smem() { return (size_t)kStreamStages * kStreamStageBytes + kStreamRedBytes + 2 * kStreamStages * 8 + 128; }

// rpc: rows per CTA (a multiple of 4); RG: rows per stage; gshift: chunk -> scale index shift
cudaError_t launch_stream_gemv(const GemvJob &job, int rpc, int RG, int gshift, int grid, cudaStream_t st) {
    const size_t smem = stream_gemv_smem();
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3((kStreamConsumerWarps + 1) * 32), smem, st, job, rpc, RG, gshift,
                          2000000000LL);
    };
    // rows of a stage per consumer warp: RG rows over G = warps / slabs-per-row groups
    const int lpr = (job.I + stream_lane_inputs(job.fmt) - 1) / stream_lane_inputs(job.fmt);
    const int G = kStreamConsumerWarps / ((lpr + 31) / 32);
    const int nr = (RG + G - 1) / G;
    constexpr int W = kStreamConsumerWarps;
    switch (job.fmt) {
    case 0: return nr <= 1 ? go(stream_gemv_kernel<W, XRegF32, 1>) : nr <= 2 ? go(stream_gemv_kernel<W, XRegF32, 2>)
                                                                          : go(stream_gemv_kernel<W, XRegF32, 4>);
    case 1: return go(stream_gemv_kernel<W, XRegS1, 4>);
    case 2:
    case 4: return go(stream_gemv_kernel<W, XRegS4, 4>);
    case 3: return go(stream_gemv_kernel<W, XRegS3, 4>);
    case 7: return go(stream_gemv_kernel<W, XRegF8, 4>);
    default: return cudaErrorInvalidValue;
    }
}

// code bytes and inputs of one lane of the streamed S = 1 matvec, per format (0: not streamed)
int stream_lane_bytes(int fmt) {
    return fmt == 0 ? XRegF32::LB : fmt == 1 ? XRegS1::LB : fmt == 3 ? XRegS3::LB : fmt == 7 ? XRegF8::LB : XRegS4::LB;
}
int stream_lane_inputs(int fmt) {
    return fmt == 0 ? XRegF32::NIN : fmt == 1 ? XRegS1::NIN : fmt == 3 ? XRegS3::NIN : fmt == 7 ? XRegF8::NIN
                                                                                       : XRegS4::NIN;
}

size_t stream_gemv_s_smem() {
    return (size_t)kStreamStages * kStreamStageBytes + kStreamGemvRedBytes + 2 * kStreamStages * 8 + 128;
}

cudaError_t launch_stream_gemv_s(const GemvJob &job, int rpc, int RG, int gshift, int grid, cudaStream_t st) {
    const size_t smem = stream_gemv_s_smem();
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3((kStreamConsumerWarps + 1) * 32), smem, st, job, rpc, RG, gshift,
                          2000000000LL);
    };
    switch (job.S) {
    case 2: return go(stream_gemv_s_kernel<kStreamConsumerWarps, 2>);
    case 3: return go(stream_gemv_s_kernel<kStreamConsumerWarps, 3>);
    case 4: return go(stream_gemv_s_kernel<kStreamConsumerWarps, 4>);
    default: return cudaErrorInvalidValue;
    }
}

// gs (fmt=4) usable by the slab kernels: a power-of-two number of 32-input chunks.
bool slab_supported(int fmt, int gs) {
    if (fmt == 3 || fmt == 7) return false;
    if (fmt == 4) return gs % 32 == 0 && log2_exact(gs / 32) >= 0;
    return true;
}

size_t slab_gemv_smem(const GemvJob &job, int n_sm) {
    const int total = job.row_start[job.n];
    int grid = 2 * n_sm;
    const int rpc = (total + grid - 1) / grid;
    return (staged_words(job.fmt, job.cpr) + (size_t)((job.cpr + 31) / 32) * rpc) * sizeof(float);
}

cudaError_t launch_slab_gemv(const GemvJob &job, int n_sm, cudaStream_t st) {
    const int gshift = job.fmt == 4 ? log2_exact(job.gs[0] / 32) : 0;
    switch (job.fmt) {
    case 0: return slab_gemv_t<0>(job, n_sm, gshift, st);
    case 1: return slab_gemv_t<1>(job, n_sm, gshift, st);
    case 2: return slab_gemv_t<2>(job, n_sm, gshift, st);
    case 4: return slab_gemv_t<4>(job, n_sm, gshift, st);
    default: return cudaErrorInvalidValue;
    }
}

// Shared memory of the slab decode kernel for `sb` experts per phase-B batch.
size_t slab_decode_smem(int fmt, int cpr_gu, int cpr_d, int F, int n_slots, int grid_min, int H, int sb) {
    const size_t xlen_gu = staged_words(fmt, cpr_gu), xlen_d = staged_words(fmt, cpr_d);
    const int n_slab_gu = (cpr_gu + 31) / 32, n_slab_d = (cpr_d + 31) / 32;
    const long long pairs_max = (long long)n_slots * F;
    const size_t ppc = (size_t)((pairs_max + grid_min - 1) / grid_min);
    const size_t rpc = (size_t)((H + grid_min - 1) / grid_min);
    const size_t a_part = xlen_gu + (size_t)n_slab_gu * ppc * 2;
    const size_t b_part = (size_t)sb * xlen_d + (size_t)sb * n_slab_d * rpc + rpc;
    return (a_part > b_part ? a_part : b_part) * sizeof(float);
}

cudaError_t slab_decode_occupancy(int fmt, size_t smem, int *per_sm) {
    switch (fmt) {
    case 0: return slab_decode_occ_t<0>(smem, per_sm);
    case 1: return slab_decode_occ_t<1>(smem, per_sm);
    case 2: return slab_decode_occ_t<2>(smem, per_sm);
    case 4: return slab_decode_occ_t<4>(smem, per_sm);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_slab_decode(const MoeDecodeArgs &a, int fmt, int grid, size_t smem, int gs_gu, int gs_d,
                               cudaStream_t st) {
    const int sh_gu = fmt == 4 ? log2_exact(gs_gu / 32) : 0, sh_d = fmt == 4 ? log2_exact(gs_d / 32) : 0;
    switch (fmt) {
    case 0: return slab_decode_t<0>(a, grid, smem, sh_gu, sh_d, st);
    case 1: return slab_decode_t<1>(a, grid, smem, sh_gu, sh_d, st);
    case 2: return slab_decode_t<2>(a, grid, smem, sh_gu, sh_d, st);
    case 4: return slab_decode_t<4>(a, grid, smem, sh_gu, sh_d, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace coli
