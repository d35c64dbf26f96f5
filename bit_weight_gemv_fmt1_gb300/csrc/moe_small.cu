// moe_small.cu -- the prefill expert block's products for experts that few
// rows are routed to, on the tensor cores as register-operand mma.sync
// (colibri-strix commit log, "metal: batched moe_block"; the block is
// gate/up GEMV, SiLU * mul, down GEMV per routed (row, expert) pair).
//
// The routing kernel lists the rows of every expert with at most a few rows
// as groups of up to four consecutive rows (positions p0 .. p0 + n - 1 of the
// expert-sorted row order).  One launch multiplies every group by the rows of
// one or two of its expert's matrices:
//   gate|up: gu[p][j] = gate[j] . x[token(p)],  gu[p][F + j] = up[j] . x[token(p)]
//   down:    slot_out[p][o] = down[o] . h[p],  h[p][j] = silu(gu[p][j]) gu[p][F + j]
// (h in f32 exactly as the plane kernel of the large experts forms it).
//
// Arithmetic: the subnormal-code products of mma_int4.cuh with the four rows
// of a group in the eight B columns: column 2 t holds row t's hi half,
// column 2 t + 1 its lo half, each row with its own power-of-two scale, so
// one mma multiplies a 16 x 16 code tile by all four rows and thread quad
// lane t holds row t's sums.  Each expert's matrices are read once per group.
//
// Roles as in gemv_mma.cu: warps 0..15 consume, warp 16 copies stages of
// NT 16-row tiles of one matrix into three shared-memory slots, warp 17 sums
// the warps' shares of each (matrix row, group row) in warp order and writes
// the result.  CTA c owns a contiguous range of (group, matrix, row block)
// items, so a warp rebuilds its B fragments only when the group changes.
// Every wait is bounded; on expiry the kernel records DEV_ERR_TIMEOUT.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "coli_internal.cuh"
#include "mbarrier.cuh"
#include "mma_int4.cuh"

namespace coli {

namespace {

constexpr int kSmThreads = (kMdWarps + 2) * 32;
constexpr int kSmSlots = 3;
constexpr int kSmRedT = 17;                   // floats per (stage row, group row): 16 warps, padded
constexpr int kSmStg = kMd4Stg;               // staging area of one round
constexpr uint32_t kSmNapE = 64, kSmNapP = 64;

// Item k: d.x = group, d.y = matrix (0 or 1 of the call), d.z = first row, d.w = rows.
__device__ __forceinline__ int4 sm_item(const SmArgs &a, int k) {
    const int per = a.n_mat * a.nb;
    const int g = k / per, r = k - g * per;
    const int m = r / a.nb, b = r - m * a.nb;
    const int r0 = b * 16 * a.nt;
    return make_int4(g, m, r0, min(16 * a.nt, a.O - r0));
}

// The four values lane `lane` holds for round r of group row p (inputs
// 64 (q0 + seg) + 4 (lane % 16) + 0..3, seg = 2 r + lane / 16, as md_load4):
// x of the row's token (gate|up) or h = silu(g) u of the row (down); zero for
// segments past the warp's and inputs past I.
template <bool DOWN>
__device__ __forceinline__ float4 sm_load4(const SmArgs &a, int p, int q0, int nq, int r, int lane) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int seg = 2 * r + (lane >> 4);
    if (seg < nq) {
        const int i0 = (q0 + seg) * 64 + 4 * (lane & 15);
        if (!DOWN) {
            const float *xr = a.x + (size_t)(a.order[p] / a.K) * a.ldx;
#pragma unroll
            for (int j = 0; j < 4; j++)
                if (i0 + j < a.I) v[j] = __ldg(xr + i0 + j);
        } else {
            const float *gr = a.gu + (size_t)p * 2 * a.I;
#pragma unroll
            for (int j = 0; j < 4; j++)
                if (i0 + j < a.I) {
                    const float g = __ldcg(gr + i0 + j), u = __ldcg(gr + a.I + i0 + j);
                    v[j] = g / (1.0f + expf(-g)) * u;
                }
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

// SEG: segments per warp (compile-time bound), NT: 16-row tiles per stage,
// DOWN: the down product (else gate|up).
template <bool GROUPED, int GSH, int SEG, int NT, bool DOWN>
__global__ void __launch_bounds__(kSmThreads, 1) moe_small_kernel(const SmArgs a) {
    static_assert(SEG % 2 == 0 && SEG <= kMdSegMax, "segments per warp");
    extern __shared__ uint8_t sraw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    float *red = reinterpret_cast<float *>(base + a.off_red);   // [slot][stage row][group row][kSmRedT]
    uint8_t *stg_all = base + a.off_stg;                         // [warp][kSmStg]
    int4 *desc = reinterpret_cast<int4 *>(base + a.off_bar);    // [slot]
    uint64_t *full = reinterpret_cast<uint64_t *>(desc + kSmSlots);
    uint64_t *empty = full + kSmSlots;
    uint64_t *redfull = empty + kSmSlots;
    __shared__ volatile int abort_flag;
    __shared__ float4 s_cf[kMdWarps][kMdSegMax + 1][4];   // chain starts per segment and group row; their sums
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int SB = a.slot_bytes;
    const uint64_t deadline = global_ns() + (uint64_t)a.timeout_ns;
    const int n_groups = *a.n_sg;
    const int total = n_groups * a.n_mat * a.nb;
    const int G = gridDim.x;
    const int k0 = (int)((long long)total * blockIdx.x / G), k1 = (int)((long long)total * (blockIdx.x + 1) / G);
    const int nk = k1 - k0;
    const int mat0 = DOWN ? 2 : 0;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < kSmSlots; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kMdWarps);
            mbar_init(&redfull[i], kMdWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (nk <= 0) return;
    auto fail = [&]() {
        if (!abort_flag) {
            abort_flag = 1;
            atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
        }
    };

    if (warp == kMdWarps) {
        // ---------------- producer: item i of the CTA into slot i % kSmSlots
        if (lane == 0) {
            const int rs = a.rs;
            int cg = -1, cm = -1;
            const uint8_t *q = nullptr;
            const float *sp = nullptr;
            int i = 0;
            for (; i < nk; i++) {
                const int s = i % kSmSlots;
                if (i >= kSmSlots && !md_wait1(&empty[s], ((i / kSmSlots) & 1) ^ 1, deadline, &abort_flag, kSmNapP)) {
                    fail();
                    break;
                }
                const int4 d = sm_item(a, k0 + i);
                if (d.x != cg || d.y != cm) {   // the group's expert matrix
                    cg = d.x;
                    cm = d.y;
                    const MatDesc &M = a.table[a.sg_e[cg]].m[mat0 + cm];
                    q = M.q;
                    sp = M.s;
                }
                desc[s] = d;
                uint8_t *dst = base + (size_t)s * SB;
                uint32_t tx = 0;
                int cnt[4];
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    cnt[b] = max(0, min(4 * NT, d.w - 4 * NT * b));
                    tx += (uint32_t)cnt[b] * (uint32_t)(rs + (GROUPED ? 4 * a.ng : 0));
                }
                mbar_expect_tx(&full[s], tx);
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    if (cnt[b] == 0) continue;
                    const size_t r = (size_t)d.z + (size_t)(4 * NT * b);
                    bulk_load(dst + b * (a.bs + 32), q + r * rs, (uint32_t)(cnt[b] * rs), &full[s]);
                    if (GROUPED)
                        bulk_load(dst + a.so + b * a.ss, sp + r * a.ng, (uint32_t)(cnt[b] * a.ng * 4), &full[s]);
                }
            }
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int qq = max(0, i - kSmSlots); qq < i; qq++)
                mbar_wait(&full[qq % kSmSlots], (qq / kSmSlots) & 1, dl2, &no_abort);
        }
        return;
    }

    if (warp == kMdWarps + 1) {
        // ---------------- epilogue: the 16 warp shares of each (stage row, group row) in warp order
        bool ok = true;
        int cg = -1, cm = -1;
        const float *sp = nullptr;
        for (int i = 0; i < nk; i++) {
            const int s = i % kSmSlots;
            const uint32_t par = (uint32_t)((i / kSmSlots) & 1);
            if (!md_wait(&full[s], par, deadline, &abort_flag, kSmNapE) ||
                !md_wait(&redfull[s], par, deadline, &abort_flag, kSmNapE)) {
                ok = false;
                break;
            }
            const int4 d = desc[s];
            if (!GROUPED && (d.x != cg || d.y != cm)) {
                cg = d.x;
                cm = d.y;
                sp = a.table[a.sg_e[cg]].m[mat0 + cm].s;
            }
            const int n = a.sg_n[d.x], p0 = a.sg_p0[d.x];
            const float *rd = red + s * (16 * NT * 4 * kSmRedT);
            float v[2 * NT];
#pragma unroll
            for (int u = 0; u < 2 * NT; u++) {
                const int idx = lane + 32 * u;   // (stage row, group row) = (idx / 4, idx % 4)
                float acc = 0.f;
                if (idx / 4 < d.w && (idx & 3) < n) {
                    const float *r = rd + idx * kSmRedT;
#pragma unroll
                    for (int w = 0; w < kMdWarps; w++) acc += r[w];
                }
                v[u] = acc;
            }
            __syncwarp();
            if (lane == 0) md_release(&empty[s]);
#pragma unroll
            for (int u = 0; u < 2 * NT; u++) {
                const int idx = lane + 32 * u, rr = idx / 4, t = idx & 3;
                if (rr < d.w && t < n) {
                    const int o = d.z + rr;
                    float val = v[u];
                    if (!GROUPED) val *= __ldg(sp + o);
                    a.out[(size_t)(p0 + t) * a.ldo + (size_t)d.y * a.O + o] = val;
                }
            }
        }
        if (!ok && lane == 0) fail();
        return;
    }

    // ---------------- consumers
    const int q0 = warp * a.spw, nq = min(a.spw, a.nseg - q0);
    constexpr int NRD = SEG / 2;
    const int g4 = lane >> 2, t4 = lane & 3;   // mma fragment row group and quad lane (= group row)
    const int blk = g4 & 3, rib = g4 >> 2;
    const uint32_t stg = smem_addr(stg_all + (size_t)warp * kSmStg);
    const uint32_t rs2 = 2u * (uint32_t)a.rs, sr2 = 8u * (uint32_t)a.ng;
    const uint32_t cofs = (uint32_t)(blk * (a.bs + 32) + rib * a.rs + 32 * q0 + 8 * t4);
    const uint32_t sofs = (uint32_t)(a.so + blk * a.ss + rib * a.ng * 4 + (q0 >> GSH) * 4);
    const uint32_t cfs = smem_addr(&s_cf[warp][0][t4]);
    const uint32_t ring_s = smem_addr(base);
    uint32_t bf[SEG][8];
    float un = 0.f;
    int cur = -1;
    for (int i = 0; i < nk; i++) {
        const int s = i % kSmSlots;
        if (!md_wait(&full[s], (uint32_t)((i / kSmSlots) & 1), deadline, &abort_flag, 0)) {
            if (lane == 0) fail();
            break;
        }
        const int4 d = desc[s];
        if (d.x != cur) {
            // a new group: B fragments of its rows (zero columns past n)
            cur = d.x;
            const int n = a.sg_n[cur], p0 = a.sg_p0[cur];
            float4 ld[4][NRD];
            MdScale sc[4];
#pragma unroll
            for (int t = 0; t < 4; t++) {
#pragma unroll
                for (int r = 0; r < NRD; r++)
                    ld[t][r] = t < n ? sm_load4<DOWN>(a, p0 + t, q0, nq, r, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
                sc[t] = md_scale<NRD>(ld[t]);
            }
            un = (t4 == 0 ? sc[0].unscale : t4 == 1 ? sc[1].unscale : t4 == 2 ? sc[2].unscale : sc[3].unscale) *
                 0x1p24f;
            float4 cft = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < NRD; r++) {
#pragma unroll
                for (int t = 0; t < 4; t++) md4_frag_store(ld[t][r], sc[t], lane, t, stg);
                __syncwarp();
                md4_frag_load(nq - 2 * r, lane, stg, bf[2 * r], bf[2 * r + 1]);
                __syncwarp();   // the staging area may be rewritten after this
                float4 c0, c1;
                md_frag_starts(bf[2 * r], bf[2 * r + 1], c0, c1);
                // quad lane t of row group 0 holds group row t's (hi, lo) starts
                if (g4 == 0) {
                    s_cf[warp][2 * r][t4] = c0;
                    s_cf[warp][2 * r + 1][t4] = c1;
                }
                cft.x += c0.x + c1.x;
                cft.y += c0.y + c1.y;
                cft.z += c0.z + c1.z;
                cft.w += c0.w + c1.w;
            }
            if (g4 == 0) s_cf[warp][kMdSegMax][t4] = cft;
            __syncwarp();
        }
        const uint32_t sb = ring_s + (uint32_t)(s * SB);
        // tile row m = g, g + 8 of tile T is stage row 4 NT (m % 4) + 4 T + m / 4
        float *rw = red + s * (16 * NT * 4 * kSmRedT) + ((blk * 4 * NT + rib) * 4 + t4) * kSmRedT + warp;
#pragma unroll
        for (int T = 0; T < NT; T++) {
            float y[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t tc = sb + cofs + (uint32_t)(4 * T * a.rs), ts = sb + sofs + (uint32_t)(4 * T * a.ng * 4);
            if (nq == SEG)
                md_tileA<GROUPED, GSH, true, SEG, 4 * 16>(y, tc, rs2, cfs, ts, sr2, nq, bf);
            else if (nq > 0)
                md_tileA<GROUPED, GSH, false, SEG, 4 * 16>(y, tc, rs2, cfs, ts, sr2, nq, bf);
            const bool on = nq > 0;
            rw[4 * T * 4 * kSmRedT] = on ? fmaf(y[1], 0x1p-11f, y[0]) * un : 0.f;
            rw[(4 * T + 2) * 4 * kSmRedT] = on ? fmaf(y[3], 0x1p-11f, y[2]) * un : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&redfull[s]);
    }
}

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

int log2_exact(int v) {
    int k = 0;
    while ((1 << k) < v) k++;
    return (1 << k) == v ? k : -1;
}

template <bool GROUPED, int GSH, int SEG, int NT, bool DOWN>
cudaError_t sm_go(const SmArgs &a, int grid, size_t smem, cudaStream_t st) {
    auto kern = moe_small_kernel<GROUPED, GSH, SEG, NT, DOWN>;
    static std::mutex mu;
    static size_t done = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (done < smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            done = smem;
        }
    }
    kern<<<grid, kSmThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

// Geometry of the small-group products of one role: gate|up (two matrices of
// O = F rows over I = H inputs) or down (one matrix of O = H rows over
// I = F inputs).  fmt 2, or fmt 4 with gs 64 or 128 and a multiple of 4 scales
// per row; I a multiple of 64 and at most 16 * 6 * 64.
bool sm_plan(bool down, int fmt, int gs, int I, int O, int rs, int ng, size_t smem_max, SmArgs *a, size_t *smem) {
    if (fmt != 2 && fmt != 4) return false;
    if (I < 64 || I % 64 != 0 || O < 1 || rs != I / 2) return false;
    const bool grouped = fmt == 4;
    int gsh = 0;
    if (grouped) {
        if (gs != 64 && gs != 128) return false;
        gsh = log2_exact(gs / 64);
        if (ng % 4 != 0 || ng * gs != I) return false;
    }
    const int nseg = I / 64, gm = 1 << gsh;
    const int spw = ((nseg + kMdWarps - 1) / kMdWarps + gm - 1) / gm * gm;
    if (spw > kMdSegMax) return false;
    // one tile per stage for rows of more than 2048 inputs, else two
    const int nt = spw <= 2 ? 2 : 1;
    memset(a, 0, sizeof *a);
    const size_t bs = round_up((size_t)4 * nt * rs + 32, 128), so = 4 * bs + 128;
    const size_t ss = grouped ? (size_t)4 * nt * ng * 4 + 16 : 0;
    const size_t SB = round_up(so + 4 * ss, 128);
    const size_t off_red = kSmSlots * SB;
    const size_t off_stg = round_up(off_red + (size_t)kSmSlots * 16 * nt * 4 * kSmRedT * 4, 128);
    const size_t off_bar = off_stg + (size_t)kMdWarps * kSmStg;
    const size_t total = off_bar + kSmSlots * 16 + 3 * kSmSlots * 8 + 128;   // + alignment slack
    if (total + 8 * 1024 > smem_max) return false;   // static shared memory: about 7 KB
    a->down = down;
    a->fmt = fmt;
    a->I = I;
    a->O = O;
    a->rs = rs;
    a->ng = grouped ? ng : 0;
    a->gsh = gsh;
    a->nseg = nseg;
    a->spw = spw;
    a->nt = nt;
    a->n_mat = down ? 1 : 2;
    a->nb = (O + 16 * nt - 1) / (16 * nt);
    a->bs = (int)bs;
    a->so = (int)so;
    a->ss = (int)ss;
    a->slot_bytes = (int)SB;
    a->off_red = (int)off_red;
    a->off_stg = (int)off_stg;
    a->off_bar = (int)off_bar;
    a->timeout_ns = 2000000000LL;
    *smem = total;
    return true;
}

template <bool DOWN>
cudaError_t sm_launch_role(const SmArgs &a, int grid, size_t smem, cudaStream_t st) {
    const bool g = a.fmt == 4;
    if (a.nt == 1) {
        if (!g) return sm_go<false, 0, kMdSegMax, 1, DOWN>(a, grid, smem, st);
        return a.gsh == 0 ? sm_go<true, 0, kMdSegMax, 1, DOWN>(a, grid, smem, st)
                          : sm_go<true, 1, kMdSegMax, 1, DOWN>(a, grid, smem, st);
    }
    if (a.nt != 2 || a.spw > 2) return cudaErrorInvalidValue;
    if (!g) return sm_go<false, 0, 2, 2, DOWN>(a, grid, smem, st);
    return a.gsh == 0 ? sm_go<true, 0, 2, 2, DOWN>(a, grid, smem, st) : sm_go<true, 1, 2, 2, DOWN>(a, grid, smem, st);
}

cudaError_t launch_moe_small(const SmArgs &a, int grid, size_t smem, cudaStream_t st) {
    return a.down ? sm_launch_role<true>(a, grid, smem, st) : sm_launch_role<false>(a, grid, smem, st);
}

}  // namespace coli
