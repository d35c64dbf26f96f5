// gemv_mma.cu -- the streamed S <= 4 matvec y = W x for int4 weights (fmt 2,
// and fmt 4 with groups of 64 or 128 inputs) on the tensor cores, for calls
// large enough that streaming the weights dominates (coli_matmul and
// coli_matmul_multi at S = 1; the pages' mm_gemv / matmul_i4_grouped).
//
// The rows of all matrices of a call form one list of stages; a stage is NT
// tiles of 16 consecutive rows of one matrix.  CTA c takes stages c, c + G
// and c + 2 G (the ones it can prefetch before the previous kernel ends), then
// claims the rest one at a time from a counter in device memory, so that the
// CTAs finish together however the bandwidth falls among them; the last CTA
// out clears the counter for the next call.  Warps 0..15 consume, warp 16 produces (its lane 0 copies
// each stage's rows and row scales into one of three shared-memory slots with
// bulk copies), warp 17 finishes a stage: it sums the consumer warps' shares
// of each row in warp order and writes y.  The dot products are the
// subnormal-code mma.sync products of mma_int4.cuh: warp w owns the 64-input
// segments [w S, (w + 1) S) of every row and builds their B fragments from x
// once per call.  For S = 1 the B operand carries x's hi and lo halves in two
// columns; for S = 2..4 every row of x has its own pair of columns
// (md4_frag_store), so one mma serves all S rows.
//
// Back-to-back calls: every CTA lets the next kernel in the stream launch as
// soon as it starts (griddepcontrol.launch_dependents; one CTA fills an SM, so
// the next kernel's CTAs take SMs only as this kernel frees them), and the
// producer issues its first stages (weights only, which no kernel writes)
// before waiting for the previous kernel (griddepcontrol.wait); x is read and
// y written only after that wait.
// Every wait is bounded; on expiry the kernel records DEV_ERR_TIMEOUT.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>

#include "coli_internal.cuh"
#include "mbarrier.cuh"
#include "mma_int4.cuh"

namespace coli {

namespace {

constexpr int kGmThreads = (kMdWarps + 2) * 32;
constexpr int kGmSlots = 3;
constexpr int kGmRedB = 20;                  // partial sums of a stage row (S = 1): 16 warps, padded
constexpr int kGmRedT = 17;                  // partial sums of a (stage row, x row) (S > 1): 16 warps, padded
constexpr int kGmStageMax = 48;              // rows of a stage (NT <= 3 tiles)
// floats of a slot's partial sums: rows x (20, or 4 x 17)
__host__ __device__ constexpr int gm_red_row(int ntok) { return ntok == 1 ? kGmRedB : 4 * kGmRedT; }
constexpr uint32_t kGmNapE = 64, kGmNapP = 64;

// Stage k: d.x = matrix, d.y = first row, d.z = rows (d.z = 0: no stage, the end).
__device__ __forceinline__ int4 gm_stage(const GmArgs &a, int k) {
    int m = 0;
    while (k >= a.stage_start[m + 1]) m++;
    const int r0 = (k - a.stage_start[m]) * 16 * a.nt;
    return make_int4(m, r0, min(16 * a.nt, a.O[m] - r0), 0);
}

// SEG: segments per warp (compile-time bound), NT: 16-row tiles per stage,
// NTOK: rows of x per B operand (1, or 4 for S = 2..4).
template <bool GROUPED, int GSH, int SEG, int NT, int NTOK>
__global__ void __launch_bounds__(kGmThreads, 1) gemv_mma_kernel(const GmArgs a) {
    static_assert(SEG % 2 == 0 && SEG <= kMdSegMax && 16 * NT <= kGmStageMax, "stage geometry");
    static_assert(NTOK == 1 || NTOK == 4, "rows per B operand");
    constexpr int RROW = gm_red_row(NTOK), RSLOT = 16 * NT * RROW;
    extern __shared__ uint8_t sraw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    float *red = reinterpret_cast<float *>(base + a.off_red);   // [slot][row][RROW]
    int4 *desc = reinterpret_cast<int4 *>(base + a.off_bar);   // [slot]: the stage it holds
    uint64_t *full = reinterpret_cast<uint64_t *>(desc + kGmSlots);
    uint64_t *empty = full + kGmSlots;
    uint64_t *redfull = empty + kGmSlots;
    __shared__ volatile int abort_flag;
    // chain starts of each warp's segments (per x row), their sum
    __shared__ float4 s_cf[kMdWarps][kMdSegMax + 1][NTOK];
    // B-fragment staging of each consumer warp: S = 1, one area per round and a
    // zero row; S > 1, one four-row area
    __shared__ __align__(16) uint8_t s_stg[kMdWarps][NTOK == 1 ? (SEG / 2) * kMdStgZero + 16 : kMd4Stg];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int SB = a.slot_bytes;
    uint64_t deadline = global_ns() + (uint64_t)a.timeout_ns;
    const int S = a.stage_start[a.n];
    const int G = gridDim.x;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < kGmSlots; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kMdWarps);
            mbar_init(&redfull[i], kMdWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // one CTA fills an SM, so the next kernel's CTAs cannot sit beside this
    // one: let it launch now, and each of its CTAs starts (and prefetches its
    // weights) on the first SM this kernel frees
    pdl_trigger();
    auto fail = [&]() {
        if (!abort_flag) {
            abort_flag = 1;
            atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
        }
    };

    if (warp == kMdWarps) {
        // ---------------- producer: stage i of the CTA into slot i % kGmSlots; an
        // end marker (a descriptor with no rows, no bytes) after the last one
        if (lane == 0) {
            const int rs = a.rs;
            int i = 0;
            bool ok = true;
            while (true) {
                const int s = i % kGmSlots;
                int k;
                if (i < kGmSlots) {
                    k = (int)blockIdx.x + G * i;
                } else {
                    if (i == kGmSlots) {
                        // the prefetched round is issued: the rest needs the
                        // previous kernel to be complete (the shared counter)
                        pdl_wait();
                        deadline = global_ns() + (uint64_t)a.timeout_ns;
                    }
                    k = 3 * G + (int)atomicAdd(a.ctr, 1u);
                }
                if (i >= kGmSlots && !md_wait1(&empty[s], ((i / kGmSlots) & 1) ^ 1, deadline, &abort_flag, kGmNapP)) {
                    fail();
                    ok = false;
                    break;
                }
                if (k >= S) {
                    desc[s] = make_int4(0, 0, 0, 0);
                    mbar_arrive(&full[s]);   // end marker
                    i++;
                    break;
                }
                const int4 d = gm_stage(a, k);
                desc[s] = d;
                uint8_t *dst = base + (size_t)s * SB;
                uint32_t tx = 0;
                int cnt[4];
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    cnt[b] = max(0, min(4 * NT, d.z - 4 * NT * b));
                    tx += (uint32_t)cnt[b] * (uint32_t)(rs + (GROUPED ? 4 * a.ng : 0));
                }
                mbar_expect_tx(&full[s], tx);
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    if (cnt[b] == 0) continue;
                    const size_t r = (size_t)d.y + (size_t)(4 * NT * b);
                    bulk_load(dst + b * (a.bs + 32), a.q[d.x] + r * rs, (uint32_t)(cnt[b] * rs), &full[s]);
                    if (GROUPED)
                        bulk_load(dst + a.so + b * a.ss, a.s[d.x] + r * a.ng, (uint32_t)(cnt[b] * a.ng * 4), &full[s]);
                }
                i++;
            }
            if (i <= kGmSlots) pdl_wait();
            // every copy issued has landed before the CTA may exit
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int q = max(0, i - kGmSlots); q < i; q++) mbar_wait(&full[q % kGmSlots], (q / kGmSlots) & 1, dl2, &no_abort);
            (void)ok;
            // the last CTA out clears the stage counter and itself for the next call
            __threadfence();
            if (atomicAdd(a.ctr + 1, 1u) == (unsigned)G - 1) {
                a.ctr[0] = 0u;
                a.ctr[1] = 0u;
                __threadfence();
            }
        }
        return;
    }

    if (warp == kMdWarps + 1) {
        // ---------------- epilogue: each stage row's 16 warp shares in warp order -> y
        pdl_wait();
        deadline = global_ns() + (uint64_t)a.timeout_ns;
        bool ok = true;
        for (int i = 0;; i++) {
            const int s = i % kGmSlots;
            const uint32_t par = (uint32_t)((i / kGmSlots) & 1);
            if (!md_wait(&full[s], par, deadline, &abort_flag, kGmNapE)) {
                ok = false;
                break;
            }
            const int4 d = desc[s];
            if (d.z == 0) break;
            if (!md_wait(&redfull[s], par, deadline, &abort_flag, kGmNapE)) {
                ok = false;
                break;
            }
            const float *rd = red + s * RSLOT;
            if (NTOK == 1) {
                float v[2] = {0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int rr = lane + 32 * h;
                    if (rr < d.z) {
                        const float4 *r4 = reinterpret_cast<const float4 *>(rd + rr * kGmRedB);
#pragma unroll
                        for (int w4 = 0; w4 < kMdWarps / 4; w4++) {
                            const float4 q = r4[w4];
                            v[h] += q.x;
                            v[h] += q.y;
                            v[h] += q.z;
                            v[h] += q.w;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) md_release(&empty[s]);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int rr = lane + 32 * h;
                    if (rr < d.z) {
                        const int o = d.y + rr;
                        if (!GROUPED) v[h] *= __ldg(a.s[d.x] + o);
                        a.y[d.x][o] = v[h];
                    }
                }
            } else {
                // (stage row, x row) = (idx / 4, idx % 4)
                float v[2 * NT];
#pragma unroll
                for (int u = 0; u < 2 * NT; u++) {
                    const int idx = lane + 32 * u;
                    float acc = 0.f;
                    if (idx / 4 < d.z && (idx & 3) < a.S) {
                        const float *r = rd + idx * kGmRedT;
#pragma unroll
                        for (int w = 0; w < kMdWarps; w++) acc += r[w];
                    }
                    v[u] = acc;
                }
                __syncwarp();
                if (lane == 0) md_release(&empty[s]);
#pragma unroll
                for (int u = 0; u < 2 * NT; u++) {
                    const int idx = lane + 32 * u, rr = idx / 4, tt = idx & 3;
                    if (rr < d.z && tt < a.S) {
                        const int o = d.y + rr;
                        float val = v[u];
                        if (!GROUPED) val *= __ldg(a.s[d.x] + o);
                        a.y[d.x][(size_t)tt * a.O[d.x] + o] = val;
                    }
                }
            }
        }
        if (!ok && lane == 0) fail();
        return;
    }

    // ---------------- consumers
    pdl_wait();
    deadline = global_ns() + (uint64_t)a.timeout_ns;
    const int q0 = warp * a.spw, nq = min(a.spw, a.nseg - q0);
    constexpr int NRD = (SEG + 1) / 2;   // rounds of two segments
    uint32_t bf[SEG][8];
    float un = 0.f;
    const int g = lane >> 2, t = lane & 3;
    if (NTOK == 4) {
        // one pair of B columns per row of x (zero columns past S)
        float4 ld[4][NRD];
        MdScale sc[4];
#pragma unroll
        for (int tt = 0; tt < 4; tt++) {
#pragma unroll
            for (int r = 0; r < NRD; r++)
                ld[tt][r] = tt < a.S ? md_load4(a.x + (size_t)tt * a.I, a.I, q0, nq, r, lane, false)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            sc[tt] = md_scale<NRD>(ld[tt]);
        }
        un = (t == 0 ? sc[0].unscale : t == 1 ? sc[1].unscale : t == 2 ? sc[2].unscale : sc[3].unscale) * 0x1p24f;
        const uint32_t stg = smem_addr(&s_stg[warp][0]);
        float4 cft = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < NRD; r++) {
#pragma unroll
            for (int tt = 0; tt < 4; tt++) md4_frag_store(ld[tt][r], sc[tt], lane, tt, stg);
            __syncwarp();
            md4_frag_load(nq - 2 * r, lane, stg, bf[2 * r], bf[2 * r + 1]);
            __syncwarp();   // the staging area may be rewritten after this
            float4 c0, c1;
            md_frag_starts(bf[2 * r], bf[2 * r + 1], c0, c1);
            // quad lane t of row group 0 holds x row t's (hi, lo) starts
            if (g == 0) {
                s_cf[warp][2 * r][t] = c0;
                s_cf[warp][2 * r + 1][t] = c1;
            }
            cft.x += c0.x + c1.x;
            cft.y += c0.y + c1.y;
            cft.z += c0.z + c1.z;
            cft.w += c0.w + c1.w;
        }
        if (g == 0) s_cf[warp][kMdSegMax][t] = cft;
        __syncwarp();
    } else {
        float4 ld[NRD];
#pragma unroll
        for (int r = 0; r < NRD; r++) ld[r] = md_load4(a.x, a.I, q0, nq, r, lane, false);
        uint32_t *zr = reinterpret_cast<uint32_t *>(&s_stg[warp][NRD * kMdStgZero]);
        if (lane < 4) zr[lane] = 0u;
        __syncwarp();
        const uint32_t stg = smem_addr(&s_stg[warp][0]), zrow = smem_addr(zr);
        const MdScale sc = md_scale<NRD>(ld);
        un = sc.unscale * 0x1p24f;
        float4 cft = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 cs[SEG];
        md_frags_n<NRD>(ld, sc, nq, lane, stg, zrow, bf, cs);
#pragma unroll
        for (int r = 0; r < NRD; r++) {
            const float4 c0 = cs[2 * r], c1 = cs[2 * r + 1];
            if (lane == 0) {
                s_cf[warp][2 * r][0] = c0;
                s_cf[warp][2 * r + 1][0] = c1;
            }
            cft.x += c0.x + c1.x;
            cft.y += c0.y + c1.y;
            cft.z += c0.z + c1.z;
            cft.w += c0.w + c1.w;
        }
        if (lane == 0) s_cf[warp][kMdSegMax][0] = cft;   // per-row formats: the whole row's chain start
        __syncwarp();
    }
    const uint32_t ring_s = smem_addr(base);
    const int blk = g & 3, rib = g >> 2;   // block and row in block of tile row g (row g + 8: rib + 2)
    const uint32_t rs2 = 2u * (uint32_t)a.rs, sr2 = 8u * (uint32_t)a.ng;
    const uint32_t cofs = (uint32_t)(blk * (a.bs + 32) + rib * a.rs + 32 * q0 + 8 * t);
    const uint32_t sofs = (uint32_t)(a.so + blk * a.ss + rib * a.ng * 4 + (q0 >> GSH) * 4);
    const uint32_t cfs = smem_addr(&s_cf[warp][0][NTOK == 4 ? t : 0]);
    const bool fullw = nq == SEG;
    for (int i = 0;; i++) {
        const int s = i % kGmSlots;
        if (!md_wait(&full[s], (uint32_t)((i / kGmSlots) & 1), deadline, &abort_flag, 0)) {
            if (lane == 0) fail();
            break;
        }
        if (desc[s].z == 0) break;   // end marker
        const uint32_t sb = ring_s + (uint32_t)(s * SB);
        // tile row m = g, g + 8 of tile T is stage row 4 NT (m % 4) + 4 T + m / 4
        // S > 1: x row t's share at [row][t][warp]
        float *rw = red + s * RSLOT + (blk * 4 * NT + rib) * RROW + (NTOK == 4 ? t * kGmRedT : 0) + warp;
#pragma unroll
        for (int T = 0; T < NT; T++) {
            float y[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t tc = sb + cofs + (uint32_t)(4 * T * a.rs), ts = sb + sofs + (uint32_t)(4 * T * a.ng * 4);
            if (fullw)
                md_tileA<GROUPED, GSH, true, SEG, 16 * NTOK>(y, tc, rs2, cfs, ts, sr2, nq, bf);
            else if (nq > 0)
                md_tileA<GROUPED, GSH, false, SEG, 16 * NTOK>(y, tc, rs2, cfs, ts, sr2, nq, bf);
            if (NTOK == 4 || t == 0) {
                const bool on = nq > 0;
                rw[4 * T * RROW] = on ? fmaf(y[1], 0x1p-11f, y[0]) * un : 0.f;
                rw[(4 * T + 2) * RROW] = on ? fmaf(y[3], 0x1p-11f, y[2]) * un : 0.f;
            }
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

template <bool GROUPED, int GSH, int SEG, int NT, int NTOK>
cudaError_t gm_go(const GmArgs &a, int grid, size_t smem, cudaStream_t st) {
    auto kern = gemv_mma_kernel<GROUPED, GSH, SEG, NT, NTOK>;
    // the shared-memory attribute is set once per kernel and size
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
    return launch_pdl(kern, dim3(grid), dim3(kGmThreads), smem, st, a);
}

}  // namespace

// Geometry of the tensor-core streamed matvec for the n matrices of a call
// (one format and row length; fmt=4: one gs of 64 or 128 inputs and a
// multiple of 4 scales per row) and S = 1..4 rows of x.  I a multiple of 64
// and at most 16 * 6 * 64.
bool gm_plan(int fmt, int gs, int I, int rs, int ng, int n, const int *O, int S, int n_sm, size_t smem_max,
             GmArgs *a, size_t *smem, int *grid) {
    if (fmt != 2 && fmt != 4) return false;
    if (S < 1 || S > 4) return false;
    if (n < 1 || n > GemvJob::MAXM || I < 64 || I % 64 != 0 || n_sm < 1) return false;
    const bool grouped = fmt == 4;
    int gsh = 0;
    if (grouped) {
        if (gs != 64 && gs != 128) return false;
        gsh = log2_exact(gs / 64);
        if (ng % 4 != 0 || ng * gs != I) return false;
    }
    if (rs != I / 2) return false;
    const int nseg = I / 64, gm = 1 << gsh;
    const int spw = ((nseg + kMdWarps - 1) / kMdWarps + gm - 1) / gm * gm;
    if (spw > kMdSegMax) return false;
    // tiles per stage: for rows of up to 2048 inputs (two segments per warp)
    // three (S = 1) or two (S > 1: four times the partial sums), so that a
    // stage is about as large as one 16-row tile of 6144 inputs
    const int ntok = S == 1 ? 1 : 4;
    const int nt = spw <= 2 ? (S == 1 ? 3 : 2) : 1;
    memset(a, 0, sizeof *a);
    a->n = n;
    a->stage_start[0] = 0;
    for (int m = 0; m < n; m++) {
        if (O[m] < 1) return false;
        a->O[m] = O[m];
        a->stage_start[m + 1] = a->stage_start[m] + (O[m] + 16 * nt - 1) / (16 * nt);
    }
    const size_t bs = round_up((size_t)4 * nt * rs + 32, 128), so = 4 * bs + 128;
    const size_t ss = grouped ? (size_t)4 * nt * ng * 4 + 16 : 0;
    const size_t SB = round_up(so + 4 * ss, 128);
    const size_t off_red = kGmSlots * SB;
    const size_t off_bar = off_red + (size_t)kGmSlots * 16 * nt * gm_red_row(ntok) * 4;
    const size_t total = off_bar + kGmSlots * 16 + 3 * kGmSlots * 8 + 128;   // + alignment slack
    // static shared memory: S = 1, about 30 KB with six segments per warp
    // (three staging areas per warp), 11 KB with two; S > 1, about 41 KB
    const size_t stat = S > 1 ? 42 : spw > 2 ? 31 : 12;
    if (total + stat * 1024 > smem_max) return false;
    a->fmt = fmt;
    a->S = S;
    a->I = I;
    a->rs = rs;
    a->ng = grouped ? ng : 0;
    a->gsh = gsh;
    a->nseg = nseg;
    a->spw = spw;
    a->nt = nt;
    a->bs = (int)bs;
    a->so = (int)so;
    a->ss = (int)ss;
    a->slot_bytes = (int)SB;
    a->off_red = (int)off_red;
    a->off_bar = (int)off_bar;
    a->timeout_ns = 2000000000LL;
    *smem = total;
    *grid = std::min(n_sm, a->stage_start[n]);
    return true;
}

size_t gm_counter_words() { return 2; }

template <int NTOK>
cudaError_t gm_launch_t(const GmArgs &a, int grid, size_t smem, cudaStream_t st) {
    constexpr int NT2 = NTOK == 1 ? 3 : 2;   // tiles per stage of the two-segment geometry
    const bool g = a.fmt == 4;
    if (a.nt == 1) {
        if (!g) return gm_go<false, 0, kMdSegMax, 1, NTOK>(a, grid, smem, st);
        return a.gsh == 0 ? gm_go<true, 0, kMdSegMax, 1, NTOK>(a, grid, smem, st)
                          : gm_go<true, 1, kMdSegMax, 1, NTOK>(a, grid, smem, st);
    }
    if (a.spw > 2 || a.nt != NT2) return cudaErrorInvalidValue;
    if (!g) return gm_go<false, 0, 2, NT2, NTOK>(a, grid, smem, st);
    return a.gsh == 0 ? gm_go<true, 0, 2, NT2, NTOK>(a, grid, smem, st) : gm_go<true, 1, 2, NT2, NTOK>(a, grid, smem, st);
}

cudaError_t launch_gemv_mma(const GmArgs &a, int grid, size_t smem, cudaStream_t st) {
    return a.S == 1 ? gm_launch_t<1>(a, grid, smem, st) : gm_launch_t<4>(a, grid, smem, st);
}

}  // namespace coli
