// gemm_tc.cu -- grouped dequantizing GEMM on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA), for int4 weights (fmt 2 and 4).
//
//   out[p][col0 + o] = sum_i W[o][i] * X[p][i]
//
// over tiles of (weight matrix, 128 weight rows, up to 64 activation rows).
// The weights are the M=128 side of the MMA, the activation rows the N side
// (most routed experts see only a handful of rows).  Codes are exact in bf16
// (code - 8 in [-8, 7]); each K-group of the scale (gs inputs, fmt=4) is
// accumulated into its own TMEM buffer and the f32 group scale is applied when
// the epilogue drains that buffer, so the products and the per-group sums are
// exact f32 tensor-core arithmetic.  Activations arrive as up to three bf16
// planes hi/mid/lo with x = hi + mid + lo to f32 precision; when the gather
// found every mid/lo zero (bf16-representable activations) only the first
// plane is loaded and multiplied.
//
// Warp roles (480 threads, persistent over a static tile schedule):
//   warps 0-7   dequant: codes (smem) -> bf16 A tile in TMEM (tcgen05.st),
//               two threads per weight row, each half a K-block; keeping A
//               out of shared memory leaves its bandwidth to the TMA streams
//   warps 8-11  epilogue: TMEM -> registers, group scale, row scale, store
//   warp  12    TMA producer of the codes: box [128 rows x 128 B] = 4 K-blocks
//   warp  13    MMA issuer (one thread), tcgen05.mma kind::f16, M=128
//   warp  14    TMA producer of the activation planes: one 4-D box per stage
//               of R rows (16, 32 or 64: the tile's rows rounded up) x the
//               planes x 64/R K-blocks, so small tiles take 4 K-blocks a copy
// A TMA copy or an MMA costs the issuing thread about 130 or 56 cycles (N <= 64),
// so each is made to carry as much of the tile as it can.
// With three planes they are stacked along N (N = 3 x R)
// so a K-step is one MMA whatever the plane count; the epilogue adds the three
// column blocks.  A tcgen05.mma with N <= 64 costs the same issue time as one
// with N = 64, so the issuing thread's loop is kept to the MMAs, the waits and
// the commits (descriptors advance by adding offsets, ring indices by wrap).
// The codes ring is released by the dequant warps as soon as they have read a
// stage, so its depth alone sets the bytes in flight from HBM; the plane ring
// (activations, mostly L2 hits) is released by the MMA commits.
// Every mbarrier wait is bounded in time; on expiry the kernel records
// DEV_ERR_TIMEOUT, drains its own copies and MMAs (bounded) and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "coli_internal.cuh"
#include "mbarrier.cuh"

namespace coli {

namespace {

constexpr int BM = 128, BK = 64, BN = 64;
constexpr int KB_PER_CS = 4;                          // K-blocks per codes stage: 128-byte row segments
constexpr int NC = 5;                                 // codes stages (16 KB each): the HBM stream
constexpr int NAMAX = 8;                              // dequantized A stages, in TMEM (32 columns each)
constexpr int NPL = 3;                                // activation planes
constexpr int CODES_BYTES = BM * BK / 2 * KB_PER_CS;  // 16384: 128 rows x 128 B, 128-byte swizzle
constexpr int PLANE_BYTES = BN * BK * 2;              // 8192: 64 rows x 128 B
constexpr int B_RING = 5 * NPL * PLANE_BYTES;         // 120 KB
constexpr int NB1 = B_RING / PLANE_BYTES;             // plane stages with one plane: 15
constexpr int NB3 = B_RING / (NPL * PLANE_BYTES);     // with three planes: 5
constexpr int NBMAX = NB1;
constexpr int NACCMAX = 4;
// TMEM (512 columns): accumulators first, then the A stages.  One plane:
// 4 accumulators of 64 columns + 8 A stages; three planes: 2 of 192 + 4.
constexpr int OFF_B = 0;
constexpr int OFF_CODES = OFF_B + B_RING;
constexpr int OFF_BAR = OFF_CODES + NC * CODES_BYTES;
constexpr int N_BAR = 2 * NC + 2 * NBMAX + 2 * NAMAX + 2 * NACCMAX + 1;
constexpr int SMEM_BYTES = OFF_BAR + N_BAR * 8 + 16 + 1024;   // + alignment slack
constexpr int kDqWarps = 8;                           // dequant warps: two per weight row (half a K-block each)
constexpr int kEpWarps = 4;                           // epilogue warps 8-11, one per TMEM lane quarter
constexpr int kCodesWarp = 12, kMmaWarp = 13, kPlanesWarp = 14;
constexpr int kTcThreads = 15 * 32;                   // <= 4 warps per SM sub-partition: 128 registers each
constexpr uint32_t TMEM_COLS = 512;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_addr(dst)), "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];"
        ::"r"(smem_addr(dst)), "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (SBO), version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for K-major SW128)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // descriptor version
    d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16: D f32, A bf16, B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// A from tensor memory (128 lanes = rows, 2 bf16 per column), B from shared memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t dtmem, uint32_t atmem, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(dtmem), "r"(atmem), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
// 16 consecutive TMEM columns of this thread's lane <- v; complete after tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
// 8 consecutive TMEM columns of this thread's lane; complete after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
}
// 16 consecutive TMEM columns of this thread's lane; complete after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct Tile {
    int mi, mb, col0, p0, p1, e;
};

__device__ __forceinline__ Tile tile_of(const TcArgs &a, int L, int n_tiles) {
    Tile t;
    int mb = L / n_tiles;
    const int ti = L - mb * n_tiles;
    t.mi = a.mi;
    t.col0 = 0;
    if (a.dual_mb > 0 && mb >= a.dual_mb) {
        mb -= a.dual_mb;
        t.mi = a.mi + 1;
        t.col0 = a.O;
    }
    t.mb = mb;
    if (a.tile_e) {
        t.e = a.tile_e[ti];
        t.p0 = a.tile_p0[ti];
        t.p1 = a.tile_p1[ti];
    } else {
        t.e = 0;
        t.p0 = ti * BN;
        t.p1 = min(a.P, t.p0 + BN);
    }
    return t;
}

__device__ __forceinline__ const MatDesc &mat_of(const TcArgs &a, const Tile &t) {
    return a.table ? a.table[t.e].m[t.mi] : a.single;
}

struct Bars {
    uint64_t *c_full, *c_empty, *b_full, *b_empty, *a_full, *a_empty, *acc_full, *acc_empty, *done;
};

// Row class of a tile: the activation rows one plane box carries (16, 32 or
// 64, at least the tile's rows) and how many K-blocks one plane stage holds
// (a stage is 64 rows x 64 inputs per plane).
__device__ __forceinline__ int rcls_of(const Tile &t) {
    const int n = t.p1 - t.p0;
    return n <= 16 ? 0 : (n <= 32 ? 1 : 2);
}

// The warp roles for NT activation planes.  With NT = 3 the planes are
// stacked along N: one MMA of N = 3 * R multiplies all three, and the
// epilogue adds the three column blocks.
template <int NT>
__device__ __forceinline__ void run_roles(const PlaneMapSet &tmx, const TcArgs &a, uint8_t *smem, const Bars &B,
                                          uint32_t tmem, volatile int &abort_flag, uint64_t deadline) {
    constexpr int NB = NT == 1 ? NB1 : NB3;
    constexpr int NACC = NT == 1 ? 4 : 2;             // TMEM accumulators of NT * 64 columns
    constexpr int NA = NT == 1 ? 8 : 4;               // A stages of 32 columns
    constexpr uint32_t A_COL0 = NACC * NT * BN;       // first A column
    static_assert(A_COL0 + NA * (BK / 2) <= TMEM_COLS, "TMEM budget");
    constexpr int B_STAGE = NT * PLANE_BYTES;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = a.tile_e ? *a.n_tiles : (a.P + BN - 1) / BN;
    const int total = n_tiles * a.n_mblk;

    auto fail = [&]() {
        if (!abort_flag) {
            abort_flag = 1;
            atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
        }
    };

    if (warp == kCodesWarp) {
        // ---------------- TMA producer: codes, 4 K-blocks (128 B of each of 128 rows) per stage
        if (lane == 0) {
            int it = 0, s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok && !abort_flag; L += gridDim.x) {
                const Tile t = tile_of(a, L, n_tiles);
                const MatDesc &M = mat_of(a, t);
                const int ncs = (a.nkb + KB_PER_CS - 1) / KB_PER_CS;
                for (int kc = 0; kc < ncs; kc++) {
                    if (it >= NC && !mbar_wait(&B.c_empty[s], ph ^ 1, deadline, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&B.c_full[s], CODES_BYTES);
                    tma_load_2d(smem + OFF_CODES + s * CODES_BYTES, (const CUtensorMap *)M.tmap,
                                kc * KB_PER_CS * (BK / 2), t.mb * BM, &B.c_full[s]);
                    it++;
                    if (++s == NC) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) fail();
            // every copy this thread issued has landed before the CTA may exit
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int k = max(0, it - NC); k < it; k++) mbar_wait(&B.c_full[k % NC], (k / NC) & 1, dl2, &no_abort);
        }
    } else if (warp == kPlanesWarp) {
        // ---------------- TMA producer: activation planes, one box of kps K-blocks x NT planes x R rows per stage
        if (lane == 0) {
            for (int c = 0; c < 3; c++) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmx.m[c + (NT == 1 ? 0 : 3)]) : "memory");
            int it = 0, s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok && !abort_flag; L += gridDim.x) {
                const Tile t = tile_of(a, L, n_tiles);
                const int rc = rcls_of(t), kps = 4 >> rc;
                const CUtensorMap *map = &tmx.m[rc + (NT == 1 ? 0 : 3)];
                for (int kb0 = 0; kb0 < a.nkb; kb0 += kps) {
                    if (it >= NB && !mbar_wait(&B.b_empty[s], ph ^ 1, deadline, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&B.b_full[s], B_STAGE);
                    tma_load_4d(smem + OFF_B + s * B_STAGE, map, 0, t.p0, 0, kb0, &B.b_full[s]);
                    it++;
                    if (++s == NB) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) fail();
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int k = max(0, it - NB); k < it; k++) mbar_wait(&B.b_full[k % NB], (k / NB) & 1, dl2, &no_abort);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer (one thread)
        if (lane == 0) {
            int ai = 0, as = 0, bs = 0, gb = 0, g = 0;
            uint32_t aph = 0, bph = 0, gph = 0;
            const uint64_t bd0 = sdesc_sw128(smem_addr(smem + OFF_B));
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok && !abort_flag; L += gridDim.x) {
                const Tile t = tile_of(a, L, n_tiles);
                const int rc = rcls_of(t), R = 16 << rc, kps = 4 >> rc;
                const uint32_t idesc = idesc_bf16(BM, NT * R);
                const uint32_t kstep = (uint32_t)(NT * R * BK * 2) >> 4;   // one K-block inside a plane stage
                int kk = 0, kg = 0;
                for (int kb = 0; kb < a.nkb; kb++) {
                    const bool first = kg == 0;
                    if (first && g >= NACC && !mbar_wait(&B.acc_empty[gb], gph ^ 1, deadline, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&B.a_full[as], aph, deadline, &abort_flag) ||
                        (kk == 0 && !mbar_wait(&B.b_full[bs], bph, deadline, &abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + A_COL0 + (uint32_t)(as * (BK / 2));
                    const uint64_t bd = bd0 + (uint64_t)(bs * (B_STAGE >> 4) + kk * kstep);
                    const uint32_t d = tmem + (uint32_t)(gb * NT * BN);
#pragma unroll
                    for (int j = 0; j < BK / 16; j++)
                        mma_bf16_ts(d, at + 8 * j, bd + 2 * j, idesc, (first && j == 0) ? 0u : 1u);
                    mma_commit(&B.a_empty[as]);
                    ai++;
                    if (++as == NA) {
                        as = 0;
                        aph ^= 1;
                    }
                    if (++kk == kps || kb == a.nkb - 1) {
                        mma_commit(&B.b_empty[bs]);
                        kk = 0;
                        if (++bs == NB) {
                            bs = 0;
                            bph ^= 1;
                        }
                    }
                    if (++kg == a.gkb || kb == a.nkb - 1) {
                        mma_commit(&B.acc_full[gb]);
                        kg = 0;
                        g++;
                        if (++gb == NACC) {
                            gb = 0;
                            gph ^= 1;
                        }
                    }
                }
            }
            if (!ok) fail();
            mma_commit(B.done);
            volatile int no_abort = 0;
            mbar_wait(B.done, 0, global_ns() + 200000000ull, &no_abort);
        }
    } else if (warp < kDqWarps) {
        // ---------------- dequant: thread (h, r) writes half h of weight row r of each K-block
        const int r = tid & (BM - 1), h = tid >> 7;
        int cs = 0, as = 0, it = 0;
        uint32_t cph = 0, aph = 0;
        bool ok = true;
        const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
        for (int L = blockIdx.x; L < total && ok && !__shfl_sync(0xffffffffu, (int)abort_flag, 0); L += gridDim.x) {
            for (int kb = 0; kb < a.nkb; kb++) {
                const int sub = kb & (KB_PER_CS - 1);
                if (sub == 0 && !warp_wait(&B.c_full[cs], cph, deadline, &abort_flag, lane)) {
                    ok = false;
                    break;
                }
                // row r of the stage is 128 B in 16-byte chunks swizzled by (r & 7)
                const uint4 c = *reinterpret_cast<const uint4 *>(smem + OFF_CODES + cs * CODES_BYTES + r * 128 +
                                                                 (((2 * sub + h) ^ (r & 7)) << 4));
                if (sub == KB_PER_CS - 1 || kb == a.nkb - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.c_empty[cs]);
                    if (++cs == NC) {
                        cs = 0;
                        cph ^= 1;
                    }
                }
                if (it >= NA && !warp_wait(&B.a_empty[as], aph ^ 1, deadline, &abort_flag, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
                uint32_t q[16];
#pragma unroll
                for (int cc = 0; cc < 4; cc++) {
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        uint32_t v = ((w[cc] >> (4 * k)) & 0x000F000Fu) | 0x43004300u;
                        __nv_bfloat162 hv = *reinterpret_cast<__nv_bfloat162 *>(&v);
                        hv = __hsub2(hv, off);
                        q[4 * cc + k] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                }
                // lane r of TMEM, columns [A_COL0 + 32 as + 16 h, +16): inputs 32h..32h+31 of the K-block
                tmem_st16(tmem + ((uint32_t)(warp & 3) << 21) + A_COL0 + (uint32_t)(as * (BK / 2) + h * 16), q);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.a_full[as]);
                it++;
                if (++as == NA) {
                    as = 0;
                    aph ^= 1;
                }
            }
        }
        if (!ok) fail();
    } else if (warp < kDqWarps + kEpWarps) {
        // ---------------- epilogue: warp 8+q reads TMEM lanes 32q..32q+31
        const int q = warp & 3;
        const int m = q * 32 + lane;
        int gb = 0;
        uint32_t gph = 0;
        bool ok = true;
        for (int L = blockIdx.x; L < total && ok && !__shfl_sync(0xffffffffu, (int)abort_flag, 0); L += gridDim.x) {
            const Tile t = tile_of(a, L, n_tiles);
            const MatDesc &M = mat_of(a, t);
            const int n_tok = t.p1 - t.p0;
            const int R = 16 << rcls_of(t);        // columns per plane block
            const int nch = (n_tok + 15) >> 4;     // 16-column chunks holding this tile's rows
            const int o = t.mb * BM + m;
            const bool row_ok = o < a.O;
            float acc[BN];
#pragma unroll
            for (int i = 0; i < BN; i++) acc[i] = 0.f;
            const int ngrp = (a.nkb + a.gkb - 1) / a.gkb;
            // group scales of this row, loaded SD groups ahead of their use
            constexpr int SD = 4;
            const bool grouped = a.fmt == 4 && row_ok;
            const float *srow = grouped ? M.s + (size_t)o * M.ng : nullptr;
            float scq[SD];
#pragma unroll
            for (int i = 0; i < SD; i++) scq[i] = (grouped && i < ngrp) ? __ldg(srow + i) : 1.0f;
            for (int grp0 = 0; grp0 < ngrp && ok; grp0 += SD) {
#pragma unroll
                for (int i = 0; i < SD; i++) {
                    const int grp = grp0 + i;
                    if (grp >= ngrp) break;
                    const float sc = scq[i];
                    scq[i] = (grouped && grp + SD < ngrp) ? __ldg(srow + grp + SD) : 1.0f;
                    if (!warp_wait(&B.acc_full[gb], gph, deadline, &abort_flag, lane)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(gb * NT * BN);
                    if (NT == 1) {
                        // two batches of 32 columns
#pragma unroll
                        for (int hb = 0; hb < 2; hb++) {
                            if (2 * hb >= nch) break;
                            uint32_t v[2][16];
#pragma unroll
                            for (int c = 0; c < 2; c++)
                                if (2 * hb + c < nch) tmem_ld16(base + (2 * hb + c) * 16, v[c]);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 2; c++)
                                if (2 * hb + c < nch) {
#pragma unroll
                                    for (int k = 0; k < 16; k++)
                                        acc[(2 * hb + c) * 16 + k] =
                                            fmaf(sc, __uint_as_float(v[c][k]), acc[(2 * hb + c) * 16 + k]);
                                }
                        }
                    } else {
                        // 8 columns of each plane at a time
#pragma unroll
                        for (int c8 = 0; c8 < BN / 8; c8++) {
                            if (c8 >= 2 * nch) break;
                            uint32_t v[NT][8];
#pragma unroll
                            for (int pl = 0; pl < NT; pl++) tmem_ld8(base + pl * R + c8 * 8, v[pl]);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 8; k++) {
                                float sum = __uint_as_float(v[NT - 1][k]);
#pragma unroll
                                for (int pl = NT - 2; pl >= 0; pl--) sum += __uint_as_float(v[pl][k]);
                                acc[c8 * 8 + k] = fmaf(sc, sum, acc[c8 * 8 + k]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.acc_empty[gb]);
                    if (++gb == NACC) {
                        gb = 0;
                        gph ^= 1;
                    }
                }
            }
            if (!ok) break;
            if (row_ok) {
                const float rs = (a.fmt == 4) ? 1.0f : __ldg(M.s + o);
                float *dst = a.out + (size_t)t.p0 * a.ldo + t.col0 + o;
#pragma unroll
                for (int n = 0; n < BN; n++)
                    if (n < n_tok) dst[(size_t)n * a.ldo] = acc[n] * rs;
            }
        }
        if (!ok) fail();
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ PlaneMapSet tmx, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + OFF_BAR);
    Bars B;
    B.c_full = bars;
    B.c_empty = B.c_full + NC;
    B.b_full = B.c_empty + NC;
    B.b_empty = B.b_full + NBMAX;
    B.a_full = B.b_empty + NBMAX;
    B.a_empty = B.a_full + NAMAX;
    B.acc_full = B.a_empty + NAMAX;
    B.acc_empty = B.acc_full + NACCMAX;
    B.done = B.acc_empty + NACCMAX;
    uint32_t *tmem_slot = (uint32_t *)(bars + N_BAR);
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint64_t deadline = global_ns() + (uint64_t)a.timeout_ns;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NC; i++) {
            mbar_init(&B.c_full[i], 1);
            mbar_init(&B.c_empty[i], kDqWarps);
        }
        for (int i = 0; i < NBMAX; i++) {
            mbar_init(&B.b_full[i], 1);
            mbar_init(&B.b_empty[i], 1);
        }
        for (int i = 0; i < NAMAX; i++) {
            mbar_init(&B.a_full[i], kDqWarps);
            mbar_init(&B.a_empty[i], 1);
        }
        for (int i = 0; i < NACCMAX; i++) {
            mbar_init(&B.acc_full[i], 1);
            mbar_init(&B.acc_empty[i], kEpWarps);
        }
        mbar_init(B.done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (*a.nterm_flag)
        run_roles<NPL>(tmx, a, smem, B, tmem, abort_flag, deadline);
    else
        run_roles<1>(tmx, a, smem, B, tmem, abort_flag, deadline);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// bf16 planes of the activations: plane t of row p holds the t-th bf16 term
// of X[src(p)], inputs permuted inside every group of 8 as 0,4,1,5,2,6,3,7 (the
// order the dequant writes the codes in), zero past I.
__global__ void gather_planes_kernel(const float *__restrict__ X, long long ldx, const int32_t *order, int kdiv,
                                     const int32_t *n_valid, int n_rows, int I, int I_pad, __nv_bfloat16 *planes,
                                     long long plane_elems, int *flag, const uint8_t *skip) {
    const int p = blockIdx.x;
    if (p >= n_rows) return;
    const int nv = n_valid ? *n_valid : n_rows;
    if (skip && p < nv && skip[p]) return;   // a row another path multiplies
    long long src = -1;
    if (p < nv) src = order ? (long long)(order[p] / kdiv) : (long long)p;
    bool nz = false;
    for (int k8 = threadIdx.x; k8 < I_pad / 8; k8 += blockDim.x) {
        __nv_bfloat16 hi[8], mid[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int e = 8 * k8 + ((i & 1) ? 4 + (i >> 1) : (i >> 1));
            const float v = (src >= 0 && e < I) ? X[src * ldx + e] : 0.f;
            hi[i] = __float2bfloat16_rn(v);
            const float r1 = v - __bfloat162float(hi[i]);
            mid[i] = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid[i]);
            lo[i] = __float2bfloat16_rn(r2);
            nz |= (r1 != 0.f);
        }
        const size_t base = (size_t)p * I_pad + 8 * k8;
        *reinterpret_cast<uint4 *>(planes + base) = *reinterpret_cast<uint4 *>(hi);
        *reinterpret_cast<uint4 *>(planes + plane_elems + base) = *reinterpret_cast<uint4 *>(mid);
        *reinterpret_cast<uint4 *>(planes + 2 * plane_elems + base) = *reinterpret_cast<uint4 *>(lo);
    }
    if (__syncthreads_or(nz) && threadIdx.x == 0) atomicOr(flag, 1);
}

// h = silu(g) * u from the fused gate|up output [rows][2F], written as bf16
// planes for the down projection (same permutation as gather_planes_kernel).
__global__ void silu_planes_kernel(const float *__restrict__ gu, int F, const int32_t *n_valid, int n_rows, int F_pad,
                                   __nv_bfloat16 *planes, long long plane_elems, int *flag, const uint8_t *skip) {
    const int p = blockIdx.x;
    if (p >= n_rows) return;
    // rows another path multiplies (skip[p]) are neither read nor written
    if (skip && p < *n_valid && skip[p]) return;
    const bool live = p < *n_valid;
    bool nz = false;
    for (int k8 = threadIdx.x; k8 < F_pad / 8; k8 += blockDim.x) {
        __nv_bfloat16 hi[8], mid[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int e = 8 * k8 + ((i & 1) ? 4 + (i >> 1) : (i >> 1));
            float v = 0.f;
            if (live && e < F) {
                const float g = gu[(size_t)p * 2 * F + e], u = gu[(size_t)p * 2 * F + F + e];
                v = g / (1.0f + expf(-g)) * u;
            }
            hi[i] = __float2bfloat16_rn(v);
            const float r1 = v - __bfloat162float(hi[i]);
            mid[i] = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid[i]);
            lo[i] = __float2bfloat16_rn(r2);
            nz |= (r1 != 0.f);
        }
        const size_t base = (size_t)p * F_pad + 8 * k8;
        *reinterpret_cast<uint4 *>(planes + base) = *reinterpret_cast<uint4 *>(hi);
        *reinterpret_cast<uint4 *>(planes + plane_elems + base) = *reinterpret_cast<uint4 *>(mid);
        *reinterpret_cast<uint4 *>(planes + 2 * plane_elems + base) = *reinterpret_cast<uint4 *>(lo);
    }
    if (__syncthreads_or(nz) && threadIdx.x == 0) atomicOr(flag, 1);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

}  // namespace

bool tc_supported_fmt(int fmt, int gs) { return fmt == 2 || (fmt == 4 && gs % BK == 0); }

int tc_block_rows() { return BN; }

cudaError_t encode_codes_map(const uint8_t *q, long long rs, long long O, void *out128) {
    CUtensorMap *out = (CUtensorMap *)out128;
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)rs, (cuuint64_t)O};
    cuuint64_t strides[1] = {(cuuint64_t)rs};
    cuuint32_t box[2] = {BK / 2 * KB_PER_CS, BM};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void *)q, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Six 4-D maps over the planes [3][rows_alloc][I_pad] bf16, dimensions
// (64 inputs, rows, plane, K-block): box (64, R, NTb, 64 / R) for R = 16, 32,
// 64 and NTb = 1 (maps 0-2) or 3 (maps 3-5).  One box fills a plane stage in
// the order [K-block][plane][row][64 inputs], 128-byte swizzled.
cudaError_t encode_plane_maps(const void *planes, long long I_pad, long long rows_alloc, PlaneMapSet *out) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[4] = {(cuuint64_t)BK, (cuuint64_t)rows_alloc, (cuuint64_t)NPL, (cuuint64_t)(I_pad / BK)};
    cuuint64_t strides[3] = {(cuuint64_t)(I_pad * 2), (cuuint64_t)(rows_alloc * I_pad * 2), (cuuint64_t)(BK * 2)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    for (int nt = 0; nt < 2; nt++)
        for (int rc = 0; rc < 3; rc++) {
            cuuint32_t box[4] = {BK, (cuuint32_t)(16 << rc), (cuuint32_t)(nt ? NPL : 1), (cuuint32_t)(4 >> rc)};
            CUresult r = fn(&out->m[rc + 3 * nt], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void *)planes, dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        }
    return cudaSuccess;
}

cudaError_t launch_gather_planes(const float *X, long long ldx, const int32_t *order, int kdiv, const int32_t *n_valid,
                                 int n_rows, int I, int I_pad, void *planes, long long plane_elems, int *flag,
                                 cudaStream_t st, const uint8_t *skip) {
    if (n_rows <= 0) return cudaSuccess;
    gather_planes_kernel<<<n_rows, 128, 0, st>>>(X, ldx, order, kdiv, n_valid, n_rows, I, I_pad,
                                                 (__nv_bfloat16 *)planes, plane_elems, flag, skip);
    return cudaGetLastError();
}

cudaError_t launch_silu_planes(const float *gu, int F, const int32_t *n_valid, int n_rows, int F_pad, void *planes,
                               long long plane_elems, int *flag, cudaStream_t st, const uint8_t *skip) {
    if (n_rows <= 0) return cudaSuccess;
    silu_planes_kernel<<<n_rows, 128, 0, st>>>(gu, F, n_valid, n_rows, F_pad, (__nv_bfloat16 *)planes, plane_elems,
                                               flag, skip);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const TcArgs &a, const PlaneMapSet &tmx, int max_tiles, int n_sm, cudaStream_t st) {
    const long long total = (long long)max_tiles * a.n_mblk;
    if (total <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = (int)(total < n_sm ? total : n_sm);
    gemm_tc_kernel<<<grid, kTcThreads, SMEM_BYTES, st>>>(tmx, a);
    return cudaGetLastError();
}

}  // namespace coli
