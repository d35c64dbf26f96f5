// decode_mma.cu -- the decode expert block at S = 1 (one token, top-K routed
// experts) for int4 expert tables (fmt 2, and fmt 4 with groups of a
// power-of-two multiple of 64 inputs), in one cooperative launch with one CTA
// per SM (colibri-strix commit log, "metal: batched moe_block": gate/up GEMV,
// SiLU * mul, down GEMV and the weighted sum over the routed experts as a
// single GPU pass).
//
// Arithmetic.  The dot products run on the tensor cores as register-operand
// mma.sync m16n8k16 (f16 inputs, f32 accumulate); this is a matrix-vector
// product, so the operands come straight from registers and only two of the
// eight B columns carry data.
//   A (weights): a 4-bit code n placed in the low mantissa bits of an f16
//     with a zero exponent field is the subnormal n * 2^-24, exact.  One AND
//     of a 32-bit word of eight codes with 0x000F000F gives the f16 pair
//     (n0, n4), with 0x00F000F0 the pair (16 n1, 16 n5); the word shifted
//     right by 8 gives (n2, n6) and (16 n3, 16 n7) the same way.  So one
//     word is four A registers for five integer operations.
//   B (activations): the warp scales its inputs by a power of two 2^k (the
//     largest magnitude lands in [2^14, 2^15)) and splits each into
//     hi = f16(v) and lo = f16((v - hi) * 2^11): column 0 holds hi, column 1
//     lo, so the pair carries 22 significant bits.  Inputs facing a 16 n code
//     are stored divided by 16.
//   The offset binary code value is n - 8: each chain of mma starts from
//   C = -8 * 2^-24 * (sum of the B values of its inputs), so the result is
//   2^-24 * sum (n - 8) v.  Per group (fmt 4) the chain result is multiplied
//   by the group's scale; per row (fmt 2) the row's scale is applied to the
//   finished dot product.
//
// Roles.  Warps 0..15 consume, warp 16 produces: its lane 0 streams stages
// into kMdSlots shared-memory slots with bulk copies (cp.async.bulk) and a
// descriptor per slot.  Warp 17 finishes every stage (below).  A stage holds whole rows in four blocks of rows; the
// blocks start 32 bytes apart modulo 128, and the 16 rows of an mma tile take
// row r of all four blocks for r = 0..3, so the 8-byte code loads of a
// half-warp fall in four different bank quarters.  Warp w owns the 64-input
// segments [w S, (w + 1) S) of every row and keeps their B fragments in
// registers.
//   phase 0: the token's routed experts, distinct and in ascending id order,
//            duplicate slots' weights summed (decode_route.cuh).
//   phase A: stages of 8 (gate, up) row pairs of one routed expert, dealt
//            round robin over the CTAs, the last routed expert's first.
//            Every consumer warp writes its segments' share of the 16 rows to
//            the slot's partial-sum table and moves on; warp 17 sums the table
//            in warp order and writes h[a][j] = silu(gate) * up to global
//            memory, each value as one 64-bit word under the call's tag.
//   phase B: each CTA serves one routed expert (md_share sizes the groups:
//            expert 0, whose h is finished last, gets more CTAs; the others
//            are interleaved so that every CTA's gate/up units plus down
//            stages come out even) and claims that expert's whole 48-row
//            stages of down rows one at a time, as its slots free up, from a
//            per-expert counter, so a group's CTAs finish together.  Each warp polls until the h
//            values of its segments carry the call's tag (no fence or grid
//            barrier: a 64-bit store is seen whole), builds their B fragments
//            once and streams the CTA's rows in stages of 48; warp 17 sums the
//            warps' shares of each row in warp order into part[a][o].
//            The sums go out as tagged 64-bit words too.
//   y:       CTA G - 1 - c sums the 64-row blocks c, c + G, ... of y over the routed
//            experts in order, with their routing weights, once every part
//            value of the block carries the call's tag: y[o] is written once.
// Results do not depend on timing or on the number of SMs.  Every wait is
// bounded (mbarrier.cuh); on expiry the kernel records DEV_ERR_TIMEOUT and
// returns.  The last CTA to leave moves the tag on for the next call.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>

#include "coli_internal.cuh"
#include "decode_route.cuh"
#include "mbarrier.cuh"
#include "mma_int4.cuh"

namespace coli {

namespace {

constexpr int kMdThreads = (kMdWarps + 2) * 32;   // consumers, then the producer warp and the epilogue warp
constexpr int kMdSlots = 3;      // shared-memory slots of the stage ring
// back-off (ns) of a waiting warp: consumer, epilogue, producer
constexpr uint32_t kMdNapC = 0, kMdNapE = 64, kMdNapP = 64;
constexpr int kMdTiles = 3;                   // 16-row mma tiles of a phase-B stage
constexpr int kMdBlockRows = 4 * kMdTiles;     // rows of each of a phase-B stage's four blocks
constexpr int kMdStageRows = 4 * kMdBlockRows; // down rows of a phase-B stage (48)
// partial sums of a stage: phase A [warp][48] (16 rows used), phase B
// [row][20] (16 warps, padded so that a lane's row is one conflict-free
// 128-bit load per 4 warps)
constexpr int kMdRedB = 20;
constexpr int kMdRedSlot = kMdStageRows * kMdRedB;
// state words of the kernel (zero before the first call): [1] CTAs out,
// [3] epoch, [4, 4 + 64) down stages claimed per routed expert, then the
// tagged h [K][F] and part [K][H] (8 bytes each)
constexpr int kMdClaim = 4;
constexpr int kMdCtrH = kMdClaim + 64;

enum : int { MD_A = 0, MD_B = 1, MD_END = 2 };
static_assert(kMaxDecodeSlots + 1 <= (int)(sizeof(MdArgs::m0) / sizeof(int)), "MdArgs::m0 covers every routed-expert count");

// Stages [s0, s1) of member j of a group of M CTAs that split nsE stages,
// where members j < Hh carry q + 1 gate/up units and the others q: units +
// stages come out T or T + 1 for every member, the + 1 going to members with
// fewer units first; when the stages are too few for that, an even split.
__device__ __forceinline__ void md_split(int j, int M, int Hh, int q, int nsE, int *s0, int *s1) {
    const int Lt = M * q + Hh + nsE;
    const int T = Lt / M, r = Lt % M;
    if (T < q + 1) {
        *s0 = nsE * j / M;
        *s1 = nsE * (j + 1) / M;
        return;
    }
    const int light = M - Hh;
    auto plus_before = [&](int jj) -> int {   // + 1s among members 0 .. jj - 1
        if (r <= light) return min(max(jj - Hh, 0), r);
        return max(jj - Hh, 0) + min(jj, r - light);
    };
    auto units_before = [&](int jj) -> int { return jj * q + min(jj, Hh); };
    *s0 = j * T - units_before(j) + plus_before(j);
    *s1 = (j + 1) * T - units_before(j + 1) + plus_before(j + 1);
}

// The down-phase share of CTA c: its routed expert eB and the stages [s0, s1)
// of that expert's nsE stages of 48 down rows.  Gate/up units are dealt round
// robin (CTA c gets q + 1 of them for c < rA, else q), the last routed
// expert's first, so expert 0's h is finished last: at the end of the final
// (partial) round, and it reaches its owners about one unit's time later.
// Expert 0 therefore gets the first M0 CTAs (those with q + 1 units, busy to
// the end anyway), M0 = md_m0(...) computed with the plan, so that its owners
// (starting at q + 2 units, even split) and the others (interleaved over CTAs
// M0 .. G - 1, md_split) finish together; with one routed expert every CTA
// owns it (md_split).
// (32-bit arithmetic: G <= 1024 CTAs, nact <= 64, fewer than 2^20 units.)
__device__ __forceinline__ void md_share(int c, int nact, int G, int totalA, int nsE, int M0, int *eB, int *s0,
                                         int *s1) {
    const int q = totalA / G, rA = totalA % G;
    if (nact == 1) {
        *eB = 0;
        md_split(c, G, rA, q, nsE, s0, s1);
        return;
    }
    const int no = nact - 1;
    if (c < M0) {
        *eB = 0;
        *s0 = nsE * c / M0;
        *s1 = nsE * (c + 1) / M0;
        return;
    }
    const int cc = c - M0, e = 1 + cc % no, j = cc / no;
    const int base = M0 + (e - 1);                           // the group's member j is CTA base + j no
    const int M = (G - base + no - 1) / no;
    const int Hh = rA > base ? min(M, (rA - base + no - 1) / no) : 0;
    *eB = e;
    md_split(j, M, Hh, q, nsE, s0, s1);
}

// The h values lane `lane` of a phase-B warp needs (inputs 64 q0 + 4 lane +
// 0..3 of the warp's segments, as md_load4): each is the f32 bits under the
// call's tag in a 64-bit word.  Polls until every value of the warp carries
// `tag`; false (for the whole warp) once the deadline passed or the CTA
// aborted.
__device__ __forceinline__ bool md_load_h(const unsigned long long *h, int n, int q0, int nq, int lane, unsigned tag,
                                          uint64_t deadline, volatile int *abort, float4 *out) {
    const int seg = lane >> 4;
    const long long i0 = (long long)(q0 + seg) * 64 + 4 * (lane & 15);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    while (true) {
        bool ok = true;
        if (seg < nq) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                if (i0 + j < n) {
                    unsigned long long w;
                    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(h + i0 + j) : "memory");
                    ok &= (unsigned)(w >> 32) == tag;
                    v[j] = __uint_as_float((unsigned)w);
                }
            }
        }
        if (__all_sync(0xffffffffu, ok)) break;
        if (__any_sync(0xffffffffu, *abort != 0 || global_ns() > deadline)) return false;
        __nanosleep(128);
    }
    *out = make_float4(v[0], v[1], v[2], v[3]);
    return true;
}

// GSH: log2(gs / 64), segments per scale group (fmt 4); 0 for fmt 2.
template <bool GROUPED, int GSH>
__global__ void __launch_bounds__(kMdThreads, 1) moe_decode_mma_kernel(const MdArgs a) {
    extern __shared__ uint8_t sraw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    float *red = reinterpret_cast<float *>(base + a.off_red);   // [slot][kMdRedSlot]: partial sums of a stage
    int4 *desc = reinterpret_cast<int4 *>(base + a.off_bar);    // [slot]
    uint64_t *full = reinterpret_cast<uint64_t *>(desc + kMdSlots);
    uint64_t *empty = full + kMdSlots;
    uint64_t *redfull = empty + kMdSlots;   // every consumer warp wrote its partial sums of the stage
    __shared__ DecodeRouting rt;
    __shared__ volatile int abort_flag;
    __shared__ float4 s_cf[kMdWarps][kMdSegMax + 1];   // phase-A chain starts of each warp's segments, their sum
    __shared__ __align__(16) uint8_t s_stg[kMdWarps][kMdStgBytes];   // B-fragment staging of each consumer warp, + a zero row
    __shared__ float s_part[kMdWarps * 32];                  // the final sum: one (expert, row) per thread
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // programmatic dependent launch: one CTA fills an SM, so the next kernel
    // may begin launching now and its CTAs take the SMs this grid frees; every
    // input of this one (x, the routing, the state words) may come from the
    // previous kernel, so nothing is read before it has completed
    pdl_trigger();
    pdl_wait();
    const int SB = a.slot_bytes;
    const uint64_t deadline = global_ns() + (uint64_t)a.timeout_ns;
    unsigned *exitc = a.ctr + 1;
    unsigned *claimB = a.ctr + kMdClaim;   // [routed expert]: down stages claimed so far
    // h values carry the call's tag in their high word: a 64-bit store is seen
    // whole or not at all, so a reader knows a value is this call's without a fence
    unsigned long long *htag = reinterpret_cast<unsigned long long *>(a.ctr + kMdCtrH);
    unsigned long long *ptag = htag + (size_t)a.K * a.F;
    const unsigned tag = *(volatile unsigned *)(a.ctr + 3) + 1u;

    // consumers load their x values now; the fragments are built after routing
    const int q0A = warp * a.spwA, nqA = min(a.spwA, a.nsegA - q0A);
    constexpr int NR = (kMdSegMax + 1) / 2;
    float4 ldA[NR];
    if (warp < kMdWarps) {
#pragma unroll
        for (int r = 0; r < NR; r++) ldA[r] = md_load4(a.x, a.H, q0A, nqA, r, lane, false);
    }

    // routing: by the producer warp alone for K <= 32 (the consumers build their
    // phase-A fragments meanwhile), else by the whole CTA
    auto md_init = [&]() {
        abort_flag = 0;
        for (int i = 0; i < kMdSlots; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kMdWarps);
            mbar_init(&redfull[i], kMdWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    };
    const bool wroute = a.K <= 32;
    if (!wroute) {
        if (tid == 0) md_init();
        decode_route(rt, a.ids, a.w, a.K, a.n_experts, a.table, kMdWarps);
    } else if (warp == kMdWarps) {
        decode_route_warp(rt, a.ids, a.w, a.K, a.n_experts, a.table);
        if (lane == 0) md_init();
        __syncwarp();
    }
    // phase-A B fragments of the consumer warps (the token's x: no routing needed)
    uint32_t bfA[kMdSegMax][8];
    float unA = 0.f;
    if (warp < kMdWarps) {
        uint32_t *zr = reinterpret_cast<uint32_t *>(&s_stg[warp][kMdStgZero]);
        if (lane < 4) zr[lane] = 0u;
        __syncwarp();
        const uint32_t stg = smem_addr(&s_stg[warp][0]), zrow = smem_addr(zr);
        const MdScale scA = md_scale<NR>(ldA);
        unA = scA.unscale * 0x1p24f;
        float4 cft = make_float4(0.f, 0.f, 0.f, 0.f);   // per-row formats: the chain start of the whole row
#pragma unroll
        for (int r = 0; r < NR; r++) {
            float4 c0, c1;
            md_frags(ldA[r], scA, nqA - 2 * r, lane, stg, zrow, bfA[2 * r], bfA[2 * r + 1], c0, c1);
            if (lane == 0) {
                s_cf[warp][2 * r] = c0;
                s_cf[warp][2 * r + 1] = c1;
            }
            cft.x += c0.x + c1.x;
            cft.y += c0.y + c1.y;
            cft.z += c0.z + c1.z;
            cft.w += c0.w + c1.w;
        }
        // lane 0 holds the hi / lo quads of tile row 0; every row's start is the same
        if (lane == 0) s_cf[warp][kMdSegMax] = cft;
        __syncwarp();
    }
    // the routing and the shared state are visible to every warp after barrier
    // 5; the producer passes it without waiting, once it has issued the first
    // stage (the other warps wait in the barrier, not spinning on the stage)
    auto release_others = [&]() { asm volatile("bar.arrive 5, %0;" ::"r"(kMdThreads) : "memory"); };
    if (warp != kMdWarps) named_sync(5, kMdThreads);
    if (rt.bad) {
        if (warp == kMdWarps) release_others();
        if (blockIdx.x == 0 && tid == 0) atomicCAS(a.err, 0, DEV_ERR_BAD_ID);
        return;
    }
    const int nact = rt.nact;
    if (nact == 0) {   // no routed expert: y = 0
        if (warp == kMdWarps) release_others();
        const int rpc = (a.H + gridDim.x - 1) / gridDim.x;
        for (int r = tid; r < rpc; r += kMdThreads)
            if ((int)blockIdx.x * rpc + r < a.H) a.y[blockIdx.x * rpc + r] = 0.f;
        return;
    }
    // phase B: this CTA's routed expert eB (md_share sizes the group of CTAs of
    // each expert); the group's CTAs claim its 48-row down stages one at a time
    const int G = gridDim.x;
    const int spe = (a.F + 7) / 8;   // phase-A stages per routed expert
    const int nsE = (a.H + kMdStageRows - 1) / kMdStageRows;   // 48-row stages of a down matrix
    int eB = 0, sB0 = 0, sB1 = 0;
    md_share(blockIdx.x, nact, G, nact * spe, nsE, a.m0[nact], &eB, &sB0, &sB1);

    if (warp == kMdWarps) {
        // ---------------- producer: lane 0 issues every stage of the CTA.  Phase-A
        // units are dealt round robin, the last routed expert's first, so that
        // the final round (a partial one) belongs to expert 0
        const unsigned totalA = (unsigned)(nact * spe);
        const int rsA = a.rs_gu, rsB = a.rs_d;
        unsigned idx = blockIdx.x;
        int i = 0, sBc = -1;   // sBc: the down stage claimed next (-1: none yet)
        bool more = true;
        // stage i into slot i % kMdSlots; false after the end marker or an abort
        auto issue = [&]() -> bool {
            const int s = i % kMdSlots;
            if (i >= kMdSlots && !md_wait1(&empty[s], ((i / kMdSlots) & 1) ^ 1, deadline, &abort_flag, kMdNapP)) {
                if (!abort_flag) {
                    abort_flag = 1;
                    atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                }
                return false;
            }
            uint8_t *dst = base + (size_t)s * SB;
            if (idx < totalA) {
                const int ai = nact - 1 - (int)(idx / spe), j0 = (int)(idx % spe) * 8;
                const int w = min(8, a.F - j0);
                desc[s] = make_int4(MD_A, ai, j0, w);
                uint32_t tx = 0;
                int cnt[4];
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    cnt[b] = max(0, min(4, w - 4 * (b & 1)));
                    tx += (uint32_t)cnt[b] * (uint32_t)(rsA + (GROUPED ? 4 * a.ng_gu : 0));
                }
                mbar_expect_tx(&full[s], tx);
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    if (cnt[b] == 0) continue;
                    const int pr0 = j0 + 4 * (b & 1), m = b >> 1;
                    bulk_load(dst + b * (a.bsA + 32), rt.q[ai][m] + (size_t)pr0 * rsA, (uint32_t)(cnt[b] * rsA),
                              &full[s]);
                    if (GROUPED)
                        bulk_load(dst + a.soA + b * a.ssA, rt.s[ai][m] + (size_t)pr0 * a.ng_gu,
                                  (uint32_t)(cnt[b] * a.ng_gu * 4), &full[s]);
                }
                idx += G;
            } else if ((sBc >= 0 ? sBc : (sBc = (int)atomicAdd(claimB + eB, 1u))) < nsE) {
                // the next unclaimed 48-row stage of expert eB's down rows: the
                // CTAs of an expert take its stages as their slots free up
                const int r0 = sBc * kMdStageRows, nr = min(kMdStageRows, a.H - r0);
                desc[s] = make_int4(MD_B, eB, r0, nr);
                uint32_t tx = 0;
                int cnt[4];
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    cnt[b] = max(0, min(kMdBlockRows, nr - b * kMdBlockRows));
                    tx += (uint32_t)cnt[b] * (uint32_t)(rsB + (GROUPED ? 4 * a.ng_d : 0));
                }
                mbar_expect_tx(&full[s], tx);
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    if (cnt[b] == 0) continue;
                    const size_t rr = (size_t)r0 + (size_t)b * kMdBlockRows;
                    bulk_load(dst + b * (a.bsB + 32), rt.q[eB][2] + rr * rsB, (uint32_t)(cnt[b] * rsB), &full[s]);
                    if (GROUPED)
                        bulk_load(dst + a.soB + b * a.ssB, rt.s[eB][2] + rr * a.ng_d, (uint32_t)(cnt[b] * a.ng_d * 4),
                                  &full[s]);
                }
                // claim the next one now: its round trip overlaps the wait for a free slot
                sBc = (int)atomicAdd(claimB + eB, 1u);
            } else {
                desc[s] = make_int4(MD_END, 0, 0, 0);
                mbar_arrive(&full[s]);   // end marker: no bytes
                i++;
                return false;
            }
            i++;
            return true;
        };
        if (lane == 0) more = issue();
        __syncwarp();
        release_others();
        if (lane == 0) {
            while (more) more = issue();
            // every copy issued has landed before the CTA may exit
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int q = max(0, i - kMdSlots); q < i; q++)
                mbar_wait(&full[q % kMdSlots], (q / kMdSlots) & 1, dl2, &no_abort);
        }
        return;
    }

    if (warp == kMdWarps + 1) {
        // ---------------- epilogue: sums the consumer warps' partials of each stage
        // in warp order, then frees the slot.  Phase A: h = silu(gate) * up, stored
        // under the call's tag; phase B: the expert's rows of part
        int i = 0;
        bool ok = true;
        while (true) {
            const int s = i % kMdSlots;
            const uint32_t par = (uint32_t)((i / kMdSlots) & 1);
            if (!md_wait(&full[s], par, deadline, &abort_flag, kMdNapE)) {
                ok = false;
                break;
            }
            const int4 d = desc[s];
            if (d.x == MD_END) break;
            if (!md_wait(&redfull[s], par, deadline, &abort_flag, kMdNapE)) {
                ok = false;
                break;
            }
            const float *rd = red + s * kMdRedSlot;
            if (d.x == MD_A) {
                // row m = lane % 16 summed over warps 8 (lane / 16) .. + 7, then the two halves
                const float *rp = rd + (lane >> 4) * 8 * kMdStageRows + (lane & 15);
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < 8; w++) v += rp[w * kMdStageRows];
                // the slot is free once its partial sums are read
                __syncwarp();
                if (lane == 0) md_release(&empty[s]);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                // tile row of gate pair p: block p / 4, row p % 4 -> 4 (p % 4) + p / 4; up: + 2
                const int p = lane & 7;
                const int mg = 4 * (p & 3) + (p >> 2);
                float gv = __shfl_sync(0xffffffffu, v, mg), uv = __shfl_sync(0xffffffffu, v, mg + 2);
                if (lane < d.w) {
                    if (!GROUPED) {
                        gv *= __ldg(rt.s[d.y][0] + d.z + lane);
                        uv *= __ldg(rt.s[d.y][1] + d.z + lane);
                    }
                    const float h = gv / (1.0f + expf(-gv)) * uv;
                    const unsigned long long hv = ((unsigned long long)tag << 32) | __float_as_uint(h);
                    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(htag + (size_t)d.y * a.F + d.z + lane),
                                 "l"(hv)
                                 : "memory");
                }
            } else {
                // stage row rr = lane (+ 32): the 16 warps' shares in warp order
                float v[2] = {0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int rr = lane + 32 * h;
                    if (rr < d.w) {
                        const float4 *rr4 = reinterpret_cast<const float4 *>(rd + rr * kMdRedB);
#pragma unroll
                        for (int w4 = 0; w4 < kMdWarps / 4; w4++) {
                            const float4 q = rr4[w4];
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
                    if (rr < d.w) {
                        if (!GROUPED) v[h] *= __ldg(rt.s[d.y][2] + d.z + rr);
                        const unsigned long long pv = ((unsigned long long)tag << 32) | __float_as_uint(v[h]);
                        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(ptag + (size_t)d.y * a.H + d.z + rr),
                                     "l"(pv)
                                     : "memory");
                    }
                }
            }
            i++;
        }
        if (!ok && lane == 0 && !abort_flag) {
            abort_flag = 1;
            atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
        }
        named_sync(2, (kMdWarps + 1) * 32);
    } else {
        // ---------------- consumers
        const uint32_t ring_s = smem_addr(base);
        const int g = lane >> 2, t = lane & 3;
        const int blk = g & 3, rib = g >> 2;   // block and row in block of tile row g (row g + 8: rib + 2)
        const uint32_t stg = smem_addr(&s_stg[warp][0]), zrow = smem_addr(&s_stg[warp][kMdStgZero]);
        int i = 0;                              // stage counter
        bool live = true;
        {
            // phase A
            uint32_t(&bf)[kMdSegMax][8] = bfA;
            const uint32_t rs2 = 2u * (uint32_t)a.rs_gu;
            const uint32_t cofs = (uint32_t)(blk * (a.bsA + 32) + rib * a.rs_gu + 32 * q0A + 8 * t);
            const uint32_t sofs = (uint32_t)(a.soA + blk * a.ssA + rib * a.ng_gu * 4 + (q0A >> GSH) * 4);
            const uint32_t sr2 = 8u * (uint32_t)a.ng_gu;
            const uint32_t cfs = smem_addr(&s_cf[warp][0]);
            const bool fullA = nqA == kMdSegMax;
            while (true) {
                const int s = i % kMdSlots;
                if (!md_wait(&full[s], (uint32_t)((i / kMdSlots) & 1), deadline, &abort_flag, kMdNapC)) {
                    if (lane == 0 && !abort_flag) {
                        abort_flag = 1;
                        atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                    }
                    live = false;
                    break;
                }
                const int4 d = desc[s];
                if (d.x != MD_A) break;   // stage i belongs to phase B (or is the end marker)
                const uint32_t sb = ring_s + (uint32_t)(s * SB);
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                if (fullA)
                    md_tileA<GROUPED, GSH, true>(y, sb + cofs, rs2, cfs, sb + sofs, sr2, nqA, bf);
                else if (nqA > 0)
                    md_tileA<GROUPED, GSH, false>(y, sb + cofs, rs2, cfs, sb + sofs, sr2, nqA, bf);
                float *rw = red + s * kMdRedSlot + warp * kMdStageRows;
                if (t == 0) {
                    const bool on = nqA > 0;
                    rw[g] = on ? fmaf(y[1], 0x1p-11f, y[0]) * unA : 0.f;
                    rw[g + 8] = on ? fmaf(y[3], 0x1p-11f, y[2]) * unA : 0.f;
                }
                // the epilogue warp turns the stage into h and frees the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(&redfull[s]);
                i++;
            }
        }
        // phase B: the warp's h values of expert eB (this call's tag on every one),
        // its B fragments built once, then the stages of down[eB] this CTA claimed
        if (live) {
            const int q0B = warp * a.spwB, nqB = min(a.spwB, a.nsegB - q0B);
            const int rs = a.rs_d;
            const uint32_t cofs = (uint32_t)(blk * (a.bsB + 32) + rib * rs + 32 * q0B + 8 * t);
            const uint32_t sofs = (uint32_t)(a.soB + blk * a.ssB + rib * a.ng_d * 4 + (q0B >> GSH) * 4);
            uint32_t bf[2][8];
            float4 cq[2];
            float unB = 0.f;
            {
                float4 ld = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!md_load_h(htag + (size_t)eB * a.F, a.F, q0B, nqB, lane, tag, deadline, &abort_flag, &ld)) {
                    if (lane == 0 && !abort_flag) {
                        abort_flag = 1;
                        atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                    }
                    live = false;
                }
                float4 lda[1] = {ld};
                const MdScale scB = md_scale<1>(lda);
                unB = scB.unscale * 0x1p24f;
                md_frags(ld, scB, nqB, lane, stg, zrow, bf[0], bf[1], cq[0], cq[1]);
            }
            const bool fullB = nqB == 2;
            // offsets of the tiles' code words and scales (rows 4 T + rib of each block)
            uint32_t tco[kMdTiles], tso[kMdTiles];
#pragma unroll
            for (int T = 0; T < kMdTiles; T++) {
                tco[T] = cofs + (uint32_t)(4 * T * rs);
                tso[T] = sofs + (uint32_t)(4 * T * a.ng_d * 4);
            }
            const uint32_t rs2 = 2u * (uint32_t)rs, sr2 = 8u * (uint32_t)a.ng_d;
            while (live) {
                const int s = i % kMdSlots;
                if (!md_wait(&full[s], (uint32_t)((i / kMdSlots) & 1), deadline, &abort_flag, kMdNapC)) {
                    if (lane == 0 && !abort_flag) {
                        abort_flag = 1;
                        atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                    }
                    break;
                }
                const int4 d = desc[s];
                if (d.x != MD_B) {   // end marker
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    break;
                }
                const uint32_t sb = ring_s + (uint32_t)(s * SB);
                // tile row m = g, g + 8 of tile T is stage row 12 (m % 4) + 4 T + m / 4
                float *rw = red + s * kMdRedSlot + (blk * kMdBlockRows + rib) * kMdRedB + warp;
#pragma unroll
                for (int T = 0; T < kMdTiles; T++) {
                    float y[4] = {0.f, 0.f, 0.f, 0.f};
                    if (nqB > 0) {
                        const uint32_t tofs = sb + tco[T], tsc = sb + tso[T];
#pragma unroll
                        for (int sg = 0; sg < 2; sg++) {
                            if (fullB || sg < nqB) {
                                const uint2 cg = lds64(tofs + 32 * sg), ch = lds64(tofs + rs2 + 32 * sg);
                                if (GROUPED) {
                                    float dd[4];
                                    md_segment_c(dd, cg, ch, bf[sg], cq[sg]);
                                    const uint32_t sa = tsc + 4 * (sg >> GSH);
                                    const float sgv = md_ldsf(sa), shv = md_ldsf(sa + sr2);
                                    y[0] = fmaf(sgv, dd[0], y[0]);
                                    y[1] = fmaf(sgv, dd[1], y[1]);
                                    y[2] = fmaf(shv, dd[2], y[2]);
                                    y[3] = fmaf(shv, dd[3], y[3]);
                                } else {
                                    y[0] += cq[sg].x;
                                    y[1] += cq[sg].y;
                                    y[2] += cq[sg].z;
                                    y[3] += cq[sg].w;
                                    md_segment(y, cg, ch, bf[sg]);
                                }
                            }
                        }
                    }
                    if (t == 0) {
                        const bool on = nqB > 0;
                        rw[4 * T * kMdRedB] = on ? fmaf(y[1], 0x1p-11f, y[0]) * unB : 0.f;
                        rw[(4 * T + 2) * kMdRedB] = on ? fmaf(y[3], 0x1p-11f, y[2]) * unB : 0.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&redfull[s]);
                i++;
            }
        }
        named_sync(2, (kMdWarps + 1) * 32);
        // y: CTA G - 1 - c sums the 64-row blocks c, c + G, ... (the CTAs at the end
        // of the grid have one gate/up unit fewer): each thread polls one
        // (expert, row) of part until it carries the call's tag, then the rows are
        // summed over the routed experts in order, with their routing weights
        const int nblk = (a.H + 63) / 64;
        // (every consumer thread runs the same passes: the named barriers inside
        // stay matched; an abort only cuts the polling short)
        for (int blkI = G - 1 - (int)blockIdx.x; blkI < nblk; blkI += G) {
            const int rows = min(64, a.H - blkI * 64);
            const int per = kMdWarps * 32 / 64;   // experts per pass
            float v = 0.f;
            for (int e0 = 0; e0 < nact; e0 += per) {
                const int e = e0 + (tid >> 6), row = blkI * 64 + (tid & 63);
                bool okp = true;
                if (e < nact && (tid & 63) < rows) {
                    const unsigned long long *pp = ptag + (size_t)e * a.H + row;
                    while (true) {
                        unsigned long long w;
                        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(pp) : "memory");
                        if ((unsigned)(w >> 32) == tag) {
                            s_part[tid] = __uint_as_float((unsigned)w);
                            break;
                        }
                        if (abort_flag || global_ns() > deadline) {
                            okp = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
                if (!okp && !abort_flag) {
                    abort_flag = 1;
                    atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                }
                named_sync(3, kMdWarps * 32);
                if (tid < rows)
                    for (int k = 0; k < per && e0 + k < nact; k++) v = fmaf(rt.ew[e0 + k], s_part[k * 64 + tid], v);
                named_sync(3, kMdWarps * 32);
            }
            if (tid < rows && !abort_flag) a.y[blkI * 64 + tid] = v;
        }
        // the last CTA out moves the tag on for the next call
        if (tid == 0) {
            __threadfence();
            if (atomicAdd(exitc, 1u) == gridDim.x - 1) {
                *(a.ctr + 3) += 1u;
                for (int k = 0; k < a.K; k++) claimB[k] = 0u;
                *exitc = 0u;
                __threadfence();
            }
        }
    }
}

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

int log2_exact(int v) {
    int k = 0;
    while ((1 << k) < v) k++;
    return (1 << k) == v ? k : -1;
}

}  // namespace

// Geometry of the tensor-core decode block for an int4 expert table.  fmt=4
// needs gs_gu and gs_d to be 64 times a power of two and a multiple of 4
// scales per row (16-byte scale copies); H and F up to 16 * 6 * 64 = 6144.
// Returns false when the table does not fit this kernel.
bool md_plan(int fmt, int H, int F, int K, int rs_gu, int rs_d, int ng_gu, int ng_d, int gs_gu, int gs_d, int n_sm,
             size_t smem_max, MdArgs *a, size_t *smem) {
    if (fmt != 2 && fmt != 4) return false;
    const bool grouped = fmt == 4;
    int gsh_gu = 0, gsh_d = 0;
    if (grouped) {
        if (gs_gu % 64 != 0 || gs_d % 64 != 0) return false;
        gsh_gu = log2_exact(gs_gu / 64);
        gsh_d = log2_exact(gs_d / 64);
        // one shift for both roles, 64 or 128 inputs per group
        if (gsh_gu < 0 || gsh_gu > 1 || gsh_d != gsh_gu || ng_gu % 4 != 0 || ng_d % 4 != 0) return false;
    }
    if (H < 1 || F < 1 || n_sm < 1 || K < 1 || K > kMaxDecodeSlots) return false;
    const int nsegA = (H + 63) / 64, nsegB = (F + 63) / 64;
    // segments per warp: a multiple of the segments per scale group, so that
    // every warp starts at a group boundary
    const int gm = 1 << gsh_gu;
    const int spwA = ((nsegA + kMdWarps - 1) / kMdWarps + gm - 1) / gm * gm;
    const int spwB = ((nsegB + kMdWarps - 1) / kMdWarps + gm - 1) / gm * gm;
    if (spwA > kMdSegMax || spwB > kMdSegMax) return false;
    // phase B: every routed expert has CTAs of its own (at most K experts)
    if (n_sm < K || spwB > 2) return false;
    // slot layouts: four code blocks 32 bytes apart modulo 128 (each followed
    // by room for the 32-byte read past a row's last segment), then four
    // scale blocks 16 bytes apart modulo 128
    const size_t bsA = round_up((size_t)4 * rs_gu + 32, 128), soA = 4 * bsA + 128;
    const size_t ssA = grouped ? (size_t)16 * ng_gu + 16 : 0;
    const size_t bsB = round_up((size_t)kMdBlockRows * rs_d + 32, 128), soB = 4 * bsB + 128;
    const size_t ssB = grouped ? (size_t)kMdBlockRows * ng_d * 4 + 16 : 0;
    const size_t SB = round_up(std::max(soA + 4 * ssA, soB + 4 * ssB), 128);
    const size_t off_red = kMdSlots * SB;
    const size_t red_bytes = (size_t)kMdSlots * kMdRedSlot * 4;
    const size_t off_bar = off_red + red_bytes;
    const size_t total = off_bar + kMdSlots * 16 + 3 * kMdSlots * 8 + 128;   // + alignment slack
    // static shared memory of the kernel: about 17 KB
    if (total + 20 * 1024 > smem_max || SB > (1u << 30)) return false;
    memset(a, 0, sizeof *a);
    // CTAs of the expert finished last (md_share), for each possible number of
    // routed experts: the balance of expert 0's owners, which start at q + 2
    // units, against the others' units and stages
    {
        const int spe = (F + 7) / 8, nsE = (H + kMdStageRows - 1) / kMdStageRows, G = n_sm;
        for (int nact = 2; nact <= K; nact++) {
            const int totalA = nact * spe, q = totalA / G, rA = totalA % G, no = nact - 1;
            const long long start0 = q + (rA > 0 ? 1 : 0) + 1;
            int M0 = 1;
            long long best = -1;
            for (int m = 1; m <= G - no; m++) {
                const long long Ao = (long long)(G - m) * q + std::max(rA - m, 0);
                const long long lhs = start0 * m * (G - m) + (long long)nsE * (G - m);
                const long long rhs = Ao * m + (long long)no * nsE * m;
                const long long d = lhs > rhs ? lhs - rhs : rhs - lhs;
                if (best < 0 || d < best) {
                    best = d;
                    M0 = m;
                }
            }
            a->m0[nact] = M0;
        }
    }
    a->K = K;
    a->H = H;
    a->F = F;
    a->fmt = fmt;
    a->rs_gu = rs_gu;
    a->rs_d = rs_d;
    a->ng_gu = grouped ? ng_gu : 0;
    a->ng_d = grouped ? ng_d : 0;
    a->gsh_gu = gsh_gu;
    a->gsh_d = gsh_d;
    a->nsegA = nsegA;
    a->nsegB = nsegB;
    a->spwA = spwA;
    a->spwB = spwB;
    a->bsA = (int)bsA;
    a->ssA = (int)ssA;
    a->soA = (int)soA;
    a->bsB = (int)bsB;
    a->ssB = (int)ssB;
    a->soB = (int)soB;
    a->slot_bytes = (int)SB;
    a->off_red = (int)off_red;
    a->off_bar = (int)off_bar;
    *smem = total;
    return true;
}


// State words of the kernel (zero before its first call): counters, epoch and
// the tagged h [K][F].
size_t md_counter_words(const MdArgs &a) { return kMdCtrH + 2 * (size_t)a.K * ((size_t)a.F + a.H); }

// The kernel instance of a plan: fmt and group shift.
template <class Fn>
cudaError_t md_dispatch(const MdArgs &a, Fn &&fn) {
    if (a.fmt == 2) return fn(moe_decode_mma_kernel<false, 0>);
    return a.gsh_gu == 0 ? fn(moe_decode_mma_kernel<true, 0>) : fn(moe_decode_mma_kernel<true, 1>);
}

cudaError_t md_occupancy(const MdArgs &a, size_t smem, int *per_sm) {
    return md_dispatch(a, [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, kMdThreads, smem);
    });
}

cudaError_t launch_decode_mma(const MdArgs &a, int grid, size_t smem, cudaStream_t st) {
    return md_dispatch(a, [&](auto kern) {
        // the shared-memory limit is set once per kernel instance and size
        static std::mutex mu;
        static std::map<const void *, size_t> done;
        {
            std::lock_guard<std::mutex> lk(mu);
            size_t &have = done[(const void *)kern];
            if (have < smem) {
                cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                if (e != cudaSuccess) return e;
                have = smem;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kMdThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        // co-resident CTAs (they wait on one another's h and part values), and
        // programmatic serialization with the previous kernel where the driver
        // takes the two together; otherwise the cooperative launch alone
        static std::atomic<bool> no_pdl{false};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        if (!no_pdl.load(std::memory_order_relaxed)) {
            cfg.numAttrs = 2;
            if (cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess) return cudaSuccess;
            (void)cudaGetLastError();   // a refused launch configuration: nothing was launched
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
            // the pair was the problem only if the cooperative launch alone goes through
            if (e == cudaSuccess) no_pdl.store(true, std::memory_order_relaxed);
            return e;
        }
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a);
    });
}

}  // namespace coli
