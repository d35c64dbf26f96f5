// mma_int4.cuh -- the int4 dot-product pieces of the tensor-core matvec
// kernels (decode_mma.cu: the decode expert block; gemv_mma.cu: the streamed
// S = 1 matvec).
//
// A 4-bit code n in the low mantissa bits of an f16 with a zero exponent field
// is the subnormal n * 2^-24, exact, and mma.sync m16n8k16 (f16 in, f32
// accumulate) multiplies subnormals exactly.  One AND of a 32-bit word of
// eight codes with 0x000F000F gives the f16 pair (n0, n4), with 0x00F000F0
// the pair (16 n1, 16 n5); the word shifted right by 8 gives (n2, n6) and
// (16 n3, 16 n7): four A registers for five integer operations.  The
// activations are the B operand: a warp scales its inputs by 2^k and splits
// each into hi = f16(v) and lo = f16((v - hi) * 2^11) (columns 0 and 1; the
// inputs that face a 16 n code divided by 16).  Every chain starts from
// C = -8 * 2^-24 * (sum of its B values), which removes the code offset.
//
// Layout of a tile in shared memory: 16 rows of whole codes, tile row m in
// block m % 4 at row m / 4 (+ 4 T for tile T of a stage); the blocks start
// 32 bytes apart modulo 128, so the 8-byte code loads of a half-warp fall in
// four different bank quarters.  A warp owns consecutive 64-input segments.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "coli_internal.cuh"
#include "mbarrier.cuh"

namespace coli {

constexpr int kMdWarps = 16;     // consumer warps of the tensor-core matvec kernels
constexpr int kMdSegMax = 6;     // 64-input segments per warp and row (rows of up to 6144 inputs)
// B-fragment staging area of a warp (md_frags): four blocks of eight 16-byte
// rows, 144 bytes apart, so that the 2-byte stores of one instruction, which
// hit row r of all four blocks, fall in four different bank quarters; then
// one all-zero row
constexpr int kMdStgBlock = 144;
constexpr int kMdStgZero = 4 * kMdStgBlock;
constexpr int kMdStgBytes = kMdStgZero + 16;

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ float md_ldsf(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// d += A B on the tensor cores, m16n8k16, f16 operands, f32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B + c (the start of a chain: c and d are different registers).
__device__ __forceinline__ void mma16816c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, float4 c) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// One 64-input segment of a 16-row tile: cg / ch are the thread's two code
// words of its rows g and g + 8 (inputs 16 t + 0..7 and 16 t + 8..15 of the
// segment), bf the segment's eight B registers.  d = c + the segment's four
// products (md_segment_c) or d += them (md_segment).
__device__ __forceinline__ void md_segment_c(float (&d)[4], uint2 cg, uint2 ch, const uint32_t (&bf)[8], float4 c) {
    // one chain of four: the other warps' chains fill the tensor pipe meanwhile
    const uint32_t L = 0x000F000Fu, Hm = 0x00F000F0u;
    mma16816c(d, cg.x & L, ch.x & L, cg.x & Hm, ch.x & Hm, bf[0], bf[1], c);
    const uint32_t ug = cg.x >> 8, uh = ch.x >> 8;
    mma16816(d, ug & L, uh & L, ug & Hm, uh & Hm, bf[2], bf[3]);
    mma16816(d, cg.y & L, ch.y & L, cg.y & Hm, ch.y & Hm, bf[4], bf[5]);
    const uint32_t vg = cg.y >> 8, vh = ch.y >> 8;
    mma16816(d, vg & L, vh & L, vg & Hm, vh & Hm, bf[6], bf[7]);
}
__device__ __forceinline__ void md_segment(float (&d)[4], uint2 cg, uint2 ch, const uint32_t (&bf)[8]) {
    const uint32_t L = 0x000F000Fu, Hm = 0x00F000F0u;
    mma16816(d, cg.x & L, ch.x & L, cg.x & Hm, ch.x & Hm, bf[0], bf[1]);
    const uint32_t ug = cg.x >> 8, uh = ch.x >> 8;
    mma16816(d, ug & L, uh & L, ug & Hm, uh & Hm, bf[2], bf[3]);
    mma16816(d, cg.y & L, ch.y & L, cg.y & Hm, ch.y & Hm, bf[4], bf[5]);
    const uint32_t vg = cg.y >> 8, vh = ch.y >> 8;
    mma16816(d, vg & L, vh & L, vg & Hm, vh & Hm, bf[6], bf[7]);
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// The value lane `lane` loads for round r: inputs 64 q0 + 128 r + 4 lane + 0..3
// of v (length n); zero past n or past the warp's nq segments.
__device__ __forceinline__ float4 md_load4(const float *v, int n, int q0, int nq, int r, int lane, bool cg) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    const int seg = 2 * r + (lane >> 4);
    if (seg >= nq) return f;
    const long long i0 = (long long)(q0 + seg) * 64 + 4 * ((lane & 15));
    if (i0 + 4 <= n && ((reinterpret_cast<uintptr_t>(v + i0) & 15) == 0)) {
        f = cg ? __ldcg(reinterpret_cast<const float4 *>(v + i0)) : __ldg(reinterpret_cast<const float4 *>(v + i0));
    } else {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (i0 + j < n) t[j] = cg ? __ldcg(v + i0 + j) : __ldg(v + i0 + j);
        f = make_float4(t[0], t[1], t[2], t[3]);
    }
    return f;
}

// The warp's scale for its values (all rounds): 2^k with the largest
// magnitude times 2^k in [2^14, 2^15), k clamped so that 2^k and 2^-k are
// normal floats; unscale = 2^-k, or NaN when an input is not finite.
struct MdScale {
    float s2k, unscale;
};
template <int NR>
__device__ __forceinline__ MdScale md_scale(const float4 (&ld)[NR]) {
    uint32_t mb = 0;
#pragma unroll
    for (int r = 0; r < NR; r++) {
        mb = max(mb, __float_as_uint(ld[r].x) & 0x7fffffffu);
        mb = max(mb, __float_as_uint(ld[r].y) & 0x7fffffffu);
        mb = max(mb, __float_as_uint(ld[r].z) & 0x7fffffffu);
        mb = max(mb, __float_as_uint(ld[r].w) & 0x7fffffffu);
    }
    mb = __reduce_max_sync(0xffffffffu, mb);
    const int k = min(141 - (int)(mb >> 23), 126);
    MdScale sc;
    sc.s2k = __uint_as_float((uint32_t)(k + 127) << 23);
    sc.unscale = mb >= 0x7f800000u ? __uint_as_float(0x7fc00000u) : __uint_as_float((uint32_t)(127 - k) << 23);
    return sc;
}

// B fragments and chain starts of one round (two segments) of the warp's
// inputs, from the four values each lane loaded for it (md_load4: lane L holds
// inputs 4 L + 0..3 of the round).  nq = the warp's segments left from this
// round on.
//   Each lane converts its values to the hi / lo f16 halves and stores them
//   into the warp's staging area `stg` (kMdStgZero bytes) as the rows of the
//   transposed B operands: for every B operand (segment, k-step, P or Q) and
//   every half of its 16 k-slots, row 0 holds the hi column and row 1 the lo
//   column, 8 slots of 2 bytes each.  ldmatrix then hands every lane its
//   fragment; the lanes of the six all-zero columns read `zrow`.
//   Input 16 t + 8 i + j of a segment feeds k-step i, operand P (j & 2 == 0)
//   or Q, k-slot 2 t + j / 4 + 8 (j & 1): the slots of 16 n codes, j odd,
//   hold the input divided by 16.
//   b0 / b1: the eight B registers of the round's segments (k-step i:
//   P b0b1, P b2b3, Q b0b1, Q b2b3 at 4 i + 0..3), zero for segments >= nq.
//   c0 / c1: -8 * 2^-24 * sum of the segment's B values, as the accumulator
//   quad (hi, lo, hi, lo) of the tile rows: four mma of the fragments with the
//   constant A = -8 * 2^-24 (-128 * 2^-24 on the 16 n slots), exact f16
//   subnormals.
// The parts of md_frags (below): the lane's stores of one round into a
// staging area, the ldmatrix loads of a round's fragments, and the chain
// starts of a round.
__device__ __forceinline__ void md_frag_store(float4 ld, MdScale sc, int lane, uint32_t stg) {
    // store: lane L = 16 seg + 4 t + 2 i + h holds j = 4 h + 0..3
    const int seg = lane >> 4, t = (lane >> 2) & 3, i = (lane >> 1) & 1, h = lane & 1;
    const uint32_t wb = stg + (uint32_t)((seg * 2 + i) * kMdStgBlock + (2 * t + h) * 2);
    const float v[4] = {ld.x, ld.y, ld.z, ld.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        // q = j % 4: operand P (q < 2) or Q, slot half q % 2 (the 16 n slots for odd q)
        const float sv = v[q] * sc.s2k * ((q & 1) ? 0.0625f : 1.f);
        // hi: sv rounded to 11 significant bits, to nearest even, in integer
        // arithmetic (the f16 value of sv wherever that is a normal f16);
        // lo: the remainder times 2^11.  One conversion packs both halves.
        const uint32_t b = __float_as_uint(sv);
        const float h32 = __uint_as_float((b + 0xFFFu + ((b >> 13) & 1u)) & 0xFFFFE000u);
        const float l32 = (sv - h32) * 2048.f;
        uint32_t pk;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(h32), "f"(l32));   // hi in the upper half
        const uint32_t ad = wb + (uint32_t)((((q >> 1) * 2 + (q & 1)) * 2) * 16);
        asm volatile("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %0;\n st.shared.u16 [%1], h;\n st.shared.u16 [%2], l;\n}"
                     ::"r"(pk), "r"(ad), "r"(ad + 16));
    }
}
__device__ __forceinline__ void md_frag_load(int nq, int lane, uint32_t stg, uint32_t zrow, uint32_t (&b0)[8],
                                             uint32_t (&b1)[8]) {
    // matrix q of ldmatrix.x4 = (operand q / 2, slot half q % 2); lane L
    // gives row L % 8 of matrix L / 8: column 0 (hi) or 1 (lo), else zeros
    const int mq = lane >> 3, mr = lane & 7;
#pragma unroll
    for (int sg = 0; sg < 2; sg++) {
        uint32_t(&bf)[8] = sg ? b1 : b0;
        const bool on = sg < nq;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const uint32_t ra = mr < 2 ? stg + (uint32_t)((sg * 2 + i) * kMdStgBlock +
                                                          ((((mq >> 1) * 2 + (mq & 1)) * 2 + mr) * 16))
                                       : zrow;
            uint32_t r0, r1, r2, r3;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                         : "r"(ra));
            bf[4 * i + 0] = on ? r0 : 0u;
            bf[4 * i + 1] = on ? r1 : 0u;
            bf[4 * i + 2] = on ? r2 : 0u;
            bf[4 * i + 3] = on ? r3 : 0u;
        }
    }
}
__device__ __forceinline__ void md_frag_starts(const uint32_t (&b0)[8], const uint32_t (&b1)[8], float4 &c0,
                                               float4 &c1) {
    const uint32_t e8 = 0x80088008u, e128 = 0x80808080u;   // -8 and -128 times 2^-24, two f16 each
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        mma16816(d0, e8, e8, e128, e128, b0[2 * k], b0[2 * k + 1]);
        mma16816(d1, e8, e8, e128, e128, b1[2 * k], b1[2 * k + 1]);
    }
    c0 = make_float4(d0[0], d0[1], d0[2], d0[3]);
    c1 = make_float4(d1[0], d1[1], d1[2], d1[3]);
}

__device__ __forceinline__ void md_frags(float4 ld, MdScale sc, int nq, int lane, uint32_t stg, uint32_t zrow,
                                         uint32_t (&b0)[8], uint32_t (&b1)[8], float4 &c0, float4 &c1) {
    md_frag_store(ld, sc, lane, stg);
    __syncwarp();
    md_frag_load(nq, lane, stg, zrow, b0, b1);
    __syncwarp();   // the staging area may be rewritten after this
    md_frag_starts(b0, b1, c0, c1);
}

// md_frags for NR rounds at once, each with its own staging area (stg +
// r * kMdStgZero): all the stores, then all the loads, then all the chain
// starts, so that the rounds' latencies overlap.  nq: the warp's segments.
template <int NR>
__device__ __forceinline__ void md_frags_n(const float4 (&ld)[NR], MdScale sc, int nq, int lane, uint32_t stg,
                                           uint32_t zrow, uint32_t (&bf)[2 * NR][8], float4 (&c)[2 * NR]) {
#pragma unroll
    for (int r = 0; r < NR; r++) md_frag_store(ld[r], sc, lane, stg + (uint32_t)(r * kMdStgZero));
    __syncwarp();
#pragma unroll
    for (int r = 0; r < NR; r++) md_frag_load(nq - 2 * r, lane, stg + (uint32_t)(r * kMdStgZero), zrow, bf[2 * r], bf[2 * r + 1]);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < NR; r++) md_frag_starts(bf[2 * r], bf[2 * r + 1], c[2 * r], c[2 * r + 1]);
}

// A warp's share of one phase-A stage: its segments of the 16 tile rows.
//   cq: shared address of the thread's code word of row g in segment 0; rs2:
//   bytes from row g to row g + 8; cfs: the warp's chain starts, one float4
//   (hi, lo, hi, lo) per segment and one more for the sum over segments;
//   sq: scale of row g for segment 0, sr2: bytes to row g + 8's scale.
// FULL: the warp owns all kMdSegMax segments (no per-segment tests).
// CFST: bytes between the chain starts of consecutive segments.
template <bool GROUPED, int GSH, bool FULL, int SEG = kMdSegMax, int CFST = 16>
__device__ __forceinline__ void md_tileA(float (&y)[4], uint32_t cq, uint32_t rs2, uint32_t cfs, uint32_t sq,
                                         uint32_t sr2, int nq, const uint32_t (&bf)[SEG][8]) {
    if (GROUPED) {
        y[0] = y[1] = y[2] = y[3] = 0.f;
#pragma unroll
        for (int q = 0; q < SEG; q++) {
            if (FULL || q < nq) {
                const uint2 cg = lds64(cq + 32 * q), ch = lds64(cq + rs2 + 32 * q);
                float dd[4];
                md_segment_c(dd, cg, ch, bf[q], lds128f(cfs + CFST * q));
                const float sg = md_ldsf(sq + 4 * (q >> GSH)), sh = md_ldsf(sq + sr2 + 4 * (q >> GSH));
                y[0] = fmaf(sg, dd[0], y[0]);
                y[1] = fmaf(sg, dd[1], y[1]);
                y[2] = fmaf(sh, dd[2], y[2]);
                y[3] = fmaf(sh, dd[3], y[3]);
            }
        }
    } else {
        // two chains (even and odd segments) over the row
        float z[4];
        const uint2 cg0 = lds64(cq), ch0 = lds64(cq + rs2);
        md_segment_c(y, cg0, ch0, bf[0], lds128f(cfs + CFST * kMdSegMax));
        if (SEG > 1 && (FULL || nq > 1)) {
            const uint2 cg1 = lds64(cq + 32), ch1 = lds64(cq + rs2 + 32);
            md_segment_c(z, cg1, ch1, bf[SEG > 1 ? 1 : 0], make_float4(0.f, 0.f, 0.f, 0.f));
        } else {
            z[0] = z[1] = z[2] = z[3] = 0.f;
        }
#pragma unroll
        for (int q = 2; q < SEG; q++) {
            if (FULL || q < nq) {
                const uint2 cg = lds64(cq + 32 * q), ch = lds64(cq + rs2 + 32 * q);
                md_segment((q & 1) ? z : y, cg, ch, bf[q]);
            }
        }
        y[0] += z[0];
        y[1] += z[1];
        y[2] += z[2];
        y[3] += z[3];
    }
}

// The epilogue's release of a slot: one arrival that counts for all the
// consumer warps.
__device__ __forceinline__ void md_release(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(kMdWarps)
                 : "memory");
}

// A warp's bounded wait for a stage (every lane polls; false for the whole
// warp once any lane hit the deadline or the CTA aborted).
// After a failed try the warp sleeps `nap` ns (0: none), so that a waiting
// warp leaves the issue slots of its SM sub-partition to the working ones.
__device__ __forceinline__ bool md_wait(uint64_t *bar, uint32_t parity, uint64_t deadline, volatile int *abort,
                                        uint32_t nap) {
    bool ok = true;
    while (!mbar_try(bar, parity)) {
        if (*abort || global_ns() > deadline) {
            ok = false;
            break;
        }
        if (nap) __nanosleep(nap);
    }
    return __all_sync(0xffffffffu, ok);
}
// The producer lane's wait for a free slot, with the same back-off.
__device__ __forceinline__ bool md_wait1(uint64_t *bar, uint32_t parity, uint64_t deadline, volatile int *abort,
                                         uint32_t nap) {
    while (!mbar_try(bar, parity)) {
        if (*abort || global_ns() > deadline) return false;
        if (nap) __nanosleep(nap);
    }
    return true;
}

constexpr int kMd4StgBlock = 528;
constexpr int kMd4Stg = 4 * kMd4StgBlock;

// Four activation rows per B operand (the prefill's small-row groups, S <= 4
// matvecs): row t's hi half in B column 2 t, its lo half in column 2 t + 1, so
// quad lane t of the mma result holds row t's sums.  md4_frag_store: one
// round's stores for row t, as md_frag_store, into matrix rows 2 t and 2 t + 1
// of a staging area of kMd4Stg bytes (blocks of one (segment, k-step) 528
// bytes apart: the stores of one instruction fall in four bank quarters).
__device__ __forceinline__ void md4_frag_store(float4 ld, MdScale sc, int lane, int t, uint32_t stg) {
    const int seg = lane >> 4, tt = (lane >> 2) & 3, i = (lane >> 1) & 1, h = lane & 1;
    const uint32_t wb = stg + (uint32_t)((seg * 2 + i) * kMd4StgBlock + (2 * t) * 16 + (2 * tt + h) * 2);
    const float v[4] = {ld.x, ld.y, ld.z, ld.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float sv = v[q] * sc.s2k * ((q & 1) ? 0.0625f : 1.f);
        const uint32_t b = __float_as_uint(sv);
        const float h32 = __uint_as_float((b + 0xFFFu + ((b >> 13) & 1u)) & 0xFFFFE000u);
        const float l32 = (sv - h32) * 2048.f;
        uint32_t pk;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(h32), "f"(l32));   // hi in the upper half
        // matrix (operand q / 2, slot half q % 2): 8 rows of 16 bytes
        const uint32_t ad = wb + (uint32_t)((((q >> 1) * 2 + (q & 1)) * 8) * 16);
        asm volatile("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %0;\n st.shared.u16 [%1], h;\n st.shared.u16 [%2], l;\n}"
                     ::"r"(pk), "r"(ad), "r"(ad + 16));
    }
}
// md4_frag_load: the round's B registers, ldmatrix.x4 of the four matrices,
// every row real.
__device__ __forceinline__ void md4_frag_load(int nq, int lane, uint32_t stg, uint32_t (&b0)[8], uint32_t (&b1)[8]) {
    const int mq = lane >> 3, mr = lane & 7;
#pragma unroll
    for (int sg = 0; sg < 2; sg++) {
        uint32_t(&bf)[8] = sg ? b1 : b0;
        const bool on = sg < nq;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const uint32_t ra = stg + (uint32_t)((sg * 2 + i) * kMd4StgBlock + (mq * 8 + mr) * 16);
            uint32_t r0, r1, r2, r3;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                         : "r"(ra));
            bf[4 * i + 0] = on ? r0 : 0u;
            bf[4 * i + 1] = on ? r1 : 0u;
            bf[4 * i + 2] = on ? r2 : 0u;
            bf[4 * i + 3] = on ? r3 : 0u;
        }
    }
}

}  // namespace coli
