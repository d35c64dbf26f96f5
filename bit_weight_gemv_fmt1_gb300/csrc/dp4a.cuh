// dp4a.cuh -- integer-dot-product decoders for int4 (fmt 2/4) and int8 (fmt 1)
// code chunks, used by the streamed S = 1 kernels.
//
// A lane owns one 16-byte chunk of every row it visits (32 int4 codes or 16
// int8 codes) and keeps the matching activations in registers as integers:
// each x_i is scaled by one power of two 2^k, shared by the warp and chosen
// from the warp's largest |x|, and rounded to the nearest integer v_i with
// |v_i| < 2^22, so v_i carries every bit of x_i down to 2^-23 of that maximum
// (a relative error below 1.2e-7 of the largest activation of the warp).
// v_i is split into three bytes, v = 65536 t + 256 m + l (t signed, m and l
// unsigned), and the bytes of four inputs are packed into one register per
// limb.  The dot product of a chunk is then a few dp4a instructions per 32-bit
// word of codes (four code bytes against four limb bytes, exact int32
// accumulation) and one conversion to f32 per chunk:
//     sum_i c_i x_i  =  2^-k (65536 sum c t + 256 sum c m + sum c l)
// int4 codes become the signed bytes 16 (n - 8) with one LOP3 per byte-vector
// ((n ^ 8) placed in the high half of a byte and read as a signed byte is
// 16 (n - 8)), so the offset is removed inside the integer sum; int8 codes
// (stored offset binary) are taken unsigned and the offset comes off as
// 128 * sum(x).  On GB300 the int4 chunk costs about 16 issue cycles per 128
// bytes of codes and warp, against about 26 for an f32 decode of the same
// codes (the integer ALU, which the f32 decode needs once per code, runs at
// half rate and does not overlap with the f32 FMA pipe).
#pragma once

#include "coli_internal.cuh"

namespace coli {

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {   // both signed bytes
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {   // a signed, b unsigned bytes
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {   // a unsigned, b signed bytes
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {   // both unsigned bytes
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// The same with a zero accumulator (no register to clear).
__device__ __forceinline__ int dp4a_ss0(uint32_t a, uint32_t b) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, 0;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ int dp4a_su0(uint32_t a, uint32_t b) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, 0;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ int dp4a_us0(uint32_t a, uint32_t b) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, 0;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ int dp4a_uu0(uint32_t a, uint32_t b) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, 0;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t lop3_xor_and(uint32_t a, uint32_t x, uint32_t m) {   // (a ^ x) & m
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(d) : "r"(a), "r"(x), "r"(m));
    return d;
}

// 2^e as a float, -126 <= e <= 127.
__device__ __forceinline__ float d4_exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Largest |x| bit pattern (sign cleared) over the NIN values of every lane of
// the warp; NaN patterns sort above infinity.
template <int NIN>
__device__ __forceinline__ uint32_t d4_warp_maxbits(const float (&x)[NIN]) {
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < NIN; i++) mb = max(mb, __float_as_uint(x[i]) & 0x7FFFFFFFu);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    return mb;
}
// Exponent k from the largest magnitude (as bits): |x| 2^k < 2^22 for every
// |x| up to it (k <= 126 so that 2^k is a normal float; values below 2^-104
// keep fewer bits, far below any representable contribution).
__device__ __forceinline__ int d4_exp(uint32_t maxbits) { return min(148 - (int)(maxbits >> 23), 126); }
// The factor that turns a reduced integer-scaled dot product back into units
// of x: 2^-(k + extra), or NaN when an activation is not finite (so that the
// result is not a finite number either).
__device__ __forceinline__ float d4_unscale(uint32_t maxbits, int extra) {
    if ((maxbits >> 23) >= 255u) return __int_as_float(0x7FC00000);
    const int k = d4_exp(maxbits);
    return d4_exp2i(-k) * d4_exp2i(-extra);
}

// round(x * 2^k) for |x * 2^k| < 2^22: adding 1.5 * 2^23 leaves the rounded
// integer in the low mantissa bits (one rounding, to nearest even).
__device__ __forceinline__ int d4_round_int(float x, float s2k) {
    return __float_as_int(fmaf(x, s2k, 12582912.0f)) - 0x4B400000;
}

__device__ __forceinline__ uint32_t d4_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The three limb words of four integers v0..v3 (|v| < 2^22): byte j of each
// word comes from v_j; t takes bits 16-23 (the signed top byte), m bits 8-15,
// l bits 0-7.
__device__ __forceinline__ void d4_pack4(int v0, int v1, int v2, int v3, uint32_t &t, uint32_t &m, uint32_t &l) {
    const uint32_t p01 = d4_prmt(v0, v1, 0x5140u), p23 = d4_prmt(v2, v3, 0x5140u);   // bytes 0 and 1
    const uint32_t q01 = d4_prmt(v0, v1, 0x7362u), q23 = d4_prmt(v2, v3, 0x7362u);   // bytes 2 and 3
    l = d4_prmt(p01, p23, 0x5410u);
    m = d4_prmt(p01, p23, 0x7632u);
    t = d4_prmt(q01, q23, 0x5410u);
}

// int4 codes, 32 inputs per lane (16 code bytes).  Byte j of word w holds
// input 8w + 2j (low nibble) and 8w + 2j + 1 (high nibble); limb word 2w + h
// packs the inputs 8w + 2j + h, j = 0..3.  dotn gives 16 * sum (n - 8) x 2^k
// per chunk: UNSCALE_EXTRA = 4.
struct D4Nib {
    static constexpr int LB = 16, NIN = 32, UNSCALE_EXTRA = 4;
    static constexpr int SPW = 1;   // 512-byte slabs one warp of the decode block's phase B covers
    uint32_t t[8], m[8], l[8];
    __device__ __forceinline__ void set(const float (&x)[NIN], int k) {
        const float s2k = d4_exp2i(k);
#pragma unroll
        for (int w = 0; w < 4; w++)
#pragma unroll
            for (int h = 0; h < 2; h++)
                d4_pack4(d4_round_int(x[8 * w + h], s2k), d4_round_int(x[8 * w + 2 + h], s2k),
                         d4_round_int(x[8 * w + 4 + h], s2k), d4_round_int(x[8 * w + 6 + h], s2k), t[2 * w + h],
                         m[2 * w + h], l[2 * w + h]);
    }
    // integer-scaled dot products (offset removed, no scale) of N code chunks
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        int at[N], am[N], al[N];
#pragma unroll
        for (int w = 0; w < 4; w++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t c = w == 0 ? q[d].x : w == 1 ? q[d].y : w == 2 ? q[d].z : q[d].w;
                // 16 (n - 8) as signed bytes: low nibbles moved up, high nibbles in place
                const uint32_t lo = lop3_xor_and(c * 16u, 0x88888880u, 0xF0F0F0F0u);
                const uint32_t hi = lop3_xor_and(c, 0x88888888u, 0xF0F0F0F0u);
                if (w == 0) {
                    at[d] = dp4a_ss0(lo, t[0]);
                    am[d] = dp4a_su0(lo, m[0]);
                    al[d] = dp4a_su0(lo, l[0]);
                } else {
                    at[d] = dp4a_ss(lo, t[2 * w], at[d]);
                    am[d] = dp4a_su(lo, m[2 * w], am[d]);
                    al[d] = dp4a_su(lo, l[2 * w], al[d]);
                }
                at[d] = dp4a_ss(hi, t[2 * w + 1], at[d]);
                am[d] = dp4a_su(hi, m[2 * w + 1], am[d]);
                al[d] = dp4a_su(hi, l[2 * w + 1], al[d]);
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = fmaf((float)at[d], 65536.0f, (float)(am[d] * 256 + al[d]));
    }
};

// int8 codes stored offset binary (u = code + 128), 16 inputs per lane; byte j
// of word w holds input 4w + j.  dotn gives (sum u x - 128 sum x) 2^k per
// chunk: UNSCALE_EXTRA = 0.
struct D4Byte {
    static constexpr int LB = 16, NIN = 16, UNSCALE_EXTRA = 0;
    static constexpr int SPW = 2;
    uint32_t t[4], m[4], l[4];
    float xo;   // 128 * sum(x) * 2^k
    __device__ __forceinline__ void set(const float (&x)[NIN], int k) {
        const float s2k = d4_exp2i(k);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NIN; i++) s += x[i];
        xo = 128.0f * s * s2k;
#pragma unroll
        for (int w = 0; w < 4; w++)
            d4_pack4(d4_round_int(x[4 * w], s2k), d4_round_int(x[4 * w + 1], s2k), d4_round_int(x[4 * w + 2], s2k),
                     d4_round_int(x[4 * w + 3], s2k), t[w], m[w], l[w]);
    }
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        int at[N], am[N], al[N];
#pragma unroll
        for (int w = 0; w < 4; w++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t c = w == 0 ? q[d].x : w == 1 ? q[d].y : w == 2 ? q[d].z : q[d].w;
                if (w == 0) {
                    at[d] = dp4a_us0(c, t[0]);
                    am[d] = dp4a_uu0(c, m[0]);
                    al[d] = dp4a_uu0(c, l[0]);
                } else {
                    at[d] = dp4a_us(c, t[w], at[d]);
                    am[d] = dp4a_uu(c, m[w], am[d]);
                    al[d] = dp4a_uu(c, l[w], al[d]);
                }
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = fmaf((float)at[d], 65536.0f, (float)(am[d] * 256 + al[d])) - xo;
    }
};

// Load the NIN activations of lane chunk c (inputs c*NIN ..) of a vector of n
// floats; inputs past n read as zero.  ld: load function (e.g. __ldg, __ldcg).
template <int NIN, class LD>
__device__ __forceinline__ void d4_load_chunk(const float *x, long long n, long long c, float (&v)[NIN], LD ld) {
    const long long i0 = c * NIN;
    if (i0 + NIN <= n && (reinterpret_cast<uintptr_t>(x + i0) & 15) == 0) {
#pragma unroll
        for (int j = 0; j < NIN / 4; j++) {
            const float4 a = ld(reinterpret_cast<const float4 *>(x + i0) + j);
            v[4 * j] = a.x;
            v[4 * j + 1] = a.y;
            v[4 * j + 2] = a.z;
            v[4 * j + 3] = a.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < NIN; j++) v[j] = (i0 + j < n) ? ld(x + i0 + j) : 0.f;
    }
}

}  // namespace coli
