// dp4a.cuh -- integer-dot-product decoders for int4 (fmt 2/4) and int8 (fmt 1)
// code chunks, used by the streamed S = 1 kernels.
//
// A lane owns one 16-byte chunk of every row it visits (32 int4 codes or 16
// int8 codes) and keeps the matching activations in registers as integers:
// each x_i of the chunk is scaled by one power of two 2^k, chosen from the
// chunk's largest |x|, and rounded to the nearest integer v_i with
// |v_i| < 2^22, so v_i carries every bit of x_i down to 2^-23 of that maximum
// (a relative error below 1.2e-7 of the chunk's largest activation).
// v_i is split into three bytes, v = 65536 t + 256 m + l (t signed, m and l
// unsigned), and the bytes of four inputs are packed into one register per
// limb.  The dot product of a chunk is then a handful of dp4a instructions per
// 32-bit word of codes (four unsigned code bytes against four limb bytes,
// exact int32 accumulation), and one conversion to f32 per chunk:
//     sum_i n_i x_i  =  2^-k (65536 sum n t + 256 sum n m + sum n l)
// The code offset (8 for int4, 128 for the offset-binary int8 layout) comes off
// as offset * sum_i x_i.  On GB300 this costs about 16 issue cycles per 128
// bytes of int4 codes and warp, against about 26 for the f32 decode of the
// same codes (the integer ALU, which the f32 decode needs once per code, runs
// at half rate and does not overlap with the f32 FMA pipe).
#pragma once

#include "coli_internal.cuh"

namespace coli {

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {   // a: unsigned bytes, b: signed bytes
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {   // both unsigned bytes
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 2^e as a float, -126 <= e <= 127.
__device__ __forceinline__ float d4_exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Chunk exponent from the largest magnitude mx: |x| 2^k < 2^22 for every
// |x| <= mx (k <= 126 so that 2^k is a normal float; chunks below 2^-104 keep
// fewer bits, far below any representable contribution).
__device__ __forceinline__ int d4_chunk_exp(float mx) {
    const int eb = (__float_as_int(mx) >> 23) & 0xFF;   // mx < 2^(eb - 126)
    return min(148 - eb, 126);
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
// packs the inputs 8w + 2j + h, j = 0..3.
struct D4Nib {
    static constexpr int LB = 16, NIN = 32, OFFSET = 8;
    static constexpr int SPW = 1;   // 512-byte slabs one warp of the decode block's phase B covers
    uint32_t t[8], m[8], l[8];
    float inv, xo;   // 2^-k, OFFSET * sum(x)
    __device__ __forceinline__ void set(const float (&x)[NIN]) {
        float mx = 0.f, s = 0.f;
#pragma unroll
        for (int i = 0; i < NIN; i++) {
            mx = fmaxf(mx, fabsf(x[i]));
            s += x[i];
        }
        const int k = d4_chunk_exp(mx);
        const float s2k = d4_exp2i(k);
        inv = d4_exp2i(-k);
        xo = (float)OFFSET * s;
#pragma unroll
        for (int w = 0; w < 4; w++)
#pragma unroll
            for (int h = 0; h < 2; h++)
                d4_pack4(d4_round_int(x[8 * w + h], s2k), d4_round_int(x[8 * w + 2 + h], s2k),
                         d4_round_int(x[8 * w + 4 + h], s2k), d4_round_int(x[8 * w + 6 + h], s2k), t[2 * w + h],
                         m[2 * w + h], l[2 * w + h]);
    }
    // dot products (offset removed, no scale) of N code chunks with the activations
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        int at[N], am[N], al[N];
#pragma unroll
        for (int d = 0; d < N; d++) at[d] = am[d] = al[d] = 0;
#pragma unroll
        for (int w = 0; w < 4; w++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t c = w == 0 ? q[d].x : w == 1 ? q[d].y : w == 2 ? q[d].z : q[d].w;
                const uint32_t lo = c & 0x0F0F0F0Fu, hi = (c >> 4) & 0x0F0F0F0Fu;
                at[d] = dp4a_us(lo, t[2 * w], at[d]);
                at[d] = dp4a_us(hi, t[2 * w + 1], at[d]);
                am[d] = dp4a_uu(lo, m[2 * w], am[d]);
                am[d] = dp4a_uu(hi, m[2 * w + 1], am[d]);
                al[d] = dp4a_uu(lo, l[2 * w], al[d]);
                al[d] = dp4a_uu(hi, l[2 * w + 1], al[d]);
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = fmaf(fmaf((float)at[d], 65536.0f, (float)(am[d] * 256 + al[d])), inv, -xo);
    }
};

// int8 codes stored offset binary (u = code + 128), 16 inputs per lane; byte j
// of word w holds input 4w + j.
struct D4Byte {
    static constexpr int LB = 16, NIN = 16, OFFSET = 128;
    static constexpr int SPW = 2;
    uint32_t t[4], m[4], l[4];
    float inv, xo;
    __device__ __forceinline__ void set(const float (&x)[NIN]) {
        float mx = 0.f, s = 0.f;
#pragma unroll
        for (int i = 0; i < NIN; i++) {
            mx = fmaxf(mx, fabsf(x[i]));
            s += x[i];
        }
        const int k = d4_chunk_exp(mx);
        const float s2k = d4_exp2i(k);
        inv = d4_exp2i(-k);
        xo = (float)OFFSET * s;
#pragma unroll
        for (int w = 0; w < 4; w++)
            d4_pack4(d4_round_int(x[4 * w], s2k), d4_round_int(x[4 * w + 1], s2k), d4_round_int(x[4 * w + 2], s2k),
                     d4_round_int(x[4 * w + 3], s2k), t[w], m[w], l[w]);
    }
    template <int N>
    __device__ __forceinline__ void dotn(const uint4 (&q)[N], float (&out)[N]) const {
        int at[N], am[N], al[N];
#pragma unroll
        for (int d = 0; d < N; d++) at[d] = am[d] = al[d] = 0;
#pragma unroll
        for (int w = 0; w < 4; w++) {
#pragma unroll
            for (int d = 0; d < N; d++) {
                const uint32_t c = w == 0 ? q[d].x : w == 1 ? q[d].y : w == 2 ? q[d].z : q[d].w;
                at[d] = dp4a_us(c, t[w], at[d]);
                am[d] = dp4a_uu(c, m[w], am[d]);
                al[d] = dp4a_uu(c, l[w], al[d]);
            }
        }
#pragma unroll
        for (int d = 0; d < N; d++) out[d] = fmaf(fmaf((float)at[d], 65536.0f, (float)(am[d] * 256 + al[d])), inv, -xo);
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
