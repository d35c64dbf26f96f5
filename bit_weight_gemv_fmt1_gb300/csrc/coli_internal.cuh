// coli_internal.cuh -- shared definitions of the CUDA library (not installed).
//
// Device layout of an uploaded matrix W [O][I]:
//   q  : O rows of `rs` bytes, rs = row_bytes rounded up to 16; the padding is
//        zero.  fmt=1 bytes are stored offset binary (b ^ 0x80) so that every
//        integer format decodes as (unsigned code - offset).  fmt 2/3/4 keep
//        the host nibble/crumb order; fmt=0 keeps the f32 values; fmt=7
//        keeps the host FP8 E4M3 bytes.
//   s  : f32 scales exactly as on the host ([O], [O][ng], or for fmt=7
//        [ceil(O/128)][ng] with ng = ceil(I/128)); none for fmt=0.
//
// The bandwidth-bound kernels stream each row as 16-byte chunks, lane l of a
// warp taking chunks l, l+32, l+64, ...  A chunk holds EPC elements (4, 16,
// 32, 64, 32 for fmt 0..4, 16 for fmt 7).  The activations are staged in shared memory in an
// order made for those chunks (see stage_vec): the four floats a lane needs
// for one 32-bit word of codes are one 16-byte shared load, and the float4
// units of a chunk are XOR-swizzled by the chunk index so that the 8 lanes of
// a shared-memory phase hit 8 different bank groups.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "coli.h"

struct coli_tensor {
    int fmt, gs, ng, device;   // fmt: the device layout's format (int3 is stored as int4, below)
    int ufmt;                  // the format the caller uploaded
    int64_t O, I;
    int64_t rs;          // device row stride in bytes (multiple of 16)
    int cpr;             // 16-byte chunks per row that hold data
    uint8_t *q;          // device codes
    float *s;            // device scales (NULL for fmt=0)
    int64_t dev_bytes, alg_bytes;
    uint64_t uid;        // unique per upload, never reused
    void *tmap;          // device copy of the codes' TMA descriptor (int4 formats), else NULL
    int host;            // 1: codes and scales live in pinned host memory (q, s are the
                         //    device-side addresses of that mapping; hq, hs the host ones)
    void *hq, *hs;
};

namespace coli {

// ------------------------------------------------------------------ errors
// Device-side error codes recorded in the per-device error word.
enum : int { DEV_ERR_NONE = 0, DEV_ERR_TIMEOUT = 1, DEV_ERR_BAD_ID = 2 };

// ------------------------------------------------------------------ traits
template <int FMT> struct Fmt;
template <> struct Fmt<0> { static constexpr int EPC = 4; };
template <> struct Fmt<1> { static constexpr int EPC = 16; };
template <> struct Fmt<2> { static constexpr int EPC = 32; };
template <> struct Fmt<3> { static constexpr int EPC = 64; };
template <> struct Fmt<4> { static constexpr int EPC = 32; };
template <> struct Fmt<7> { static constexpr int EPC = 16; };

__host__ __device__ inline int epc_of(int fmt) {
    return fmt == 0 ? 4 : (fmt == 1 || fmt == 7) ? 16 : fmt == 3 ? 64 : 32;
}

// Formats whose scale changes along a row: fmt=4 (one scale per gs inputs)
// and fmt=7 (one scale per 128 x 128 block).
template <int FMT> constexpr bool kGrouped = FMT == 4 || FMT == 7;
constexpr int kFp8Block = 128;   // fmt=7 block edge, rows and inputs

// 16-byte chunks per scale group of a row: gs / 32 for fmt=4, 8 for fmt=7.
__host__ __device__ inline int chunks_per_group(int fmt, int gs) {
    return fmt == 7 ? kFp8Block / 16 : fmt == 4 ? gs / 32 : 1;
}

// Length (floats) of one staged activation vector for a row of `cpr` chunks:
// a whole number of warp iterations, so every lane of the last iteration
// reads zeros instead of running past the end.
__host__ __device__ inline int staged_len(int fmt, int cpr) {
    return ((cpr + 31) / 32) * 32 * epc_of(fmt);
}

// Position of element e of a staged vector.
template <int FMT>
__device__ __forceinline__ int stage_pos(int e) {
    if constexpr (FMT == 0) {
        return e;
    } else if constexpr (FMT == 1 || FMT == 7) {
        const int c = e >> 4, r = e & 15;
        return c * 16 + (((r >> 2) ^ ((c >> 1) & 3)) << 2) + (r & 3);
    } else if constexpr (FMT == 2 || FMT == 4) {
        // per 8-element word: order x0 x1 x2 x5 | x3 x6 x4 x7 (pairs that
        // match the packed f32x2 lanes of dot_word4)
        const int c = e >> 5, r = e & 31;
        const int k = r & 7;
        const int pos = (0x75364210 >> (4 * k)) & 0xF;   // 0,1,2,4,6,3,5,7
        const int within = (r & ~7) + pos;
        return c * 32 + (((within >> 2) ^ (c & 7)) << 2) + (within & 3);
    } else {
        const int c = e >> 6, r = e & 63;
        return c * 64 + (((r >> 2) ^ (c & 7)) << 2) + (r & 3);
    }
}

// Stage one activation vector src[0..n) into dst[0..len) (zeros past n);
// len is a multiple of 8.  Each thread takes groups of 8 consecutive inputs
// and issues the loads of UN groups (two 16-byte loads each when src is
// 16-byte aligned) before any store, so a CTA pays about one memory round
// trip per UN * nthreads * 8 inputs instead of one per nthreads inputs.
// Loads go through L2 (.cg): src may have been written earlier in the same
// kernel by other CTAs.
template <int FMT>
__device__ __forceinline__ void stage_vec(float *dst, const float *src, int n, int len, int tid, int nthreads) {
    constexpr int UN = 4;
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    const int ng = len >> 3;
    for (int g0 = tid; g0 < ng; g0 += nthreads * UN) {
        float v[UN][8];
#pragma unroll
        for (int u = 0; u < UN; u++) {
            const int e0 = (g0 + u * nthreads) * 8;
            if (g0 + u * nthreads < ng && vec && e0 + 8 <= n) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + e0));
                const float4 b = __ldcg(reinterpret_cast<const float4 *>(src + e0 + 4));
                v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                v[u][4] = b.x; v[u][5] = b.y; v[u][6] = b.z; v[u][7] = b.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++) v[u][i] = (g0 + u * nthreads < ng && e0 + i < n) ? __ldcg(src + e0 + i) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < UN; u++) {
            const int g = g0 + u * nthreads;
            if (g < ng) {
#pragma unroll
                for (int i = 0; i < 8; i++) dst[stage_pos<FMT>(g * 8 + i)] = v[u][i];
            }
        }
    }
}

// ------------------------------------------------------------- primitives
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float lop_mag(uint32_t w, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(magic));   // (w & mask) | magic
    return __uint_as_float(r);
}

__device__ __forceinline__ float prmt_byte(uint32_t w, uint32_t magic, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(magic), "r"(sel));
    return __uint_as_float(r);
}

union F2U {
    float2 f;
    unsigned long long u;
};

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    F2U A{a}, B{b}, D;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(D.u) : "l"(A.u), "l"(B.u));
    return D.f;
}

__device__ __forceinline__ void ffma2(float2 &acc, float2 a, float2 b) {
    F2U A{a}, B{b}, C{acc};
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(C.u) : "l"(A.u), "l"(B.u));
    acc = C.f;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ----------------------------------------------------- per-format decode
// Each 32-bit word of codes is turned into f32 values with one lop3 / prmt
// per element: the code is OR-ed into the mantissa of 1.0 (or 2^23 for int8),
// which gives 1 + code * 2^(p-23) exactly, and one packed subtract removes the
// offset exactly (both operands lie in [1,2)).  The result (code - offset) *
// 2^(p-23) is multiplied into a per-bit-position ("class") accumulator; the
// classes are re-scaled by 2^(23-p), a power of two, when they are combined.

// int4, 8 elements: classes (p0|p4) (p8|p8) (p12|p12) (p16|p16)
struct Acc4 { float2 a01, a25, a36, a47; };
__device__ __forceinline__ void acc_zero(Acc4 &a) {
    a.a01 = a.a25 = a.a36 = a.a47 = make_float2(0.f, 0.f);
}
__device__ __forceinline__ float acc_combine(const Acc4 &a) {
    return a.a01.x * 8388608.0f + a.a01.y * 524288.0f + (a.a25.x + a.a25.y) * 32768.0f +
           (a.a36.x + a.a36.y) * 2048.0f + (a.a47.x + a.a47.y) * 128.0f;
}
struct Dec4 { float2 v01, v25, v36, v47; };
__device__ __forceinline__ Dec4 decode4(uint32_t w) {
    const uint32_t M = 0x3F800000u;
    const uint32_t b = w >> 12;
    Dec4 d;
    d.v01 = fadd2(make_float2(lop_mag(w, 0xFu, M), lop_mag(w, 0xF0u, M)),
                  make_float2(-__uint_as_float(M | (8u << 0)), -__uint_as_float(M | (8u << 4))));
    d.v25 = fadd2(make_float2(lop_mag(w, 0xF00u, M), lop_mag(b, 0xF00u, M)),
                  make_float2(-__uint_as_float(M | (8u << 8)), -__uint_as_float(M | (8u << 8))));
    d.v36 = fadd2(make_float2(lop_mag(w, 0xF000u, M), lop_mag(b, 0xF000u, M)),
                  make_float2(-__uint_as_float(M | (8u << 12)), -__uint_as_float(M | (8u << 12))));
    d.v47 = fadd2(make_float2(lop_mag(w, 0xF0000u, M), lop_mag(b, 0xF0000u, M)),
                  make_float2(-__uint_as_float(M | (8u << 16)), -__uint_as_float(M | (8u << 16))));
    return d;
}
__device__ __forceinline__ void fma4(Acc4 &a, const Dec4 &d, float4 x0, float4 x1) {
    ffma2(a.a01, d.v01, make_float2(x0.x, x0.y));
    ffma2(a.a25, d.v25, make_float2(x0.z, x0.w));
    ffma2(a.a36, d.v36, make_float2(x1.x, x1.y));
    ffma2(a.a47, d.v47, make_float2(x1.z, x1.w));
}

// int8 (stored offset binary), 4 elements, one class: 2^23 + u - (2^23 + 128)
struct Acc1 { float2 a, b; };
__device__ __forceinline__ void acc_zero(Acc1 &a) { a.a = a.b = make_float2(0.f, 0.f); }
__device__ __forceinline__ float acc_combine(const Acc1 &a) { return (a.a.x + a.a.y) + (a.b.x + a.b.y); }
struct Dec1 { float2 v01, v23; };
__device__ __forceinline__ Dec1 decode1(uint32_t w) {
    const uint32_t M = 0x4B000000u;
    const float2 off = make_float2(-8388736.0f, -8388736.0f);   // -(2^23 + 128)
    Dec1 d;
    d.v01 = fadd2(make_float2(prmt_byte(w, M, 0x7650u), prmt_byte(w, M, 0x7651u)), off);
    d.v23 = fadd2(make_float2(prmt_byte(w, M, 0x7652u), prmt_byte(w, M, 0x7653u)), off);
    return d;
}
__device__ __forceinline__ void fma1(Acc1 &a, const Dec1 &d, float4 x) {
    ffma2(a.a, d.v01, make_float2(x.x, x.y));
    ffma2(a.b, d.v23, make_float2(x.z, x.w));
}

// int2, 16 elements as 4 byte views (shift 0/8/16/24), classes (p0|p2) (p4|p6);
// two copies of the accumulators (even / odd views) for instruction-level
// parallelism.
struct Acc3 { float2 a0, b0, a1, b1; };
__device__ __forceinline__ void acc_zero(Acc3 &a) {
    a.a0 = a.b0 = a.a1 = a.b1 = make_float2(0.f, 0.f);
}
__device__ __forceinline__ float acc_combine(const Acc3 &a) {
    return (a.a0.x + a.a1.x) * 8388608.0f + (a.a0.y + a.a1.y) * 2097152.0f +
           (a.b0.x + a.b1.x) * 524288.0f + (a.b0.y + a.b1.y) * 131072.0f;
}
__device__ __forceinline__ void view3(float2 &va, float2 &vb, uint32_t v) {
    const uint32_t M = 0x3F800000u;
    va = fadd2(make_float2(lop_mag(v, 0x3u, M), lop_mag(v, 0xCu, M)),
               make_float2(-__uint_as_float(M | (2u << 0)), -__uint_as_float(M | (2u << 2))));
    vb = fadd2(make_float2(lop_mag(v, 0x30u, M), lop_mag(v, 0xC0u, M)),
               make_float2(-__uint_as_float(M | (2u << 4)), -__uint_as_float(M | (2u << 6))));
}

// FP8 E4M3, 4 elements: the conversion instruction turns each byte pair into
// an exact f16 pair (E4M3 values, subnormals and NaN included, are all f16
// values), widened exactly to f32.  Accumulates into an Acc1.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t pair16) {
    uint32_t h2;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h2) : "r"(pair16));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}
__device__ __forceinline__ Dec1 decode7(uint32_t w) {
    Dec1 d;
    d.v01 = e4m3x2_to_f32x2(w & 0xFFFFu);
    d.v23 = e4m3x2_to_f32x2(w >> 16);
    return d;
}

// f32 weights, 4 per chunk
struct Acc0 { float2 a, b; };
__device__ __forceinline__ void acc_zero(Acc0 &a) { a.a = a.b = make_float2(0.f, 0.f); }
__device__ __forceinline__ float acc_combine(const Acc0 &a) { return (a.a.x + a.a.y) + (a.b.x + a.b.y); }

template <int FMT> struct AccOf;
template <> struct AccOf<0> { using T = Acc0; };
template <> struct AccOf<1> { using T = Acc1; };
template <> struct AccOf<2> { using T = Acc4; };
template <> struct AccOf<3> { using T = Acc3; };
template <> struct AccOf<4> { using T = Acc4; };
template <> struct AccOf<7> { using T = Acc1; };

// Multiply-accumulate one 16-byte chunk `q` of codes against the staged
// activations of that chunk (xs4 points at the chunk's first float4 unit of
// one activation vector; c7 = chunk index & 7 selects the swizzle).
template <int FMT>
__device__ __forceinline__ void chunk_fma(typename AccOf<FMT>::T &acc, uint4 q, const float4 *xs4, int c) {
    if constexpr (FMT == 2 || FMT == 4) {
        const int sw = c & 7;
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const Dec4 d = decode4(wv[t]);
            fma4(acc, d, xs4[(2 * t) ^ sw], xs4[(2 * t + 1) ^ sw]);
        }
    } else if constexpr (FMT == 1) {
        const int sw = (c >> 1) & 3;
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; t++) fma1(acc, decode1(wv[t]), xs4[t ^ sw]);
    } else if constexpr (FMT == 7) {
        const int sw = (c >> 1) & 3;
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; t++) fma1(acc, decode7(wv[t]), xs4[t ^ sw]);
    } else if constexpr (FMT == 3) {
        const int sw = c & 7;
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; t++) {
#pragma unroll
            for (int m = 0; m < 4; m++) {
                const uint32_t v = m == 0 ? wv[t] : (wv[t] >> (8 * m));
                float2 va, vb;
                view3(va, vb, v);
                const float4 x = xs4[(4 * t + m) ^ sw];
                if (m & 1) {
                    ffma2(acc.a1, va, make_float2(x.x, x.y));
                    ffma2(acc.b1, vb, make_float2(x.z, x.w));
                } else {
                    ffma2(acc.a0, va, make_float2(x.x, x.y));
                    ffma2(acc.b0, vb, make_float2(x.z, x.w));
                }
            }
        }
    } else {
        const float4 x = xs4[0];
        ffma2(acc.a, make_float2(__uint_as_float(q.x), __uint_as_float(q.y)), make_float2(x.x, x.y));
        ffma2(acc.b, make_float2(__uint_as_float(q.z), __uint_as_float(q.w)), make_float2(x.z, x.w));
    }
}

// Dot products of R matrix rows against NS staged activation vectors, by one
// warp.  rows[r] = row base pointers (16-byte aligned), scl[r] = the row's
// scales (per-row formats: one float; fmt=4: ng floats; fmt=7: the ng floats
// of the row's block-row), gpc[r] = chunks per scale group of row r for the
// grouped formats (chunks_per_group).  xsv[n] = staged vector n.  Results are the
// warp-reduced sums, valid in every lane.
template <int FMT, int R, int NS>
__device__ __forceinline__ void dot_rows(const uint8_t *const (&rows)[R], const float *const (&scl)[R],
                                         const int (&gpc)[R], const float *const (&xsv)[NS], int cpr,
                                         int lane, float (&out)[R][NS]) {
    using Acc = typename AccOf<FMT>::T;
    constexpr int U = ((FMT == 3) ? 4 : 8) / R > 0 ? ((FMT == 3) ? 4 : 8) / R : 1;   // chunks per row loaded ahead
    float y[R][NS];
#pragma unroll
    for (int r = 0; r < R; r++)
#pragma unroll
        for (int n = 0; n < NS; n++) y[r][n] = 0.f;
    Acc acc[R][NS];
    if constexpr (!kGrouped<FMT>) {
#pragma unroll
        for (int r = 0; r < R; r++)
#pragma unroll
            for (int n = 0; n < NS; n++) acc_zero(acc[r][n]);
    }
    const int n_iter = (cpr + 31) >> 5;
    for (int it0 = 0; it0 < n_iter; it0 += U) {
        uint4 q[U][R];
        float sc[U][R];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int c = (it0 + u) * 32 + lane;
            const bool ok = (it0 + u < n_iter) && c < cpr;
#pragma unroll
            for (int r = 0; r < R; r++) {
                q[u][r] = ok ? ld_stream(rows[r] + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
                if constexpr (kGrouped<FMT>) sc[u][r] = ok ? __ldg(scl[r] + c / gpc[r]) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            if (it0 + u >= n_iter) break;
            const int c = (it0 + u) * 32 + lane;
            const int EPC = Fmt<FMT>::EPC;
            if constexpr (kGrouped<FMT>) {
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int n = 0; n < NS; n++) acc_zero(acc[r][n]);
            }
#pragma unroll
            for (int n = 0; n < NS; n++) {
                const float4 *xs4 = reinterpret_cast<const float4 *>(xsv[n] + (size_t)c * EPC);
#pragma unroll
                for (int r = 0; r < R; r++) chunk_fma<FMT>(acc[r][n], q[u][r], xs4, c);
            }
            if constexpr (kGrouped<FMT>) {
#pragma unroll
                for (int r = 0; r < R; r++)
#pragma unroll
                    for (int n = 0; n < NS; n++) y[r][n] = fmaf(sc[u][r], acc_combine(acc[r][n]), y[r][n]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; r++) {
        float rs = 1.f;
        if constexpr (FMT == 1 || FMT == 2 || FMT == 3) rs = __ldg(scl[r]);
#pragma unroll
        for (int n = 0; n < NS; n++) {
            float v;
            if constexpr (kGrouped<FMT>) v = y[r][n];
            else if constexpr (FMT == 0) v = acc_combine(acc[r][n]);
            else v = rs * acc_combine(acc[r][n]);
            out[r][n] = warp_sum(v);
        }
    }
}

// Generic path for fmt=4 with a group size that is not a multiple of 32
// (any even gs): one element at a time with its own group scale.
__device__ __forceinline__ float dot_row_fmt4_generic(const uint8_t *row, const float *scl, int gs, int I,
                                                      const float *x, int lane) {
    float acc = 0.f;
    for (int i = lane; i < I; i += 32) {
        const uint8_t b = row[i >> 1];
        const int code = (i & 1) ? (b >> 4) : (b & 0xF);
        acc = fmaf((float)(code - 8) * __ldg(scl + i / gs), x[i], acc);
    }
    return warp_sum(acc);
}

// ------------------------------------------------- programmatic dependent launch
// The matvec kernels are launched with programmatic stream serialization: a
// kernel lets the next one in the stream begin launching once every thread of
// every CTA has finished its main loop (pdl_trigger; only the short epilogue
// is left), and waits for the previous kernel to complete, with its writes
// visible, before it reads activations or writes outputs (pdl_wait).
// Weights and scales never change between kernels, so their loads may be
// issued before the wait.  Triggering at the end of the main loop keeps at
// most one kernel ahead resident; an early trigger let several waiting grids
// pile up on the SMs and cut the running kernel's occupancy.  Without a
// programmatic predecessor or dependent both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- timing
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ------------------------------------------------------------- host side

// Launch helpers implemented in the .cu files.
struct GemvJob {
    static constexpr int MAXM = 16;
    const uint8_t *q[MAXM];
    const float *s[MAXM];
    float *y[MAXM];
    int O[MAXM];
    int gs[MAXM];
    int ng[MAXM];
    long long rs[MAXM];
    int row_start[MAXM + 1];   // prefix of O over matrices
    int n, fmt, I, cpr, S;
    const float *x;
    int *err;                  // device error word (streamed matvec only)
};

cudaError_t launch_gemv(const GemvJob &job, cudaStream_t st, int *n_launch);

// Launch `kern` with programmatic stream serialization allowed (see pdl_wait).
template <class... P, class... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

}  // namespace coli

namespace coli {

// Device view of one uploaded matrix.
struct MatDesc {
    const uint8_t *q;
    const float *s;
    long long rs;
    int gs, ng;
    const void *tmap;         // device copy of the codes' TMA descriptor (int4 formats), else NULL
};
// gate, up, down of one routed expert.
struct ExpertDesc {
    MatDesc m[3];
};

// Scales of row `row` of a matrix as dot_rows and decode_elem take them: the
// row's own scale(s), or for fmt=7 the scales of the row's block-row.
__device__ __forceinline__ const float *row_scales(int fmt, const MatDesc &m, int row) {
    if (fmt == 0) return nullptr;
    if (fmt == 4) return m.s + (size_t)row * m.ng;
    if (fmt == 7) return m.s + (size_t)(row / kFp8Block) * m.ng;
    return m.s + row;
}

// Value of one FP8 E4M3 byte (exact, through f16).
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) { return e4m3x2_to_f32x2(b).x; }

// Decode one element (o fixed by `row`, input index i) of the device layout,
// scale included (rscale = row_scales of the row).  Used by the tiled GEMM
// and the gather kernels.
__device__ __forceinline__ float decode_elem(int fmt, const uint8_t *row, const float *rscale, int gs, int i) {
    switch (fmt) {
    case 0: return reinterpret_cast<const float *>(row)[i];
    case 1: return (float)((int)row[i] - 128) * rscale[0];
    case 2: { const uint8_t b = row[i >> 1]; return (float)(((i & 1) ? (b >> 4) : (b & 0xF)) - 8) * rscale[0]; }
    case 3: { const uint8_t b = row[i >> 2]; return (float)(((b >> (2 * (i & 3))) & 3) - 2) * rscale[0]; }
    case 7: return e4m3_to_f32(row[i]) * rscale[i / kFp8Block];
    default: { const uint8_t b = row[i >> 1]; return (float)(((i & 1) ? (b >> 4) : (b & 0xF)) - 8) * rscale[i / gs]; }
    }
}

// Arguments of the single-launch decode expert block.
struct MoeDecodeArgs {
    const float *x;
    const int32_t *ids;
    const float *w;
    float *y;
    const ExpertDesc *table;
    int n_experts, S, K, H, F;
    int cpr_gu, cpr_d;       // 16-byte chunks per gate/up row (H inputs) and per down row (F inputs)
    float *hbuf;             // [S*K][F] scratch
    unsigned *bar;           // grid barrier words [2]
    int *err;                // device error word
    int sb;                  // slots per phase-B shared-memory batch
    int rpc;                 // phase-B output rows per CTA
    long long timeout_ns;    // bound of the grid-wide wait
};

// Arguments of the tiled CUDA-core GEMM (prefill / S > 8).
struct GemmArgs {
    const ExpertDesc *table;  // expert table (NULL: use `single`)
    MatDesc single;
    int mi;                   // matrix index in the expert (0 gate, 1 up, 2 down); DUAL uses mi and mi+1
    int fmt, O, I;
    const float *X;           // activations, rows of ldx floats
    long long ldx;
    const int32_t *order;     // p -> slot (s*K+k); source row = order[p] / kdiv.  NULL: source row = p
    int kdiv;
    const int32_t *tile_e, *tile_p0, *tile_p1, *n_tiles;   // NULL: tiles of BP rows over [0, P)
    int P;
    float *out;               // out[p][o], rows of ldo floats
    long long ldo;
};

// Arguments of the routing inversion.
struct RouteArgs {
    const int32_t *ids;
    int S, K, E;
    int32_t *offsets;         // [E+1]
    int32_t *order;           // [S*K]
    int32_t *inv;             // [S*K] slot -> position or -1 (may be NULL)
    int32_t *tile_e, *tile_p0, *tile_p1, *n_tiles;   // may be NULL
    int tile_rows;
    // experts with at most small_rows rows (0: none) go to the small-row list
    // instead, in groups of up to 4 consecutive rows (moe_small.cu)
    int small_rows;
    int32_t *sg_e, *sg_p0, *sg_n, *n_sg;
    uint8_t *row_small;       // [S*K]: 1 for the rows of such experts (may be NULL)
    int *err;
};

// Arguments of the tensor-core grouped GEMM (gemm_tc.cu).
struct TcArgs {
    const ExpertDesc *table;  // expert table (NULL: use `single`)
    MatDesc single;
    int mi;                   // matrix index in the expert
    int dual_mb;              // > 0: m-blocks >= dual_mb belong to matrix mi+1, written at column offset O
    int fmt, O, I;
    int nkb, gkb;             // K-blocks of 64 inputs; K-blocks per scale group
    int n_mblk;               // m-blocks (of 128 rows) in the launch
    const int32_t *tile_e, *tile_p0, *tile_p1, *n_tiles;   // NULL: tiles of 64 rows over [0, P)
    int P;
    int rows_alloc;           // rows per activation plane
    const int *nterm_flag;    // device: non-zero when the mid/lo planes are needed
    float *out;
    long long ldo;
    int *err;
    long long timeout_ns;
};

bool tc_supported_fmt(int fmt, int gs);
int tc_block_rows();
cudaError_t encode_codes_map(const uint8_t *q, long long rs, long long O, void *out128);
// TMA maps of the activation planes (see encode_plane_maps); CUtensorMap blobs
struct PlaneMapSet {
    CUtensorMap m[6];
};
cudaError_t encode_plane_maps(const void *planes, long long I_pad, long long rows_alloc, PlaneMapSet *out);
cudaError_t launch_gather_planes(const float *X, long long ldx, const int32_t *order, int kdiv, const int32_t *n_valid,
                                 int n_rows, int I, int I_pad, void *planes, long long plane_elems, int *flag,
                                 cudaStream_t st, const uint8_t *skip = nullptr);
cudaError_t launch_silu_planes(const float *gu, int F, const int32_t *n_valid, int n_rows, int F_pad, void *planes,
                               long long plane_elems, int *flag, cudaStream_t st,
                               const uint8_t *skip = nullptr);
cudaError_t launch_gemm_tc(const TcArgs &a, const PlaneMapSet &maps, int max_tiles, int n_sm, cudaStream_t st);

cudaError_t launch_moe_decode(const MoeDecodeArgs &a, int fmt, int grid, size_t smem, cudaStream_t st);
cudaError_t moe_decode_occupancy(int fmt, size_t smem, int *per_sm);
cudaError_t launch_route(const RouteArgs &a, cudaStream_t st);
cudaError_t launch_gemm_cc(const GemmArgs &a, bool dual, int max_tiles, cudaStream_t st);
cudaError_t launch_combine(const float *slot_out, const int32_t *inv, const float *w, int S, int K, int H,
                           float *y, cudaStream_t st);
cudaError_t launch_fmt1_encode(uint8_t *q, long long n, cudaStream_t st);
size_t gemv_smem_bytes(int fmt, int cpr, int S, int I, bool generic);

// Streamed decode expert block, S = 1, int4 (fmt 2/4) and int8 (fmt 1) tables
// (stream_decode.cu): weights arrive in shared memory by bulk copies, the
// activations live in registers as dp4a limbs.  sd_plan fills the geometry.
struct SdArgs {
    const float *x;
    const int32_t *ids;
    const float *w;
    float *y;
    const ExpertDesc *table;
    int n_experts, K, H, F;
    int fmt;
    int nc;                    // consumer warps (the producer is one more)
    int n_groups, group_warps; // consumer groups (stage k goes to group k mod n_groups) and warps per group
    int nsA, nsB;              // 512-byte slabs per gate/up row and per down row
    int cpr_gu, cpr_d;         // 16-byte chunks per gate/up row and per down row
    int rs_gu, rs_d;           // device row strides (bytes)
    int ng_gu, ng_d;           // scales per row (1 for per-row formats)
    int gshift_gu, gshift_d;   // chunk -> group index shift (grouped formats)
    int grouped;               // 1: per-group scales copied with the rows; 0: one scale per row
    int RP, RB;                // gate/up pairs per phase-A stage, down rows per expert and phase-B stage
    int stage_bytes, n_stages;
    int off_redA, off_redB, off_desc, off_bar;   // dynamic shared-memory layout (bytes)
    float *hbuf;               // [K][F] scratch: h
    unsigned *ctr;             // zeroed counters: unused, CTAs out, barrier arrivals
    int *err;                  // device error word
    long long timeout_ns;      // bound of every wait
};
bool sd_plan(int fmt, int H, int F, int K, int cpr_gu, int cpr_d, int rs_gu, int rs_d, int ng_gu, int ng_d,
             int n_sm, size_t smem_max, SdArgs *a, size_t *smem);
cudaError_t sd_occupancy(const SdArgs &a, size_t smem, int *per_sm);
size_t sd_scratch_bytes(const SdArgs &a);
size_t sd_counter_words(const SdArgs &a);
cudaError_t launch_stream_decode(const SdArgs &a, int grid, size_t smem, cudaStream_t st);

// Decode expert block, S = 1, int4 tables on the tensor cores (decode_mma.cu):
// weights streamed into shared memory by bulk copies, decoded to f16
// subnormals, mma.sync against hi/lo f16 activations.  md_plan fills the
// geometry.
struct MdArgs {
    const float *x;
    const int32_t *ids;
    const float *w;
    float *y;
    const ExpertDesc *table;
    int n_experts, K, H, F;
    int fmt;
    int rs_gu, rs_d;           // device row strides (bytes)
    int ng_gu, ng_d;           // scales per row (fmt 4)
    int gsh_gu, gsh_d;         // segment -> scale group shift: log2(gs / 64)
    int nsegA, nsegB;          // 64-input segments per gate/up row and per down row
    int spwA, spwB;            // segments per consumer warp
    int bsA, ssA, soA;         // phase-A stage: code-block stride, scale-block stride, scale offset (bytes)
    int bsB, ssB, soB;         // phase-B stage
    int slot_bytes;
    int off_red, off_bar;      // dynamic shared-memory layout (bytes)
    unsigned *ctr;             // kernel state, zero before the first call (md_counter_words)
    int m0[65];                // [routed experts <= 64]: CTAs of the expert finished last in the down phase
    int *err;                  // device error word
    long long timeout_ns;      // bound of every wait
};
// Streamed S = 1 int4 matvec on the tensor cores (gemv_mma.cu).
struct GmArgs {
    const uint8_t *q[GemvJob::MAXM];
    const float *s[GemvJob::MAXM];
    float *y[GemvJob::MAXM];
    int O[GemvJob::MAXM];
    int stage_start[GemvJob::MAXM + 1];   // prefix of the matrices' stage counts
    int n, fmt, S, I, rs, ng, gsh;         // S rows of x (1..4); rs: device row stride (bytes); gsh: log2(gs / 64)
    int nseg, spw, nt;                     // 64-input segments per row and per warp; 16-row tiles per stage
    int bs, so, ss, slot_bytes;            // stage layout: code-block stride, scale offset and block stride
    int off_red, off_bar;                  // dynamic shared-memory layout (bytes)
    const float *x;
    unsigned *ctr;                         // [0] next claimed stage, [1] CTAs out: zero between calls
    int *err;
    long long timeout_ns;
};
size_t gm_counter_words();
bool gm_plan(int fmt, int gs, int I, int rs, int ng, int n, const int *O, int S, int n_sm, size_t smem_max,
             GmArgs *a, size_t *smem, int *grid);
cudaError_t launch_gemv_mma(const GmArgs &a, int grid, size_t smem, cudaStream_t st);

// Prefill products of the experts with few rows (moe_small.cu).
struct SmArgs {
    const ExpertDesc *table;
    const int32_t *sg_e, *sg_p0, *sg_n, *n_sg;   // groups of up to 4 rows (routing kernel)
    const float *x;                              // gate|up: activations, row stride ldx, token of row p = order[p] / K
    long long ldx;
    const int32_t *order;
    int K;
    const float *gu;                             // down: the gate|up results [rows][2 I]
    float *out;                                  // gate|up: gu [rows][2 O]; down: slot outputs [rows][O]
    long long ldo;
    int down, fmt, I, O, rs, ng, gsh;
    int nseg, spw, nt, n_mat, nb;                // segments per row / warp, tiles per stage, matrices, row blocks
    int bs, so, ss, slot_bytes, off_red, off_stg, off_bar;
    int *err;
    long long timeout_ns;
};
bool sm_plan(bool down, int fmt, int gs, int I, int O, int rs, int ng, size_t smem_max, SmArgs *a, size_t *smem);
cudaError_t launch_moe_small(const SmArgs &a, int grid, size_t smem, cudaStream_t st);

bool md_plan(int fmt, int H, int F, int K, int rs_gu, int rs_d, int ng_gu, int ng_d, int gs_gu, int gs_d, int n_sm,
             size_t smem_max, MdArgs *a, size_t *smem);
cudaError_t md_occupancy(const MdArgs &a, size_t smem, int *per_sm);
size_t md_counter_words(const MdArgs &a);
cudaError_t launch_decode_mma(const MdArgs &a, int grid, size_t smem, cudaStream_t st);

// Streamed S = 1 matvec (slab.cu): the same bulk-copy ring over the rows of all
// matrices of the call.
constexpr size_t kBarrierBytes = 256;           // per-workspace grid-barrier words (see workspace())
constexpr int kStreamStageBytes = 27 * 1024;
constexpr int kStreamStages = 5;
constexpr int kStreamRedBytes = 12 * 1024;
constexpr int kStreamConsumerWarps = 12;
size_t stream_gemv_smem();
constexpr int kStreamGemvRedBytes = 64 * 1024;   // partial sums of the S = 2..4 streamed matvec
size_t stream_gemv_s_smem();
cudaError_t launch_stream_gemv_s(const GemvJob &job, int rpc, int RG, int gshift, int grid, cudaStream_t st);
cudaError_t launch_stream_gemv(const GemvJob &job, int rpc, int RG, int gshift, int grid, cudaStream_t st);
int stream_lane_bytes(int fmt);
int stream_lane_inputs(int fmt);

// kv_b absorption products (absorb.cu)
size_t absorb_smem(int fmt, bool transposed, int units, int n_rows, int S);
cudaError_t launch_absorb(const MatDesc &m, int fmt, int I, int units, long long o0, long long stride, int n_rows,
                          int n_heads, int S, const float *x, float *y, bool transposed, cudaStream_t st,
                          int *n_launch);

size_t topk_smem(int E);
cudaError_t launch_topk(const float *logits, const float *bias, int S, int E, int K, float top_p, int norm_topk,
                        float routed_scale, int32_t *ids, float *w, cudaStream_t st);

bool slab_supported(int fmt, int gs);
size_t slab_gemv_smem(const GemvJob &job, int n_sm);
cudaError_t launch_slab_gemv(const GemvJob &job, int n_sm, cudaStream_t st);
size_t slab_decode_smem(int fmt, int cpr_gu, int cpr_d, int F, int n_slots, int grid_min, int H, int sb);
cudaError_t slab_decode_occupancy(int fmt, size_t smem, int *per_sm);
cudaError_t launch_slab_decode(const MoeDecodeArgs &a, int fmt, int grid, size_t smem, int gs_gu, int gs_d,
                               cudaStream_t st);

// Record `msg` as the calling thread's last error (coli_last_error) and return code.
int set_last_error(int code, const char *msg);
// Clear the calling thread's last error message (an entry point's first step).
void clear_last_error();
// The host-side fault-injection gate of compute calls (coli_set_fail_after):
// COLI_EINJECTED once the counter has run out, else COLI_OK.
int injected_gate();
// Count one compute call with its launches and weight bytes (coli_get_stats).
void count_call(int launches, uint64_t weight_bytes);
// Copy n expert descriptors, passed by value in kernel parameters, to the
// device table dst (stream-ordered, no host memory involved).
cudaError_t launch_table_fill(ExpertDesc *dst, const ExpertDesc *src, int n, cudaStream_t st);

constexpr int kDecodeThreads = 256;
constexpr int kMaxDecodeSlots = 64;

constexpr int kGemmBP = 32;    // token rows per GEMM tile

}  // namespace coli
