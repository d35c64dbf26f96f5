// absorb.cu -- the two quantized products of the kv_b MLA-absorption path
// (PR #298 page, commit message on qt_addrow / qt_matvec_rows: a matvec over
// a range of rows, and coefficient-times-row accumulation, of one quantized
// matrix), batched over attention heads.  Head h owns rows o0 + h*stride + j,
// j < n_rows:
//   forward     y[s][h][j] = sum_i W[o0 + h*stride + j][i] * x[s][h][i]
//   transposed  y[s][h][i] = sum_j x[s][h][j] * W[o0 + h*stride + j][i]
//
// Both kernels read the device layout in 8-byte units (2 f32, 8 int8/FP8, 16
// int4, 32 int2 values), decode them exactly and accumulate in f32.  The
// forward kernel gives each warp eight head rows at once (lanes over the rows'
// units, the head's activations staged in shared memory, shuffle reductions);
// the transposed kernel gives each lane one unit column of the head and a
// slice of its rows, sixteen rows' loads in flight at a time, keeps the
// coefficients in shared memory and reduces the row slices through shared
// memory.  Weight loads that need nothing from the previous kernel are issued
// before the dependency wait.  Rows are read exactly once per call for S <= 4.
#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int kAbsorbThreads = 256;

template <int FMT> struct Unit;   // elements per 8-byte unit
template <> struct Unit<0> { static constexpr int N = 2; };
template <> struct Unit<1> { static constexpr int N = 8; };
template <> struct Unit<2> { static constexpr int N = 16; };
template <> struct Unit<3> { static constexpr int N = 32; };
template <> struct Unit<4> { static constexpr int N = 16; };
template <> struct Unit<7> { static constexpr int N = 8; };

// Exact values of the unit's elements, scale not applied: code - offset for
// the integer formats (int8 is stored offset binary), the f32 / E4M3 value
// otherwise.  Element e of the unit is input e0 + e.  An integer code c is
// OR-ed into the mantissa of 2^23, giving 2^23 + c exactly, and one subtract
// of 2^23 + offset leaves c - offset exactly (no integer-to-float conversion,
// which runs on a slow pipe).
__device__ __forceinline__ float mag23(uint32_t c) { return __uint_as_float(0x4B000000u | c); }

template <int FMT>
__device__ __forceinline__ void decode_unit(uint2 u, float (&v)[Unit<FMT>::N]) {
    const uint32_t w[2] = {u.x, u.y};
    if constexpr (FMT == 0) {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
    } else if constexpr (FMT == 1) {
#pragma unroll
        for (int k = 0; k < 8; k++) v[k] = mag23((w[k >> 2] >> (8 * (k & 3))) & 0xFFu) - 8388736.0f;   // 2^23 + 128
    } else if constexpr (FMT == 2 || FMT == 4) {
#pragma unroll
        for (int k = 0; k < 16; k++) v[k] = mag23((w[k >> 3] >> (4 * (k & 7))) & 0xFu) - 8388616.0f;   // 2^23 + 8
    } else if constexpr (FMT == 3) {
#pragma unroll
        for (int k = 0; k < 32; k++) v[k] = mag23((w[k >> 4] >> (2 * (k & 15))) & 0x3u) - 8388610.0f;   // 2^23 + 2
    } else {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float2 p = e4m3x2_to_f32x2((w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu);
            v[2 * k] = p.x;
            v[2 * k + 1] = p.y;
        }
    }
}

// Scale of element (row, i) given the row's scales (row_scales); one lookup per
// element, hoisted by the callers where the unit shares one scale.
template <int FMT>
__device__ __forceinline__ float elem_scale(const float *rsc, int gs, int i) {
    if constexpr (FMT == 0) return 1.0f;
    else if constexpr (FMT == 4) return __ldg(rsc + i / gs);
    else if constexpr (FMT == 7) return __ldg(rsc + i / kFp8Block);
    else return __ldg(rsc);
}

struct AbsorbArgs {
    MatDesc m;
    int I;                // inputs per row
    int units;            // 8-byte units holding a row's I inputs
    long long o0, stride;
    int n_rows, n_heads, S;
    const float *x;
    float *y;
};

// Forward: grid (n_heads, row blocks of RU * warps rows); warp w handles rows
// jb + w + r * nw, r < RU, of its head together (RU loads in flight per lane);
// the first units of those rows are requested before the activations, which
// may come from the previous kernel, are staged.  S_T rows of activations at once.
// PS: fmt=4 with a group size that splits a unit (each element looks its scale
// up); otherwise one scale per unit.  Kept apart so the common loop stays small
// (the per-element variant unrolled into it overflowed the instruction cache).
template <int FMT, int S_T, bool PS>
__global__ void __launch_bounds__(kAbsorbThreads) absorb_fwd_kernel(const AbsorbArgs a, int s0) {
    extern __shared__ float xs[];   // [S_T][units * N]
    constexpr int N = Unit<FMT>::N, RU = 8;
    const int h = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int xlen = a.units * N;
    const int jb = blockIdx.y * nw * RU + warp;
    const uint2 *rp[RU];
    const float *rsc[RU];
    bool rok[RU];
    uint2 q[RU];
    float sq[RU];   // scale of the unit's first input, requested with its codes
#pragma unroll
    for (int r = 0; r < RU; r++) {
        const int j = jb + r * nw;
        rok[r] = j < a.n_rows;
        const long long row = a.o0 + (long long)h * a.stride + (rok[r] ? j : 0);
        rp[r] = reinterpret_cast<const uint2 *>(a.m.q + (size_t)row * a.m.rs);
        rsc[r] = row_scales(FMT, a.m, (int)row);
        const bool ok = rok[r] && lane < a.units;
        q[r] = ok ? __ldg(rp[r] + lane) : make_uint2(0u, 0u);
        sq[r] = ok ? elem_scale<FMT>(rsc[r], a.m.gs, min(lane * N, a.I - 1)) : 0.f;
    }
    pdl_wait();
    for (int e = threadIdx.x; e < S_T * xlen; e += blockDim.x) {
        const int s = e / xlen, i = e - s * xlen;
        xs[e] = (i < a.I) ? a.x[((size_t)(s0 + s) * a.n_heads + h) * a.I + i] : 0.f;
    }
    __syncthreads();
    float acc[RU][S_T];
#pragma unroll
    for (int r = 0; r < RU; r++)
#pragma unroll
        for (int s = 0; s < S_T; s++) acc[r][s] = 0.f;
    for (int u = lane; u < a.units; u += 32) {
        const int i0 = u * N;
        if (u != lane) {
#pragma unroll
            for (int r = 0; r < RU; r++) {
                q[r] = rok[r] ? __ldg(rp[r] + u) : make_uint2(0u, 0u);
                sq[r] = rok[r] ? elem_scale<FMT>(rsc[r], a.m.gs, min(i0, a.I - 1)) : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < RU; r++) {
            float v[N];
            decode_unit<FMT>(q[r], v);
            const float sc0 = sq[r];
#pragma unroll
            for (int k = 0; k < N; k++) {
                float wv;
                if constexpr (PS) wv = v[k] * elem_scale<FMT>(rsc[r], a.m.gs, min(i0 + k, a.I - 1));
                else wv = v[k] * sc0;
#pragma unroll
                for (int s = 0; s < S_T; s++) acc[r][s] = fmaf(wv, xs[s * xlen + i0 + k], acc[r][s]);
            }
        }
    }
    pdl_trigger();
#pragma unroll
    for (int r = 0; r < RU; r++)
#pragma unroll
        for (int s = 0; s < S_T; s++) {
            const float t = warp_sum(acc[r][s]);
            if (lane == 0 && rok[r]) a.y[((size_t)(s0 + s) * a.n_heads + h) * a.n_rows + jb + r * nw] = t;
        }
}

// Transposed: grid (n_heads, unit-column blocks of 32); thread (p, c) with
// c = lane owns unit column u = 32 * blockIdx.y + c and rows j = p + P * t
// (P = warps), requested RT at a time; S_T coefficient rows at once; the P
// partial sums meet in shared memory.  The first batch of rows is requested
// before the coefficients, which may come from the previous kernel, are staged.
template <int FMT, int S_T, bool PS>
__global__ void __launch_bounds__(kAbsorbThreads) absorb_t_kernel(const AbsorbArgs a, int s0) {
    extern __shared__ float sm[];   // coef [S_T][n_rows], then partials [P][S_T][N][32]
    constexpr int N = Unit<FMT>::N, RT = 16;
    const int h = blockIdx.x;
    const int lane = threadIdx.x & 31, p = threadIdx.x >> 5, P = blockDim.x >> 5;
    float *coef = sm;
    float *part = sm + S_T * a.n_rows;
    const int u = blockIdx.y * 32 + lane;
    const bool live = u < a.units;
    const int i0 = u * N;
    // codes and the scale of the unit's first input, RT rows at a time
    auto load_batch = [&](int j0, uint2 (&q)[RT], float (&sq)[RT]) {
#pragma unroll
        for (int t = 0; t < RT; t++) {
            const int j = j0 + t * P;
            const bool ok = live && j < a.n_rows;
            const long long row = a.o0 + (long long)h * a.stride + (ok ? j : 0);
            q[t] = ok ? __ldg(reinterpret_cast<const uint2 *>(a.m.q + (size_t)row * a.m.rs) + u) : make_uint2(0u, 0u);
            sq[t] = ok ? elem_scale<FMT>(row_scales(FMT, a.m, (int)row), a.m.gs, min(i0, a.I - 1)) : 0.f;
        }
    };
    uint2 q[RT];
    float sq[RT];
    load_batch(p, q, sq);
    pdl_wait();
    for (int e = threadIdx.x; e < S_T * a.n_rows; e += blockDim.x) {
        const int s = e / a.n_rows, j = e - s * a.n_rows;
        coef[e] = a.x[((size_t)(s0 + s) * a.n_heads + h) * a.n_rows + j];
    }
    __syncthreads();
    float acc[S_T][N];
#pragma unroll
    for (int s = 0; s < S_T; s++)
#pragma unroll
        for (int k = 0; k < N; k++) acc[s][k] = 0.f;
    for (int j0 = p; j0 < a.n_rows; j0 += P * RT) {
        if (j0 != p) load_batch(j0, q, sq);
#pragma unroll
        for (int t = 0; t < RT; t++) {
            const int j = j0 + t * P;
            if (!live || j >= a.n_rows) break;
            const long long row = a.o0 + (long long)h * a.stride + j;
            const float *rsc = row_scales(FMT, a.m, (int)row);
            float v[N];
            decode_unit<FMT>(q[t], v);
            const float sc0 = sq[t];
#pragma unroll
            for (int k = 0; k < N; k++) {
                float wv;
                if constexpr (PS) wv = v[k] * elem_scale<FMT>(rsc, a.m.gs, min(i0 + k, a.I - 1));
                else wv = v[k] * sc0;
#pragma unroll
                for (int s = 0; s < S_T; s++) acc[s][k] = fmaf(coef[s * a.n_rows + j], wv, acc[s][k]);
            }
        }
    }
    // partial sums of the P row slices -> shared memory, then one thread per output
#pragma unroll
    for (int s = 0; s < S_T; s++)
#pragma unroll
        for (int k = 0; k < N; k++) part[(((size_t)p * S_T + s) * N + k) * 32 + lane] = acc[s][k];
    __syncthreads();
    pdl_trigger();
    for (int e = threadIdx.x; e < S_T * 32 * N; e += blockDim.x) {
        const int s = e / (32 * N), c = e - s * (32 * N);
        const int i = blockIdx.y * 32 * N + c;
        if (i >= a.I) continue;
        const int cl = c / N, ck = c - cl * N;   // column c of the block = element ck of lane cl's unit
        float t = 0.f;
        for (int qq = 0; qq < P; qq++) t += part[(((size_t)qq * S_T + s) * N + ck) * 32 + cl];
        a.y[((size_t)(s0 + s) * a.n_heads + h) * a.I + i] = t;
    }
}

template <int FMT, int S_T, bool PS>
cudaError_t launch_one(const AbsorbArgs &a, bool transposed, int s0, cudaStream_t st) {
    constexpr int N = Unit<FMT>::N;
    if (!transposed) {
        const size_t smem = (size_t)S_T * a.units * N * sizeof(float);
        auto kern = absorb_fwd_kernel<FMT, S_T, PS>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int rows_per_cta = (kAbsorbThreads / 32) * 8;   // RU rows per warp
        const dim3 grid(a.n_heads, (a.n_rows + rows_per_cta - 1) / rows_per_cta);
        return launch_pdl(kern, grid, dim3(kAbsorbThreads), smem, st, a, s0);
    }
    const size_t smem = ((size_t)S_T * a.n_rows + (size_t)(kAbsorbThreads / 32) * S_T * 32 * N) * sizeof(float);
    auto kern = absorb_t_kernel<FMT, S_T, PS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.n_heads, (a.units + 31) / 32);
    return launch_pdl(kern, grid, dim3(kAbsorbThreads), smem, st, a, s0);
}

// Rows of activations per launch: all S up to 4 (every weight row read once),
// chunks of 4 beyond; the wide int2 unit takes 2 (its accumulators are 32 wide).
template <int FMT, bool PS>
cudaError_t launch_fmt(const AbsorbArgs &a, bool transposed, cudaStream_t st, int *n_launch) {
    const int cap = (FMT == 3 && transposed) ? 2 : 4;
    *n_launch = 0;
    for (int s0 = 0; s0 < a.S; s0 += cap) {
        const int n = a.S - s0 < cap ? a.S - s0 : cap;
        cudaError_t e;
        switch (n) {
        case 1: e = launch_one<FMT, 1, PS>(a, transposed, s0, st); break;
        case 2: e = launch_one<FMT, 2, PS>(a, transposed, s0, st); break;
        case 3: e = launch_one<FMT, 3, PS>(a, transposed, s0, st); break;
        default: e = launch_one<FMT, 4, PS>(a, transposed, s0, st); break;
        }
        if (e != cudaSuccess) return e;
        ++*n_launch;
    }
    return cudaSuccess;
}

}  // namespace

size_t absorb_smem(int fmt, bool transposed, int units, int n_rows, int S) {
    const int N = fmt == 0 ? 2 : (fmt == 1 || fmt == 7) ? 8 : fmt == 3 ? 32 : 16;
    const int cap = (fmt == 3 && transposed) ? 2 : 4;
    const int s_t = S < cap ? S : cap;
    if (!transposed) return (size_t)s_t * units * N * sizeof(float);
    return ((size_t)s_t * n_rows + (size_t)(kAbsorbThreads / 32) * s_t * 32 * N) * sizeof(float);
}

cudaError_t launch_absorb(const MatDesc &m, int fmt, int I, int units, long long o0, long long stride, int n_rows,
                          int n_heads, int S, const float *x, float *y, bool transposed, cudaStream_t st,
                          int *n_launch) {
    AbsorbArgs a;
    a.m = m;
    a.I = I;
    a.units = units;
    a.o0 = o0;
    a.stride = stride;
    a.n_rows = n_rows;
    a.n_heads = n_heads;
    a.S = S;
    a.x = x;
    a.y = y;
    switch (fmt) {
    case 0: return launch_fmt<0, false>(a, transposed, st, n_launch);
    case 1: return launch_fmt<1, false>(a, transposed, st, n_launch);
    case 2: return launch_fmt<2, false>(a, transposed, st, n_launch);
    case 3: return launch_fmt<3, false>(a, transposed, st, n_launch);
    case 4:
        // a group size that is a multiple of the 16-element unit gives one scale per unit
        return m.gs % Unit<4>::N == 0 ? launch_fmt<4, false>(a, transposed, st, n_launch)
                                      : launch_fmt<4, true>(a, transposed, st, n_launch);
    case 7: return launch_fmt<7, false>(a, transposed, st, n_launch);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace coli
