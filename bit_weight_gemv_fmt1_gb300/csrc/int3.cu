// int3.cu -- the S <= 8 matvec y = W x for int3 weights (fmt=5), on the CUDA
// cores, for coli_matmul and coli_matmul_multi.
//
// Layout (the pages name fmt=5 as int3 with scales that vary along the row,
// like fmt=4's -- PR #298 page, the #377 retarget list and the Vulkan fmt=4
// commit message -- but print no bit layout; the library documents the
// reading it uses): element 8j+t of a row is bits [3t, 3t+2] of the
// little-endian 24-bit word in bytes 3j..3j+2, the value is code - 4, times
// the f32 scale of group i/gs (gs a multiple of 8, O*ceil(I/gs) scales).
//
// One warp per row.  A lane takes units of 12 bytes -- four 3-byte groups,
// 32 consecutive inputs -- as three aligned 32-bit words (device rows are
// padded to 16 bytes, so a word that holds any byte of the row lies inside
// it), units u = lane, lane + 32, ... of the row.  Code j of a unit is bits
// [3j, 3j+2] of the unit's 96-bit little-endian value; OR-ing it into the
// mantissa of 2^23 and subtracting 2^23 + 4 gives code - 4 exactly.  Each
// 8-input group of codes is dotted with the S activation rows in f32 and
// multiplied by its scale (gs is a multiple of 8, so a group of codes never
// straddles two scales); the lanes' sums are combined with shuffles.
#include <algorithm>

#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int kI3Warps = 8;

template <int S, bool VEC>
__global__ void __launch_bounds__(kI3Warps * 32) gemv_i3_kernel(const GemvJob job) {
    const int lane = threadIdx.x & 31;
    const int warp_g = blockIdx.x * kI3Warps + (threadIdx.x >> 5), n_warps = gridDim.x * kI3Warps;
    const int I = job.I, total = job.row_start[job.n];
    const int units = (I + 31) / 32;
    const int hb = 3 * ((I + 7) / 8);   // bytes of a row that hold codes
    pdl_wait();
    int m = 0;
    for (int r = warp_g; r < total; r += n_warps) {
        while (r >= job.row_start[m + 1]) m++;
        const int o = r - job.row_start[m];
        const uint8_t *row = job.q[m] + (size_t)o * (size_t)job.rs[m];
        const float *srow = job.s[m] + (size_t)o * (size_t)job.ng[m];
        const int gs = job.gs[m];
        float acc[S];
#pragma unroll
        for (int s = 0; s < S; s++) acc[s] = 0.f;
        for (int u = lane; u < units; u += 32) {
            const int b0 = 12 * u;
            uint32_t w[3];
#pragma unroll
            for (int k = 0; k < 3; k++)
                w[k] = b0 + 4 * k < hb ? __ldg(reinterpret_cast<const uint32_t *>(row + b0 + 4 * k)) : 0u;
            const int i0 = 32 * u;
#pragma unroll
            for (int t = 0; t < 4; t++) {   // the unit's four 8-input groups of codes
                float v[8];
#pragma unroll
                for (int jj = 0; jj < 8; jj++) {
                    constexpr uint32_t kOne = 0x4B000000u;   // 2^23
                    const int bit = 3 * (8 * t + jj), k = bit >> 5, sh = bit & 31;
                    const uint32_t c =
                        sh <= 29 ? (w[k] >> sh) & 7u : __funnelshift_r(w[k], w[k < 2 ? k + 1 : 2], sh) & 7u;
                    v[jj] = __uint_as_float(kOne | c) - 8388612.0f;
                }
                const int ig = i0 + 8 * t;
                if (ig >= I) break;
                const float sc = __ldg(srow + ig / gs);
#pragma unroll
                for (int s = 0; s < S; s++) {
                    const float *xs = job.x + (size_t)s * I + ig;
                    float xv[8];
                    if (VEC && ig + 8 <= I) {
                        const float4 f0 = __ldg(reinterpret_cast<const float4 *>(xs));
                        const float4 f1 = __ldg(reinterpret_cast<const float4 *>(xs) + 1);
                        xv[0] = f0.x; xv[1] = f0.y; xv[2] = f0.z; xv[3] = f0.w;
                        xv[4] = f1.x; xv[5] = f1.y; xv[6] = f1.z; xv[7] = f1.w;
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 8; jj++) xv[jj] = ig + jj < I ? __ldg(xs + jj) : 0.f;
                    }
                    float part = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) part = fmaf(v[jj], xv[jj], part);
                    acc[s] = fmaf(part, sc, acc[s]);
                }
            }
        }
#pragma unroll
        for (int s = 0; s < S; s++) {
            float a = acc[s];
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) a += __shfl_xor_sync(0xffffffffu, a, d);
            if (lane == 0) job.y[m][(size_t)s * job.O[m] + o] = a;
        }
    }
    pdl_trigger();
}

template <int S>
cudaError_t launch_s(const GemvJob &job, bool vec, int grid, cudaStream_t st) {
    return vec ? launch_pdl(gemv_i3_kernel<S, true>, dim3(grid), dim3(kI3Warps * 32), 0, st, job)
               : launch_pdl(gemv_i3_kernel<S, false>, dim3(grid), dim3(kI3Warps * 32), 0, st, job);
}

}  // namespace

cudaError_t launch_gemv_i3(const GemvJob &job, int n_sm, cudaStream_t st) {
    const int total = job.row_start[job.n];
    const int grid = std::max(1, std::min((total + kI3Warps - 1) / kI3Warps, 8 * n_sm));
    // whole float4 loads of x need 16-byte rows: x 16-byte aligned and I a multiple of 4
    const bool vec = ((uintptr_t)job.x & 15) == 0 && job.I % 4 == 0;
    switch (job.S) {
    case 1: return launch_s<1>(job, vec, grid, st);
    case 2: return launch_s<2>(job, vec, grid, st);
    case 3: return launch_s<3>(job, vec, grid, st);
    case 4: return launch_s<4>(job, vec, grid, st);
    case 5: return launch_s<5>(job, vec, grid, st);
    case 6: return launch_s<6>(job, vec, grid, st);
    case 7: return launch_s<7>(job, vec, grid, st);
    case 8: return launch_s<8>(job, vec, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace coli
