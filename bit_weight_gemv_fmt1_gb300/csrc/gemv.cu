// gemv.cu -- bandwidth-bound quantized matvec / small-S matmul (S <= 8).
//
// y_m[s][o] = sum_i W_m[o][i] x[s][i] for one or several matrices W_m sharing
// the activations x (PR #298 page, "metal: grouped-int4 (fmt=4) GEMV support"
// commit message, Shader paragraph: per-row scale after the dot product for
// fmt 1-3, the group scale folded in per group for fmt=4; fmt=7 folds in the
// scale of each 128 x 128 block the same way).
//
// One CTA stages x (all S rows) in shared memory once, then its warps stream
// weight rows: a warp task is R consecutive rows of one matrix, each lane
// loading 16-byte chunks l, l+32, ... of those rows (coalesced 512-byte warp
// loads) with U chunks per row in flight, decoding them in registers and
// accumulating against the staged x; a warp-shuffle reduction finishes each
// output.  Weights are read exactly once per call.
#include <atomic>

#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int kThreads = 256;

template <int FMT, int S, int R>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvJob job) {
    extern __shared__ float4 smem4[];
    float *xs = reinterpret_cast<float *>(smem4);
    const int xlen = staged_len(FMT, job.cpr);
    pdl_wait();
#pragma unroll
    for (int s = 0; s < S; s++)
        stage_vec<FMT>(xs + s * xlen, job.x + (size_t)s * job.I, job.I, xlen, threadIdx.x, blockDim.x);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int gw = blockIdx.x * nwarps + (threadIdx.x >> 5);
    const int gstride = gridDim.x * nwarps;

    // task t -> (matrix m, first row): tasks are numbered matrix by matrix
    int task_start[GemvJob::MAXM + 1];
    task_start[0] = 0;
    for (int m = 0; m < job.n; m++) task_start[m + 1] = task_start[m] + (job.O[m] + R - 1) / R;
    const int n_tasks = task_start[job.n];

    const float *xsv[S];
#pragma unroll
    for (int s = 0; s < S; s++) xsv[s] = xs + s * xlen;

    for (int t = gw; t < n_tasks; t += gstride) {
        int m = 0;
        while (t >= task_start[m + 1]) m++;
        const int o0 = (t - task_start[m]) * R;
        const int Om = job.O[m];
        const uint8_t *rows[R];
        const float *scl[R];
        int gpc[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const int o = min(o0 + r, Om - 1);
            rows[r] = job.q[m] + (size_t)o * job.rs[m];
            scl[r] = FMT == 4   ? job.s[m] + (size_t)o * job.ng[m]
                     : FMT == 7 ? job.s[m] + (size_t)(o / kFp8Block) * job.ng[m]
                     : FMT == 0 ? nullptr
                                : job.s[m] + o;
            gpc[r] = chunks_per_group(FMT, job.gs[m]);
        }
        float out[R][S];
        dot_rows<FMT, R, S>(rows, scl, gpc, xsv, job.cpr, lane, out);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; r++) {
                if (o0 + r < Om) {
#pragma unroll
                    for (int s = 0; s < S; s++) job.y[m][(size_t)s * Om + o0 + r] = out[r][s];
                }
            }
        }
    }
    pdl_trigger();
}

// fmt=4 with gs not a multiple of 32: one warp per (matrix, row), plain
// layout of x in shared memory, element by element.
__global__ void __launch_bounds__(kThreads) gemv_fmt4_generic_kernel(const GemvJob job) {
    extern __shared__ float4 smem4[];
    float *xs = reinterpret_cast<float *>(smem4);
    pdl_wait();
    for (int e = threadIdx.x; e < job.S * job.I; e += blockDim.x) xs[e] = job.x[e];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int gw = blockIdx.x * nwarps + (threadIdx.x >> 5);
    const int n_rows = job.row_start[job.n];
    for (int t = gw; t < n_rows; t += gridDim.x * nwarps) {
        int m = 0;
        while (t >= job.row_start[m + 1]) m++;
        const int o = t - job.row_start[m];
        const uint8_t *row = job.q[m] + (size_t)o * job.rs[m];
        const float *scl = job.s[m] + (size_t)o * job.ng[m];
        for (int s = 0; s < job.S; s++) {
            const float v = dot_row_fmt4_generic(row, scl, job.gs[m], job.I, xs + (size_t)s * job.I, lane);
            if (lane == 0) job.y[m][(size_t)s * job.O[m] + o] = v;
        }
    }
    pdl_trigger();
}

template <int FMT, int S, int R>
cudaError_t launch_t(const GemvJob &job, cudaStream_t st, int n_sm) {
    const size_t smem = (size_t)S * staged_len(FMT, job.cpr) * sizeof(float);
    auto kern = gemv_kernel<FMT, S, R>;
    // attribute and occupancy per (instantiation, device, shared-memory size), queried once
    static std::atomic<long long> cache[16];   // zero = not queried yet (smem is never 0)
    int dev = 0;
    cudaGetDevice(&dev);
    std::atomic<long long> &cached = cache[dev & 15];
    int per_sm = 0;
    const long long c = dev < 16 ? cached.load(std::memory_order_relaxed) : -1;
    if (c >= 0 && (c >> 8) == (long long)smem) {
        per_sm = (int)(c & 0xFF);
    } else {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        cached.store(((long long)smem << 8) | (per_sm & 0xFF), std::memory_order_relaxed);
    }
    int n_tasks = 0;
    for (int m = 0; m < job.n; m++) n_tasks += (job.O[m] + R - 1) / R;
    const int want = (n_tasks + kThreads / 32 - 1) / (kThreads / 32);
    const int grid = max(1, min(want, per_sm * n_sm));
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, job);
}

template <int FMT, int S>
cudaError_t launch_s(const GemvJob &job, cudaStream_t st, int n_sm) {
    if constexpr (S <= 2) return launch_t<FMT, S, 2>(job, st, n_sm);
    else return launch_t<FMT, S, 1>(job, st, n_sm);
}

template <int FMT>
cudaError_t launch_f(const GemvJob &job, cudaStream_t st, int n_sm) {
    switch (job.S) {
    case 1: return launch_s<FMT, 1>(job, st, n_sm);
    case 2: return launch_s<FMT, 2>(job, st, n_sm);
    case 3: return launch_s<FMT, 3>(job, st, n_sm);
    case 4: return launch_s<FMT, 4>(job, st, n_sm);
    case 5: return launch_s<FMT, 5>(job, st, n_sm);
    case 6: return launch_s<FMT, 6>(job, st, n_sm);
    case 7: return launch_s<FMT, 7>(job, st, n_sm);
    case 8: return launch_s<FMT, 8>(job, st, n_sm);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Shared memory the GEMV needs for this job (host side check before launch).
size_t gemv_smem_bytes(int fmt, int cpr, int S, int I, bool generic) {
    if (generic) return (size_t)S * I * sizeof(float);
    return (size_t)S * staged_len(fmt, cpr) * sizeof(float);
}

cudaError_t launch_gemv(const GemvJob &job, cudaStream_t st, int *n_launch) {
    int dev = 0, n_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    bool generic = false;
    if (job.fmt == 4)
        for (int m = 0; m < job.n; m++) generic |= (job.gs[m] % 32) != 0;
    *n_launch = 1;
    if (generic) {
        const size_t smem = gemv_smem_bytes(4, job.cpr, job.S, job.I, true);
        cudaError_t e = cudaFuncSetAttribute(gemv_fmt4_generic_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int rows = job.row_start[job.n];
        const int grid = max(1, min((rows + 7) / 8, n_sm * 4));
        return launch_pdl(gemv_fmt4_generic_kernel, dim3(grid), dim3(kThreads), smem, st, job);
    }
    switch (job.fmt) {
    case 0: return launch_f<0>(job, st, n_sm);
    case 1: return launch_f<1>(job, st, n_sm);
    case 2: return launch_f<2>(job, st, n_sm);
    case 3: return launch_f<3>(job, st, n_sm);
    case 4: return launch_f<4>(job, st, n_sm);
    case 7: return launch_f<7>(job, st, n_sm);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace coli
