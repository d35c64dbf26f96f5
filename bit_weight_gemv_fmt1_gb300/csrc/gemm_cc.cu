// gemm_cc.cu -- tiled dequantizing GEMM on the CUDA cores.
//
// out[p][o] = sum_i W[o][i] X[src(p)][i] over token tiles: the grouped form
// used by the routed-expert prefill (one tile list entry = one expert and a
// run of at most kGemmBP of its routed rows, from the routing inversion) and
// the plain form used by coli_matmul when S is above the matvec range.  With
// DUAL the tile computes the gate and up products of an expert together and
// stores silu(gate) * up.  Weights are decoded (scale included) into shared
// memory one 64 x 32 block at a time.
#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int BO = 64, BP = kGemmBP, BK = 32, NT = 256;

__device__ __forceinline__ float silu_g(float g) { return g / (1.0f + expf(-g)); }

template <bool DUAL>
__global__ void __launch_bounds__(NT) gemm_cc_kernel(const GemmArgs a) {
    __shared__ float Ws[DUAL ? 2 : 1][BK][BO + 1];
    __shared__ float Xs[BK][BP + 1];
    const int tid = threadIdx.x;
    int e = -1, p0, p1;
    if (a.tile_e) {
        if ((int)blockIdx.y >= *a.n_tiles) return;
        e = a.tile_e[blockIdx.y];
        p0 = a.tile_p0[blockIdx.y];
        p1 = a.tile_p1[blockIdx.y];
    } else {
        p0 = blockIdx.y * BP;
        p1 = min(a.P, p0 + BP);
        if (p0 >= p1) return;
    }
    const MatDesc W0 = a.table ? a.table[e].m[a.mi] : a.single;
    const MatDesc W1 = (DUAL && a.table) ? a.table[e].m[a.mi + 1] : W0;
    const int o_base = blockIdx.x * BO;
    const int oq = tid & 15, pq = tid >> 4;   // outputs oq + 16i, tokens pq + 16j
    float acc[2][4][2] = {};

    // element loader coordinates: 8 consecutive inputs of one row per thread
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    const int lo = o_base + lr;
    // token loader coordinates: 4 inputs of one token per thread
    const int tp = tid >> 3, tk = (tid & 7) * 4;
    const int tok_p = p0 + tp;
    long long src = -1;
    if (tok_p < p1) src = a.order ? (long long)(a.order[tok_p] / a.kdiv) : (long long)tok_p;

    for (int k0 = 0; k0 < a.I; k0 += BK) {
        // decode weights
#pragma unroll
        for (int mtx = 0; mtx < (DUAL ? 2 : 1); mtx++) {
            const MatDesc &M = mtx ? W1 : W0;
            const uint8_t *row = lo < a.O ? M.q + (size_t)lo * M.rs : nullptr;
            const float *rsc = row ? row_scales(a.fmt, M, lo) : nullptr;
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int i = k0 + lk + u;
                Ws[mtx][lk + u][lr] = (row && i < a.I) ? decode_elem(a.fmt, row, rsc, M.gs, i) : 0.f;
            }
        }
        // activations
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int i = k0 + tk + u;
            Xs[tk + u][tp] = (src >= 0 && i < a.I) ? a.X[src * a.ldx + i] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; kk++) {
            float xv[2];
#pragma unroll
            for (int j = 0; j < 2; j++) xv[j] = Xs[kk][pq + 16 * j];
#pragma unroll
            for (int mtx = 0; mtx < (DUAL ? 2 : 1); mtx++)
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float wv = Ws[mtx][kk][oq + 16 * i];
#pragma unroll
                    for (int j = 0; j < 2; j++) acc[mtx][i][j] = fmaf(wv, xv[j], acc[mtx][i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int p = p0 + pq + 16 * j;
        if (p >= p1) continue;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int o = o_base + oq + 16 * i;
            if (o >= a.O) continue;
            const float v = DUAL ? silu_g(acc[0][i][j]) * acc[1][i][j] : acc[0][i][j];
            a.out[(size_t)p * a.ldo + o] = v;
        }
    }
}

}  // namespace

cudaError_t launch_gemm_cc(const GemmArgs &a, bool dual, int max_tiles, cudaStream_t st) {
    dim3 grid((a.O + BO - 1) / BO, max_tiles);
    if (grid.y == 0) return cudaSuccess;
    if (dual) gemm_cc_kernel<true><<<grid, NT, 0, st>>>(a);
    else gemm_cc_kernel<false><<<grid, NT, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace coli
