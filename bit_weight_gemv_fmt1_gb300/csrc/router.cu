// router.cu -- router top-K that turns router logits into the (ids, weights)
// coli_moe_block consumes (colibri-strix commit log, "metal: full decode layer
// in ONE command buffer": sigmoid of the f32 router matvec, greedy argmax over
// sigmoid + bias with the CPU tie order, --topp truncation, norm_topk,
// routed_scale).
//
// One CTA per token row.  The score of expert e is sigmoid(logit_e) computed
// in double and rounded to f32, its key score + bias in f32; K rounds of a
// block-wide argmax (ties to the lower id) pick the experts; thread 0 then
// applies top-p, norm_topk and routed_scale with one IEEE rounding per
// operation (explicit _rn intrinsics, no contraction), so every decision and
// every weight is the f32 value of the definition.
#include <math.h>

#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int kTopkThreads = 256;

// (key, id) pair order of the argmax: larger key first, then lower id.
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
    if (ia < 0) return false;
    if (ib < 0) return true;
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *logits, const float *bias, int S, int E,
                                                            int K, float top_p, int norm_topk, float routed_scale,
                                                            int32_t *ids, float *w) {
    extern __shared__ float tsm[];
    float *score = tsm;                                          // [E]
    float *key = tsm + E;                                        // [E]
    unsigned char *taken = reinterpret_cast<unsigned char *>(tsm + 2 * E);
    __shared__ float s_k[kTopkThreads / 32];
    __shared__ int s_i[kTopkThreads / 32];
    __shared__ int s_sel[64];
    const int s = blockIdx.x;
    if (s >= S) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched as a programmatic dependent of the router matvec: its logits are
    // visible once the wait returns
    pdl_wait();
    const float *l = logits + (size_t)s * E;
    for (int e = tid; e < E; e += blockDim.x) {
        const float sc = (float)(1.0 / (1.0 + exp(-(double)l[e])));
        score[e] = sc;
        key[e] = __fadd_rn(sc, bias ? bias[e] : 0.0f);
        taken[e] = 0;
    }
    __syncthreads();
    for (int k = 0; k < K; k++) {
        float bk = 0.f;
        int bi = -1;
        for (int e = tid; e < E; e += blockDim.x)
            if (!taken[e] && better(key[e], e, bk, bi)) {
                bk = key[e];
                bi = e;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok_ = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ok_, oi, bk, bi)) {
                bk = ok_;
                bi = oi;
            }
        }
        if (lane == 0) {
            s_k[warp] = bk;
            s_i[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            float fk = s_k[0];
            int fi = s_i[0];
            for (int q = 1; q < (int)(blockDim.x >> 5); q++)
                if (better(s_k[q], s_i[q], fk, fi)) {
                    fk = s_k[q];
                    fi = s_i[q];
                }
            s_sel[k] = fi;
            taken[fi] = 1;
        }
        __syncthreads();
    }
    pdl_trigger();
    if (tid == 0) {
        float wt[64];
        for (int k = 0; k < K; k++) wt[k] = score[s_sel[k]];
        int keep = K;
        if (top_p > 0.0f && top_p < 1.0f) {
            float total = 0.0f;
            for (int k = 0; k < K; k++) total = __fadd_rn(total, wt[k]);
            const float limit = __fmul_rn(top_p, total);
            float cum = 0.0f;
            keep = 0;
            for (int k = 0; k < K; k++) {
                if (!(cum < limit)) break;
                cum = __fadd_rn(cum, wt[k]);
                keep++;
            }
        }
        if (norm_topk) {
            float sum = 0.0f;
            for (int k = 0; k < keep; k++) sum = __fadd_rn(sum, wt[k]);
            for (int k = 0; k < keep; k++) wt[k] = __fdiv_rn(wt[k], sum);
        }
        int32_t *id = ids + (size_t)s * K;
        float *wo = w + (size_t)s * K;
        for (int k = 0; k < K; k++) {
            const bool kept = k < keep;
            id[k] = kept ? s_sel[k] : -1;
            wo[k] = kept ? __fmul_rn(wt[k], routed_scale) : 0.0f;
        }
    }
}

}  // namespace

size_t topk_smem(int E) { return (size_t)E * (2 * sizeof(float) + 1) + 16; }

cudaError_t launch_topk(const float *logits, const float *bias, int S, int E, int K, float top_p, int norm_topk,
                        float routed_scale, int32_t *ids, float *w, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    const size_t smem = topk_smem(E);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_kernel, dim3(S), dim3(kTopkThreads), smem, st, logits, bias, S, E, K, top_p, norm_topk,
                      routed_scale, ids, w);
}

}  // namespace coli
