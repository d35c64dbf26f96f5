// decode_route.cuh -- pieces shared by the single-launch decode expert-block
// kernels (stream_decode.cu, decode_mma.cu): the routing of the one token
// (phase 0) and the grid-wide barrier between the gate/up and down phases.
#pragma once
#include <stdint.h>

#include "coli_internal.cuh"
#include "mbarrier.cuh"

namespace coli {

// The token's routed experts after phase 0: distinct ids in ascending order,
// the routing weights of duplicate slots summed (moe_block sums w_k * expert
// output over the K slots, so a repeated id contributes the sum of its
// weights), and the expert-table pointers of each.
struct DecodeRouting {
    int ids[kMaxDecodeSlots];
    float w[kMaxDecodeSlots];
    int exp[kMaxDecodeSlots];
    float ew[kMaxDecodeSlots];
    const uint8_t *q[kMaxDecodeSlots][3];   // gate, up, down codes
    const float *s[kMaxDecodeSlots][3];     // and scales
    int nact, bad;
};

// Phase 0 by one warp, for n <= 32 slots: the lanes rank the slots with
// shuffles and ballots.  Ids outside [-1, n_experts) set r.bad.  The results
// are in shared memory once the warp has passed a barrier with the readers.
__device__ __forceinline__ void decode_route_warp(DecodeRouting &r, const int32_t *ids, const float *w, int n,
                                                  int n_experts, const ExpertDesc *table) {
    const int lane = threadIdx.x & 31;
    const bool valid = lane < n;
    int my_id = -1;
    float my_w = 0.f;
    if (valid) {
        my_id = ids[lane];
        my_w = w[lane];
    }
    const bool bad = valid && (my_id < -1 || my_id >= n_experts);
    // the slot's expert pointers are fetched while the ranks are formed
    const uint8_t *eq[3] = {nullptr, nullptr, nullptr};
    const float *es[3] = {nullptr, nullptr, nullptr};
    if (valid && !bad && my_id >= 0) {
        const ExpertDesc &E = table[my_id];
#pragma unroll
        for (int m = 0; m < 3; m++) {
            eq[m] = E.m[m].q;
            es[m] = E.m[m].s;
        }
    }
    const unsigned any_bad = __ballot_sync(0xffffffffu, bad);
    bool first = valid && my_id >= 0;
    int rank = 0;
    float wsum = 0.f;
    for (int t = 0; t < n; t++) {
        const int f = __shfl_sync(0xffffffffu, my_id, t);
        const float wt = __shfl_sync(0xffffffffu, my_w, t);
        if (f == my_id) {
            wsum += wt;
            if (t < lane) first = false;
        }
        // count each smaller id once, at its first slot
        const unsigned same_before = __ballot_sync(0xffffffffu, lane < t && my_id == f);
        if (f >= 0 && f < my_id && same_before == 0u) rank++;
    }
    if (first && !any_bad) {
        r.exp[rank] = my_id;
        r.ew[rank] = wsum;
#pragma unroll
        for (int m = 0; m < 3; m++) {
            r.q[rank][m] = eq[m];
            r.s[rank][m] = es[m];
        }
    }
    const unsigned nf = __popc(__ballot_sync(0xffffffffu, first));
    if (lane == 0) {
        r.bad = any_bad != 0u;
        r.nact = (int)nf;
    }
}

// Phase 0, called by every thread of the CTA (it contains __syncthreads).
// For n <= 32 slots warp `rw` ranks the slots (decode_route_warp) while the
// rest of the CTA waits; above that the first n threads rank through shared
// memory.  Ids outside [-1, n_experts) set r.bad.
__device__ __forceinline__ void decode_route(DecodeRouting &r, const int32_t *ids, const float *w, int n,
                                             int n_experts, const ExpertDesc *table, int rw) {
    const int tid = threadIdx.x, warp = tid >> 5;
    if (n <= 32) {
        if (warp == rw) decode_route_warp(r, ids, w, n, n_experts, table);
        __syncthreads();
        return;
    }
    if (tid == 0) {
        r.bad = 0;
        r.nact = 0;
    }
    __syncthreads();
    if (tid < n) {
        const int e = ids[tid];
        r.ids[tid] = e;
        r.w[tid] = w[tid];
        if (e < -1 || e >= n_experts) atomicOr(&r.bad, 1);
    }
    __syncthreads();
    if (!r.bad && tid < n) {
        const int e = r.ids[tid];
        bool first = e >= 0;
        int rank = 0;
        float wsum = 0.f;
        for (int t = 0; t < n; t++) {
            const int f = r.ids[t];
            if (f == e) {
                wsum += r.w[t];
                if (t < tid) first = false;
            }
            if (f >= 0 && f < e) {
                bool fst = true;   // count each smaller id once, at its first slot
                for (int u = 0; u < t; u++) fst &= r.ids[u] != f;
                rank += fst;
            }
        }
        if (first) {
            r.exp[rank] = e;
            r.ew[rank] = wsum;
            const ExpertDesc &E = table[e];
#pragma unroll
            for (int m = 0; m < 3; m++) {
                r.q[rank][m] = E.m[m].q;
                r.s[rank][m] = E.m[m].s;
            }
            atomicAdd(&r.nact, 1);
        }
    }
    __syncthreads();
}

// One thread per CTA: arrive at the grid barrier (counter `arrived`, zero
// before the call) and wait, bounded, until every CTA of the grid has
// arrived.  The release before the arrival publishes the CTA's global writes;
// the acquire loads order the other CTAs' writes before what follows.
// False on expiry (DEV_ERR_TIMEOUT recorded).
__device__ __forceinline__ bool decode_grid_barrier(unsigned *arrived, uint64_t deadline, int *err) {
    __threadfence();
    atomicAdd(arrived, 1u);
    while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(arrived) : "memory");
        if (v >= gridDim.x) break;
        if (global_ns() > deadline) {
            atomicCAS(err, 0, DEV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    __threadfence();
    return true;
}

// One thread per CTA, as the CTA leaves: the last CTA out zeroes the barrier
// counter and itself for the next call, also after an aborted call.
__device__ __forceinline__ void decode_exit(unsigned *exitc, unsigned *arrived) {
    __threadfence();
    if (atomicAdd(exitc, 1u) == gridDim.x - 1) {
        *arrived = 0u;
        *exitc = 0u;
        __threadfence();
    }
}

}  // namespace coli
