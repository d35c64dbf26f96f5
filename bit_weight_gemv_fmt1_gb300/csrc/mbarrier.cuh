// mbarrier.cuh -- shared-memory mbarrier waits, bulk copies and named
// barriers used by the pipelined kernels (tensor-core GEMM, streamed decode).
//
// Every wait is bounded: it gives up once a deadline (globaltimer ns) has
// passed or the CTA has raised its abort flag, so a kernel whose partner
// never arrives records an error and returns instead of hanging the GPU.
#pragma once
#include <stdint.h>

#include "coli_internal.cuh"

namespace coli {

// try_wait sleeps up to this long (ns) while the phase is incomplete, so a
// waiting warp leaves the issue slots to the working ones.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
// One thread's bounded wait: false once `deadline` has passed or the CTA aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, uint64_t deadline, volatile int *abort) {
    while (!mbar_try(b, parity)) {
        if (*abort) return false;
        if (global_ns() > deadline) return false;
    }
    return true;
}
// A whole warp's bounded wait: every lane polls, lane 0 decides on expiry,
// so the warp leaves together either way.
__device__ __forceinline__ bool warp_wait(uint64_t *b, uint32_t parity, uint64_t deadline, volatile int *abort,
                                          int lane) {
    while (true) {
        const bool done = mbar_try(b, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int stop = 0;
        if (lane == 0) stop = (*abort != 0) || global_ns() > deadline;
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}
// Contiguous global -> shared copy on the TMA engine; both addresses and the
// size must be multiples of 16 bytes.  Completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
// Barrier among the first `n` threads of the CTA (named barrier `id`).
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

}  // namespace coli
