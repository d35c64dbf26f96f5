// noalloc.cu -- the decode expert block for callers that cannot allocate
// device memory.
//
// Some callers must not call cudaMalloc/cudaFree (or anything that does):
// latency-critical decode loops, because cudaMalloc/cudaFree synchronise the
// whole device, and processes in which another allocator (a framework's
// caching allocator, a pre-reserved pool) already owns the GPU memory, so a
// surprise allocation can fail.  coli_moe_block allocates its scratch (per
// stream) and its expert-table copy (per device) on first use; this variant
// keeps them in one file-scope device array instead, sized for the decode path
// only.
//
// The scratch array lives in every GPU that loads the library until the
// process exits.  Its device address is looked up once per device with
// cudaGetSymbolAddress, by the first call on that device.  All calls share the
// array: calls that may overlap on the GPU (different streams without
// ordering, several host threads) race and must be serialised by the caller.
// The expert descriptors reach the array through the parameters of a small
// copy kernel (no host buffer is read by the GPU), and only when they differ
// from the ones the previous call on the device left there.  The barrier words
// are cleared at the start of every call; the other regions are fully written
// before they are read.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "coli_internal.cuh"

using namespace coli;

namespace {

// Limits of the shared scratch.
constexpr int kNoallocMaxExperts = 1024;              // expert descriptors
constexpr long long kNoallocMaxHidden = 512 * 1024;   // floats of h: S*K*F
constexpr size_t kOffTable = 0;
constexpr size_t kOffBar = kOffTable + sizeof(ExpertDesc) * kNoallocMaxExperts;
constexpr size_t kOffH = (kOffBar + 2 * sizeof(unsigned) + 255) / 256 * 256;
constexpr size_t kScratchBytes = kOffH + sizeof(float) * kNoallocMaxHidden;   // about 2.2 MB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[64];   // device address of g_noalloc_scratch, per device ordinal
std::vector<ExpertDesc> g_mirror[64];   // per device: the descriptors the scratch holds

// Descriptors per copy launch: 128 x 120 bytes of kernel parameters.
constexpr int kFillChunk = 128;
struct FillArgs {
    ExpertDesc *dst;
    int n;
    ExpertDesc d[kFillChunk];
};
__global__ void table_fill_kernel(const FillArgs a) {
    for (int i = threadIdx.x; i < a.n; i += blockDim.x) a.dst[i] = a.d[i];
}

bool same_desc(const ExpertDesc &p, const ExpertDesc &q) { return memcmp(&p, &q, sizeof p) == 0; }

__attribute__((format(printf, 2, 3))) int bad(int code, const char *fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    return set_last_error(code, msg);
}

}  // namespace

namespace coli {
cudaError_t launch_table_fill(ExpertDesc *dst, const ExpertDesc *src, int n, cudaStream_t st) {
    for (int i0 = 0; i0 < n; i0 += kFillChunk) {
        FillArgs a;
        a.dst = dst + i0;
        a.n = std::min(kFillChunk, n - i0);
        memcpy(a.d, src + i0, sizeof(ExpertDesc) * (size_t)a.n);
        table_fill_kernel<<<1, 128, 0, st>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
}  // namespace coli

extern "C" int coli_moe_block_noalloc(const float *x, int S, const coli_expert *experts, int n_experts,
                                      const int32_t *ids, const float *w, int K, float *y, int32_t *dev_error,
                                      void *stream) {
    clear_last_error();
    cudaStream_t st = (cudaStream_t)stream;
    if (!x || !y || !ids || !w || !experts || !dev_error) return bad(COLI_EINVAL, "a pointer argument is NULL");
    if (S < 1 || K < 1 || K > 64) return bad(COLI_EINVAL, "need S >= 1 and 1 <= K <= 64 (got S=%d K=%d)", S, K);
    if ((long long)S * K > kMaxDecodeSlots)
        return bad(COLI_EINVAL, "S*K=%lld exceeds the no-allocation limit of %d routed slots", (long long)S * K,
                   kMaxDecodeSlots);
    if (n_experts < 1 || n_experts > kNoallocMaxExperts)
        return bad(COLI_EINVAL, "n_experts=%d outside 1..%d (no-allocation table limit)", n_experts,
                   kNoallocMaxExperts);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return bad(COLI_ECUDA, "cudaGetDevice failed");
    const coli_tensor *g0 = experts[0].gate;
    if (!g0) return bad(COLI_EINVAL, "expert 0 gate is NULL");
    const long long F = g0->O, H = g0->I;
    const int fmt = g0->fmt;
    for (int e = 0; e < n_experts; e++) {
        const coli_tensor *m[3] = {experts[e].gate, experts[e].up, experts[e].down};
        for (int k = 0; k < 3; k++) {
            if (!m[k]) return bad(COLI_EINVAL, "expert %d matrix %d is NULL", e, k);
            if (m[k]->device != dev) return bad(COLI_EDEVICE, "expert %d lives on another device", e);
            if (m[k]->fmt != fmt) return bad(COLI_EFMT, "expert %d matrix %d: one format per table", e, k);
            if (fmt == 4 && m[k]->gs % 32 != 0)
                return bad(COLI_EFMT, "expert %d matrix %d: gs=%d is not a multiple of 32", e, k, m[k]->gs);
        }
        if (m[0]->O != F || m[0]->I != H || m[1]->O != F || m[1]->I != H || m[2]->O != H || m[2]->I != F)
            return bad(COLI_EINVAL, "expert %d: gate/up must be [%lld][%lld] and down [%lld][%lld]", e, F, H, H, F);
    }
    const int n_slots = S * K;
    if ((long long)n_slots * F > kNoallocMaxHidden)
        return bad(COLI_EINVAL, "S*K*F=%lld exceeds the no-allocation scratch (%lld floats)", (long long)n_slots * F,
                   kNoallocMaxHidden);
    if (int rc = injected_gate()) return rc;

    // scratch address, once per device
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_addr[dev]) {
            void *p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return bad(COLI_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            g_addr[dev] = p;
        }
        base = g_addr[dev];
    }
    int n_sm = 0, optin = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return bad(COLI_ECUDA, "cudaDeviceGetAttribute failed");

    // shared-memory plan of the decode kernel (two CTAs per SM)
    const int cpr_gu = g0->cpr, cpr_d = experts[0].down->cpr;
    const int xlen_gu = staged_len(fmt, cpr_gu), xlen_d = staged_len(fmt, cpr_d);
    const size_t budget = 110 * 1024 / 4;
    const int rpc_alloc = (int)((H + n_sm - 1) / n_sm);
    const size_t fixed = (size_t)S * rpc_alloc;
    int sb = 0;
    if (budget > fixed + xlen_d + rpc_alloc)
        sb = (int)std::min<size_t>((size_t)n_slots, (budget - fixed) / (size_t)(xlen_d + rpc_alloc));
    const size_t stage = std::max((size_t)S * xlen_gu, (size_t)sb * xlen_d);
    const size_t smem = (stage + (size_t)sb * rpc_alloc + fixed) * sizeof(float);
    if (sb < 1 || (size_t)S * xlen_gu > budget || smem > (size_t)optin)
        return bad(COLI_EINVAL, "activations too large for the single-launch decode kernel (S=%d, H=%lld)", S, H);
    int per_sm = 0;
    if (moe_decode_occupancy(fmt, smem, &per_sm) != cudaSuccess || per_sm < 1)
        return bad(COLI_ECUDA, "decode kernel occupancy query failed");
    const int grid = per_sm * n_sm;

    // descriptors -> scratch table (only when they changed since the previous
    // call on this device); clear the barrier words and the error output
    std::vector<ExpertDesc> h((size_t)n_experts);
    for (int e = 0; e < n_experts; e++) {
        const coli_tensor *m[3] = {experts[e].gate, experts[e].up, experts[e].down};
        for (int k = 0; k < 3; k++) {
            MatDesc &d = h[e].m[k];
            memset(&d, 0, sizeof d);
            d.q = m[k]->q;
            d.s = m[k]->s;
            d.rs = m[k]->rs;
            d.gs = m[k]->fmt == 4 ? m[k]->gs : m[k]->fmt == 7 ? kFp8Block : 0;
            d.ng = m[k]->ng;
            d.tmap = m[k]->tmap;
        }
    }
    unsigned char *b = (unsigned char *)base;
    cudaError_t e = cudaSuccess;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        std::vector<ExpertDesc> &mir = g_mirror[dev];
        bool same = mir.size() >= h.size();
        for (size_t i = 0; i < h.size() && same; i++) same = same_desc(mir[i], h[i]);
        if (!same) {
            e = launch_table_fill((ExpertDesc *)(b + kOffTable), h.data(), n_experts, st);
            if (e == cudaSuccess) {
                if (mir.size() < h.size()) mir.resize(h.size());
                std::copy(h.begin(), h.end(), mir.begin());
            } else {
                mir.clear();
            }
        }
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(b + kOffBar, 0, 2 * sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dev_error, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return bad(COLI_ECUDA, "scratch set-up: %s", cudaGetErrorString(e));

    MoeDecodeArgs a;
    memset(&a, 0, sizeof a);
    a.x = x;
    a.ids = ids;
    a.w = w;
    a.y = y;
    a.table = (const ExpertDesc *)(b + kOffTable);
    a.n_experts = n_experts;
    a.S = S;
    a.K = K;
    a.H = (int)H;
    a.F = (int)F;
    a.cpr_gu = cpr_gu;
    a.cpr_d = cpr_d;
    a.hbuf = (float *)(b + kOffH);
    a.bar = (unsigned *)(b + kOffBar);
    a.err = dev_error;
    a.sb = sb;
    a.rpc = (int)((H + grid - 1) / grid);
    a.timeout_ns = 2000000000LL;
    e = launch_moe_decode(a, fmt, grid, smem, st);
    if (e != cudaSuccess) return bad(COLI_ECUDA, "decode expert-block launch: %s", cudaGetErrorString(e));
    count_call(1, 0);
    return COLI_OK;
}
