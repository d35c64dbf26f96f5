// api.cu -- the C ABI declared in include/coli.h: argument checks, uploads,
// per-device / per-stream scratch, dispatch to the kernels, error reporting.
// Every entry point refuses what it cannot compute (with a code and a
// message) before launching anything; there is no other implementation to
// fall back to.
#include <array>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <unordered_map>
#include <algorithm>
#include <vector>

#include "coli_internal.cuh"

using namespace coli;

namespace {

// ------------------------------------------------------------------ errors
thread_local char g_msg[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    if (e == cudaErrorMemoryAllocation)
        return fail(COLI_ENOMEM, "%s: %s", what, cudaGetErrorString(e));
    return fail(COLI_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CU(call, what)                                   \
    do {                                                 \
        cudaError_t e_ = (call);                         \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// ------------------------------------------------------------------ stats
std::atomic<uint64_t> g_calls{0}, g_launches{0}, g_wbytes{0};
std::atomic<uint64_t> g_uid{1};

std::atomic<int64_t> &fail_after() {
    static std::atomic<int64_t> v{[] {
        const char *s = getenv("COLI_FAIL_AFTER");
        return s && *s ? (int64_t)atoll(s) : (int64_t)-1;
    }()};
    return v;
}

// Host-side fault injection gate for compute calls.
int injected() {
    auto &f = fail_after();
    int64_t cur = f.load();
    while (cur > 0 && !f.compare_exchange_weak(cur, cur - 1)) {
    }
    if (cur == 0) return fail(COLI_EINJECTED, "failure injected (fail-after counter reached zero)");
    return COLI_OK;
}

void count(int launches, uint64_t wbytes) {
    g_calls++;
    g_launches += launches;
    g_wbytes += wbytes;
}

// ------------------------------------------------------------------ device state
struct Workspace {
    unsigned *bar = nullptr;      // grid barrier words (kBarrierBytes)
    void *buf = nullptr;          // scratch
    size_t cap = 0;
    void *rbuf = nullptr;         // router logits (kept apart from buf, which the router matvec may use)
    size_t rcap = 0;
    unsigned *cnt = nullptr;      // counters of the streamed decode block (zero between calls)
    size_t cnt_cap = 0;           // words
};

struct CachedTable {
    ExpertDesc *d = nullptr;
    int n = 0;
    uint64_t last_use = 0;
};

struct DeviceState {
    std::mutex mu;
    int *err = nullptr;           // device error word
    int n_sm = 0;
    size_t smem_optin = 0;
    std::map<cudaStream_t, Workspace> ws;
    std::unordered_map<uint64_t, CachedTable> tables;
    uint64_t tick = 0;
};

std::mutex g_dev_mu;
std::map<int, DeviceState *> g_dev;

int device_state(DeviceState **out) {
    int dev = 0;
    CU(cudaGetDevice(&dev), "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
        *out = it->second;
        return COLI_OK;
    }
    DeviceState *d = new DeviceState();
    CU(cudaMalloc(&d->err, sizeof(int)), "cudaMalloc(error word)");
    CU(cudaMemset(d->err, 0, sizeof(int)), "cudaMemset(error word)");
    CU(cudaDeviceGetAttribute(&d->n_sm, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
    int optin = 0;
    CU(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "cudaDeviceGetAttribute");
    d->smem_optin = (size_t)optin;
    g_dev[dev] = d;
    *out = d;
    return COLI_OK;
}

// Router-logit scratch of at least `bytes` for this stream (grown like workspace()).
int router_scratch(DeviceState *d, cudaStream_t st, size_t bytes, float **out) {
    std::lock_guard<std::mutex> lk(d->mu);
    Workspace &w = d->ws[st];
    if (w.rcap < bytes) {
        if (w.rbuf) {
            CU(cudaDeviceSynchronize(), "cudaDeviceSynchronize(router scratch growth)");
            CU(cudaFree(w.rbuf), "cudaFree(router scratch)");
            w.rbuf = nullptr;
            w.rcap = 0;
        }
        CU(cudaMalloc(&w.rbuf, bytes), "cudaMalloc(router scratch)");
        w.rcap = bytes;
    }
    *out = (float *)w.rbuf;
    return COLI_OK;
}

// Scratch of at least `bytes` for this stream (grown on demand; growing waits
// for the device so that no queued kernel still uses the old buffer).
int workspace(DeviceState *d, cudaStream_t st, size_t bytes, Workspace **out) {
    std::lock_guard<std::mutex> lk(d->mu);
    Workspace &w = d->ws[st];
    if (!w.bar) {
        // words 0-1: counter and generation of the resetting grid barrier
        CU(cudaMalloc(&w.bar, kBarrierBytes), "cudaMalloc(barrier)");
        CU(cudaMemset(w.bar, 0, kBarrierBytes), "cudaMemset(barrier)");
    }
    if (w.cap < bytes) {
        if (w.buf) {
            CU(cudaDeviceSynchronize(), "cudaDeviceSynchronize(workspace growth)");
            CU(cudaFree(w.buf), "cudaFree(workspace)");
            w.buf = nullptr;
            w.cap = 0;
        }
        const size_t want = bytes + bytes / 4;
        CU(cudaMalloc(&w.buf, want), "cudaMalloc(workspace)");
        w.cap = want;
    }
    *out = &w;
    return COLI_OK;
}

// Counter words of the streamed decode block for this stream, zero at
// allocation; the kernel leaves them zero at the end of every call.
int decode_counters(DeviceState *d, cudaStream_t st, size_t words, unsigned **out) {
    std::lock_guard<std::mutex> lk(d->mu);
    Workspace &w = d->ws[st];
    if (w.cnt_cap < words) {
        if (w.cnt) {
            CU(cudaDeviceSynchronize(), "cudaDeviceSynchronize(counter growth)");
            CU(cudaFree(w.cnt), "cudaFree(counters)");
            w.cnt = nullptr;
            w.cnt_cap = 0;
        }
        const size_t want = std::max<size_t>(words, 4096);
        CU(cudaMalloc(&w.cnt, want * sizeof(unsigned)), "cudaMalloc(counters)");
        CU(cudaMemset(w.cnt, 0, want * sizeof(unsigned)), "cudaMemset(counters)");
        w.cnt_cap = want;
    }
    *out = w.cnt;
    return COLI_OK;
}

int check_tensor(const coli_tensor *t, const char *name) {
    if (!t) return fail(COLI_EINVAL, "%s is NULL", name);
    int dev = 0;
    CU(cudaGetDevice(&dev), "cudaGetDevice");
    if (t->device != dev)
        return fail(COLI_EDEVICE, "%s lives on device %d but device %d is current", name, t->device, dev);
    return COLI_OK;
}

int64_t host_row_bytes(int fmt, int64_t I) {
    switch (fmt) {
    case 0: return 4 * I;
    case 1: return I;
    case 2: case 4: return (I + 1) / 2;
    case 3: return (I + 3) / 4;
    case 5: return 3 * ((I + 7) / 8);
    case 7: return I;
    default: return -1;
    }
}

// Row of an int3 (fmt=5) upload, 3*ceil(I/8) bytes (element 8j+t is bits [3t, 3t+2] of the
// little-endian 24-bit word in bytes 3j..3j+2), written as the int4 row of the device layout,
// ceil(I/2) bytes: element i's code c becomes the nibble c + 4, element 2j the low nibble of
// byte j.  Each output byte holds two consecutive codes, i.e. one 6-bit field of the word,
// looked up in a table; the nibbles past I are zero.
void int3_row_to_int4(const uint8_t *src, int64_t I, uint8_t *dst) {
    static const auto lut = [] {
        std::array<uint8_t, 64> t{};
        for (int v = 0; v < 64; v++) t[v] = (uint8_t)(((v & 7) + 4) | (((v >> 3) + 4) << 4));
        return t;
    }();
    const int64_t full = I / 8;   // units whose 8 codes all lie inside the row
    for (int64_t u = 0; u < full; u++) {
        const uint32_t w = (uint32_t)src[3 * u] | ((uint32_t)src[3 * u + 1] << 8) | ((uint32_t)src[3 * u + 2] << 16);
        for (int k = 0; k < 4; k++) dst[4 * u + k] = lut[(w >> (6 * k)) & 63u];
    }
    if (I % 8) {   // the last, partial unit
        const int64_t u = full;
        const uint32_t w = (uint32_t)src[3 * u] | ((uint32_t)src[3 * u + 1] << 8) | ((uint32_t)src[3 * u + 2] << 16);
        for (int64_t i = 8 * u; i < 8 * u + 8; i += 2) {
            const uint8_t lo = i < I ? (uint8_t)(((w >> (3 * (i - 8 * u))) & 7u) + 4u) : 0;
            const uint8_t hi = i + 1 < I ? (uint8_t)(((w >> (3 * (i + 1 - 8 * u))) & 7u) + 4u) : 0;
            if (i < I) dst[i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

MatDesc desc_of(const coli_tensor *t) {
    MatDesc m;
    m.q = t->q;
    m.s = t->s;
    m.rs = t->rs;
    m.gs = t->fmt == 4 ? t->gs : t->fmt == 7 ? kFp8Block : 0;
    m.ng = t->ng;
    m.tmap = t->tmap;
    return m;
}

}  // namespace

namespace coli {
// Record `msg` as this thread's last error (for coli_last_error) and return code.
int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }
void clear_last_error() { g_msg[0] = 0; }
int injected_gate() { return injected(); }
void count_call(int launches, uint64_t weight_bytes) { count(launches, weight_bytes); }
}  // namespace coli

// =================================================================== ABI
extern "C" {

const char *coli_version(void) { return "coli-gb300 1.0 (sm_103a)"; }

const char *coli_last_error(void) { return g_msg; }

void coli_get_stats(coli_stats *out) {
    if (!out) return;
    out->calls = g_calls.load();
    out->launches = g_launches.load();
    out->weight_bytes = g_wbytes.load();
}

void coli_reset_stats(void) {
    g_calls = 0;
    g_launches = 0;
    g_wbytes = 0;
}

void coli_set_fail_after(int64_t n) { fail_after().store(n < 0 ? -1 : n); }

// Argument checks shared by both uploads.
static int check_upload(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                        coli_tensor **out) {
    if (!out) return fail(COLI_EINVAL, "out is NULL");
    *out = nullptr;
    if (fmt < 0 || fmt == 6 || fmt > 7)
        return fail(COLI_EFMT, "unknown weight format %d (supported: 0..5, 7)", fmt);
    if (fmt == 4 && (gs < 2 || (gs & 1)))
        return fail(COLI_EFMT, "fmt=4 needs an even group size >= 2, got gs=%d", gs);
    if (fmt == 5 && (gs < 8 || gs % 8 != 0))
        return fail(COLI_EFMT, "fmt=5 needs a group size that is a multiple of 8, got gs=%d", gs);
    if (O < 1 || I < 1) return fail(COLI_EINVAL, "O and I must be >= 1 (got O=%lld I=%lld)", (long long)O, (long long)I);
    if (O > (1LL << 31) - 1 || I > (1LL << 30))
        return fail(COLI_EINVAL, "matrix too large (O=%lld I=%lld)", (long long)O, (long long)I);
    if (!data) return fail(COLI_EINVAL, "data is NULL");
    if (fmt != 0 && !scales) return fail(COLI_EINVAL, "fmt=%d needs scales", fmt);
    return COLI_OK;
}

// A new tensor with the shape, layout and byte counts of (fmt, gs, O, I); no storage yet.
// int3 (fmt=5) is stored as int4 nibbles with fmt=4's group scales: code c becomes the nibble
// c + 4, whose int4 value (nibble - 8) is the int3 value c - 4, so every int4 kernel serves it
// (the device copy, and what the kernels read, is 4/3 of the int3 bytes).
static coli_tensor *new_tensor(int fmt, int gs, int64_t O, int64_t I, int64_t *n_scales) {
    coli_tensor *t = new coli_tensor();
    const int dfmt = fmt == 5 ? 4 : fmt;
    t->ufmt = fmt;
    t->fmt = dfmt;
    t->gs = dfmt == 4 ? gs : 0;
    t->O = O;
    t->I = I;
    t->ng = dfmt == 4 ? (int)((I + gs - 1) / gs) : dfmt == 7 ? (int)((I + kFp8Block - 1) / kFp8Block) : 1;
    const int64_t hrb = host_row_bytes(dfmt, I);
    t->rs = (hrb + 15) / 16 * 16;
    t->cpr = (int)((I + epc_of(dfmt) - 1) / epc_of(dfmt));
    *n_scales = dfmt == 0   ? 0
                : dfmt == 4 ? O * t->ng
                : dfmt == 7 ? (O + kFp8Block - 1) / kFp8Block * t->ng
                            : O;
    t->alg_bytes = O * host_row_bytes(fmt, I) + 4 * *n_scales;
    t->dev_bytes = O * t->rs + 4 * *n_scales;
    t->uid = g_uid++;
    return t;
}

int coli_tensor_upload(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                       void *stream, coli_tensor **out) {
    g_msg[0] = 0;
    if (int rc = check_upload(fmt, gs, O, I, data, scales, out)) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int device = 0;
    CU(cudaGetDevice(&device), "cudaGetDevice");

    int64_t n_scales = 0;
    coli_tensor *t = new_tensor(fmt, gs, O, I, &n_scales);
    const int64_t hrb = host_row_bytes(t->fmt, I);   // bytes of a row in the device layout, unpadded
    std::vector<uint8_t> conv;                        // int3 rows as int4 (kept until the copy completed)
    if (fmt == 5) {
        conv.resize((size_t)(O * hrb));
        const int64_t srb = host_row_bytes(5, I);
        for (int64_t o = 0; o < O; o++)
            int3_row_to_int4((const uint8_t *)data + o * srb, I, conv.data() + o * hrb);
        data = conv.data();
    }
    t->device = device;
    cudaError_t e = cudaMalloc(&t->q, (size_t)(O * t->rs));
    if (e == cudaSuccess && n_scales) e = cudaMalloc(&t->s, (size_t)n_scales * 4);
    if (e == cudaSuccess) e = cudaMemsetAsync(t->q, 0, (size_t)(O * t->rs), st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(t->q, (size_t)t->rs, data, (size_t)hrb, (size_t)hrb, (size_t)O,
                              cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && n_scales)
        e = cudaMemcpyAsync(t->s, scales, (size_t)n_scales * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && fmt == 1) {
        e = launch_fmt1_encode(t->q, O * t->rs, st);
        g_launches++;
    }
    if (e == cudaSuccess && (t->fmt == 2 || t->fmt == 4)) {
        // without a map (a shape the TMA descriptor rejects) the tensor-core path is not used for this tensor
        alignas(64) unsigned char map[128];
        if (encode_codes_map(t->q, t->rs, O, map) == cudaSuccess) {
            e = cudaMalloc(&t->tmap, 128);
            if (e == cudaSuccess) e = cudaMemcpyAsync(t->tmap, map, 128, cudaMemcpyHostToDevice, st);
        }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        coli_tensor_free(t);
        return cuda_fail(e, "coli_tensor_upload");
    }
    *out = t;
    return COLI_OK;
}

int coli_tensor_upload_host(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                            coli_tensor **out) {
    g_msg[0] = 0;
    if (int rc = check_upload(fmt, gs, O, I, data, scales, out)) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    int device = 0;
    CU(cudaGetDevice(&device), "cudaGetDevice");
    int64_t n_scales = 0;
    coli_tensor *t = new_tensor(fmt, gs, O, I, &n_scales);
    const int64_t hrb = host_row_bytes(t->fmt, I);   // bytes of a row in the device layout, unpadded
    const int64_t srb = host_row_bytes(fmt, I);      // bytes of a row as uploaded
    t->host = 1;
    t->dev_bytes = 0;
    t->device = device;
    const unsigned flags = cudaHostAllocMapped | cudaHostAllocPortable;
    cudaError_t e = cudaHostAlloc(&t->hq, (size_t)(O * t->rs), flags);
    if (e == cudaSuccess && n_scales) e = cudaHostAlloc(&t->hs, (size_t)n_scales * 4, flags);
    if (e == cudaSuccess) {
        // the device layout, written by the CPU: rows padded to 16 bytes with zeros,
        // int8 stored offset binary
        uint8_t *q = (uint8_t *)t->hq;
        const uint8_t *src = (const uint8_t *)data;
        for (int64_t o = 0; o < O; o++) {
            uint8_t *row = q + o * t->rs;
            if (fmt == 5)
                int3_row_to_int4(src + o * srb, I, row);
            else
                memcpy(row, src + o * srb, (size_t)hrb);
            memset(row + hrb, 0, (size_t)(t->rs - hrb));
            if (fmt == 1)
                for (int64_t i = 0; i < hrb; i++) row[i] ^= 0x80;
        }
        if (n_scales) memcpy(t->hs, scales, (size_t)n_scales * 4);
        e = cudaHostGetDevicePointer((void **)&t->q, t->hq, 0);
        if (e == cudaSuccess && n_scales) e = cudaHostGetDevicePointer((void **)&t->s, t->hs, 0);
    }
    if (e != cudaSuccess) {
        coli_tensor_free(t);
        return cuda_fail(e, "coli_tensor_upload_host");
    }
    *out = t;
    return COLI_OK;
}

void coli_tensor_free(coli_tensor *t) {
    if (!t) return;
    if (t->host) {
        if (t->hq) cudaFreeHost(t->hq);
        if (t->hs) cudaFreeHost(t->hs);
        delete t;
        return;
    }
    if (t->q) cudaFree(t->q);
    if (t->s) cudaFree(t->s);
    if (t->tmap) cudaFree(t->tmap);
    delete t;
}

int coli_tensor_info(const coli_tensor *t, int *fmt, int *gs, int64_t *O, int64_t *I, int64_t *device_bytes,
                     int64_t *alg_bytes) {
    if (!t) return fail(COLI_EINVAL, "tensor is NULL");
    if (fmt) *fmt = t->ufmt;
    if (gs) *gs = t->gs;
    if (O) *O = t->O;
    if (I) *I = t->I;
    if (device_bytes) *device_bytes = t->dev_bytes;
    if (alg_bytes) *alg_bytes = t->alg_bytes;
    return COLI_OK;
}

// ------------------------------------------------------------------ matmul
static int run_matmul(int n, const coli_tensor *const *W, const float *x, float *const *y, int S,
                      cudaStream_t st) {
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    const coli_tensor *W0 = W[0];
    uint64_t wbytes = 0;
    for (int m = 0; m < n; m++) wbytes += (uint64_t)W[m]->alg_bytes;
    bool generic = false, host_any = false;
    for (int m = 0; m < n; m++) generic |= (W0->fmt == 4 && (W[m]->gs % 32) != 0);
    // host-resident weights are read with plain loads only (no bulk copies, no TMA)
    for (int m = 0; m < n; m++) host_any |= W[m]->host != 0;
    const size_t smem = gemv_smem_bytes(W0->fmt, W0->cpr, S, (int)W0->I, generic);
    bool slab = S == 1 && !generic;
    for (int m = 0; m < n && slab; m++) slab = slab_supported(W[m]->fmt, W[m]->gs) && W[m]->gs == W0->gs;
    if (S <= 8 && smem <= ds->smem_optin) {
        GemvJob job;
        memset(&job, 0, sizeof job);
        job.n = n;
        job.fmt = W0->fmt;
        job.I = (int)W0->I;
        job.cpr = W0->cpr;
        job.S = S;
        job.x = x;
        job.row_start[0] = 0;
        for (int m = 0; m < n; m++) {
            job.q[m] = W[m]->q;
            job.s[m] = W[m]->s;
            job.y[m] = y[m];
            job.O[m] = (int)W[m]->O;
            job.gs[m] = W[m]->fmt == 4 ? W[m]->gs : 32;
            job.ng[m] = W[m]->ng;
            job.rs[m] = W[m]->rs;
            job.row_start[m + 1] = job.row_start[m] + job.O[m];
        }
        job.err = ds->err;
        int nl = 0;
        cudaError_t e;
        // S = 1..4, int4 (fmt 2; fmt 4 with gs 64 or 128), one row length and gs for all matrices,
        // at least 4 MB: the tensor-core streamed matvec (gemv_mma.cu)
        bool mma = S <= 4 && !host_any && (W0->fmt == 2 || W0->fmt == 4) && wbytes >= (4u << 20);
        for (int m = 0; m < n && mma; m++)
            mma = W[m]->fmt == W0->fmt && W[m]->I == W0->I && W[m]->rs == W0->rs && W[m]->ng == W0->ng &&
                  (W0->fmt != 4 || W[m]->gs == W0->gs);
        if (mma) {
            GmArgs ga;
            size_t gsm = 0;
            int ggrid = 0;
            if (gm_plan(W0->fmt, W0->fmt == 4 ? W0->gs : 0, (int)W0->I, (int)W0->rs, W0->ng, n, job.O, S, ds->n_sm,
                        (size_t)ds->smem_optin, &ga, &gsm, &ggrid)) {
                for (int m = 0; m < n; m++) {
                    ga.q[m] = W[m]->q;
                    ga.s[m] = W[m]->s;
                    ga.y[m] = y[m];
                }
                ga.x = x;
                ga.err = ds->err;
                if (int rc = decode_counters(ds, st, gm_counter_words(), &ga.ctr)) return rc;
                e = launch_gemv_mma(ga, ggrid, gsm, st);
                if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
                count(1, wbytes);
                return COLI_OK;
            }
        }
        // S = 1, fmt 1-4 (fmt 4: gs a power-of-two multiple of 32 and a multiple of 4
        // groups per row; fmt 1-3: every O a multiple of 4, for the row-scale copies):
        // weights streamed by bulk copies (below ~4 MB the slab kernel's shorter start-up wins)
        const int fmt0 = W0->fmt;
        // (fmt 0 and 7 copy no scales with the rows: f32 has none, FP8 block scales are read from global)
        const bool no_row_scales = fmt0 == 0 || fmt0 == 7;
        bool stream = S == 1 && !host_any && ((fmt0 >= 0 && fmt0 <= 4) || fmt0 == 7) && W0->I % 128 == 0 &&
                      ((uintptr_t)x & 15) == 0 && wbytes >= (4u << 20);
        for (int m = 0; m < n && stream; m++)
            stream = fmt0 == 4 ? (W[m]->gs == W0->gs && slab_supported(4, W[m]->gs) && W[m]->ng % 4 == 0)
                               : (no_row_scales || W[m]->O % 4 == 0);
        const int lpr = stream ? (int)(W0->I / stream_lane_inputs(fmt0)) : 1;
        const int ns = (lpr + 31) / 32;
        stream = stream && kStreamConsumerWarps % ns == 0;
        if (stream) {
            const int ng = fmt0 == 4 ? W0->ng : no_row_scales ? 0 : 1;
            const int G = kStreamConsumerWarps / ns;
            int RG = std::min(4 * G, (int)(kStreamStageBytes / (W0->rs + 4 * ng)));
            if (!no_row_scales) RG = RG / 4 * 4;   // row-scale copies need whole groups of 4 rows
            const int total = job.row_start[n];
            int rpc = (total + ds->n_sm - 1) / ds->n_sm;
            if (!no_row_scales) rpc = (rpc + 3) / 4 * 4;   // CTA row blocks start on whole groups of 4 row scales
            const int grid = (total + rpc - 1) / rpc;
            // chunk -> scale index: fmt=4 groups of gs/32 chunks, FP8 blocks of 8 16-byte chunks
            const int gshift = fmt0 == 4 ? __builtin_ctz(W0->gs / 32) : fmt0 == 7 ? 3 : 30;
            if (RG >= (no_row_scales ? 1 : 4) && (size_t)rpc * ns * 4 <= (size_t)kStreamRedBytes &&
                stream_gemv_smem() <= ds->smem_optin) {
                e = launch_stream_gemv(job, rpc, RG, gshift, grid, st);
                if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
                count(1, wbytes);
                return COLI_OK;
            }
        }
        // S = 2..4 of the same int4 formats: half-chunk lanes keep all S activation rows in registers
        // (measured crossover against the row-pair kernel: S = 2 from ~16 MB of weights, S = 3-4 from ~4 MB)
        bool stream_s = S >= 2 && S <= 4 && !host_any && (W0->fmt == 4 || W0->fmt == 2) && W0->I % 128 == 0 &&
                        ((uintptr_t)x & 15) == 0 && wbytes >= (S == 2 ? (16u << 20) : (4u << 20));
        for (int m = 0; m < n && stream_s; m++)
            stream_s = W0->fmt == 4 ? (W[m]->gs == W0->gs && slab_supported(4, W[m]->gs) && W[m]->ng % 4 == 0)
                                    : W[m]->O % 4 == 0;
        const int nh = (2 * W0->cpr + 31) / 32;
        stream_s = stream_s && kStreamConsumerWarps % nh == 0;
        if (stream_s) {
            const int ng = W0->fmt == 4 ? W0->ng : 1;
            const int RG = (int)(kStreamStageBytes / (W0->rs + 4 * ng)) / 4 * 4;
            const int total = job.row_start[n];
            int rpc = (total + ds->n_sm - 1) / ds->n_sm;
            rpc = (rpc + 3) / 4 * 4;
            const int grid = (total + rpc - 1) / rpc;
            const int gshift = W0->fmt == 4 ? __builtin_ctz(W0->gs / 16) : 30;
            if (RG >= 4 && (size_t)rpc * S * nh * 4 <= (size_t)kStreamGemvRedBytes &&
                stream_gemv_s_smem() <= ds->smem_optin) {
                e = launch_stream_gemv_s(job, rpc, RG, gshift, grid, st);
                if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
                count(1, wbytes);
                return COLI_OK;
            }
        }
        if (slab && slab_gemv_smem(job, ds->n_sm) <= ds->smem_optin) {
            e = launch_slab_gemv(job, ds->n_sm, st);
            nl = 1;
        } else {
            e = launch_gemv(job, st, &nl);
        }
        if (e != cudaSuccess) return cuda_fail(e, "matvec launch");
        count(nl, wbytes);
        return COLI_OK;
    }
    // larger S (or activations too large to stage): tensor-core GEMM for int4
    // formats, tiled CUDA-core GEMM otherwise; one pass per matrix
    for (int m = 0; m < n; m++) {
        if (tc_supported_fmt(W[m]->fmt, W[m]->gs) && W[m]->tmap) {
            const int I = (int)W[m]->I, I_pad = (I + 63) / 64 * 64;
            const int rows_alloc = std::max(S, 64);
            Workspace *ws = nullptr;
            const size_t planes = (size_t)3 * rows_alloc * I_pad * 2;
            if (int rc = workspace(ds, st, planes + 256, &ws)) return rc;
            int *flag = (int *)ws->buf;
            void *pl = (char *)ws->buf + 256;
            CU(cudaMemsetAsync(flag, 0, sizeof(int), st), "cudaMemsetAsync(flag)");
            cudaError_t e = launch_gather_planes(x, I, nullptr, 1, nullptr, S, I, I_pad, pl, (long long)rows_alloc * I_pad,
                                                 flag, st);
            if (e != cudaSuccess) return cuda_fail(e, "activation planes launch");
            PlaneMapSet map;
            e = encode_plane_maps(pl, I_pad, rows_alloc, &map);
            if (e != cudaSuccess) return cuda_fail(e, "activation tensor map");
            TcArgs a;
            memset(&a, 0, sizeof a);
            a.single = desc_of(W[m]);
            a.fmt = W[m]->fmt;
            a.O = (int)W[m]->O;
            a.I = I;
            a.nkb = I_pad / 64;
            a.gkb = W[m]->fmt == 4 ? W[m]->gs / 64 : a.nkb;
            a.n_mblk = (a.O + 127) / 128;
            a.P = S;
            a.rows_alloc = rows_alloc;
            a.nterm_flag = flag;
            a.out = y[m];
            a.ldo = W[m]->O;
            a.err = ds->err;
            a.timeout_ns = 2000000000LL;
            e = launch_gemm_tc(a, map, (S + 63) / 64, ds->n_sm, st);
            if (e != cudaSuccess) return cuda_fail(e, "tensor-core gemm launch");
            count(2, (uint64_t)W[m]->alg_bytes);
            continue;
        }
        GemmArgs a;
        memset(&a, 0, sizeof a);
        a.single = desc_of(W[m]);
        a.fmt = W[m]->fmt;
        a.O = (int)W[m]->O;
        a.I = (int)W[m]->I;
        a.X = x;
        a.ldx = W[m]->I;
        a.kdiv = 1;
        a.P = S;
        a.out = y[m];
        a.ldo = W[m]->O;
        cudaError_t e = launch_gemm_cc(a, false, (S + kGemmBP - 1) / kGemmBP, st);
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
        count(1, (uint64_t)W[m]->alg_bytes);
    }
    return COLI_OK;
}

static int check_ptr(const void *p, const char *name) {
    if (!p) return fail(COLI_EINVAL, "%s is NULL", name);
    if ((uintptr_t)p & 3) return fail(COLI_EINVAL, "%s is not 4-byte aligned", name);
    return COLI_OK;
}

int coli_matmul(const coli_tensor *W, const float *x, float *y, int S, void *stream) {
    g_msg[0] = 0;
    if (int rc = check_tensor(W, "W")) return rc;
    if (int rc = check_ptr(x, "x")) return rc;
    if (int rc = check_ptr(y, "y")) return rc;
    if (S < 1) return fail(COLI_EINVAL, "S must be >= 1 (got %d)", S);
    if (int rc = injected()) return rc;
    return run_matmul(1, &W, x, &y, S, (cudaStream_t)stream);
}

int coli_matmul_multi(int n, const coli_tensor *const *W, const float *x, float *const *y, int S, void *stream) {
    g_msg[0] = 0;
    if (n < 1 || n > GemvJob::MAXM) return fail(COLI_EINVAL, "n must be in 1..%d (got %d)", GemvJob::MAXM, n);
    if (!W || !y) return fail(COLI_EINVAL, "W or y array is NULL");
    for (int m = 0; m < n; m++) {
        if (int rc = check_tensor(W[m], "W[m]")) return rc;
        if (int rc = check_ptr(y[m], "y[m]")) return rc;
        if (W[m]->fmt != W[0]->fmt || W[m]->I != W[0]->I)
            return fail(COLI_EINVAL, "matrix %d differs in format or I from matrix 0", m);
    }
    if (int rc = check_ptr(x, "x")) return rc;
    if (S < 1) return fail(COLI_EINVAL, "S must be >= 1 (got %d)", S);
    if (int rc = injected()) return rc;
    return run_matmul(n, W, x, y, S, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ absorption
static int run_rows(const coli_tensor *W, int64_t o0, int64_t stride, int64_t n_rows, int n_heads, const float *x,
                    float *y, int S, void *stream, bool transposed) {
    g_msg[0] = 0;
    if (int rc = check_tensor(W, "W")) return rc;
    if (int rc = check_ptr(x, "x")) return rc;
    if (int rc = check_ptr(y, "y")) return rc;
    if (S < 1) return fail(COLI_EINVAL, "S must be >= 1 (got %d)", S);
    if (n_heads < 1 || n_rows < 1 || n_rows > (1 << 30) || o0 < 0 || stride < 0)
        return fail(COLI_EINVAL, "need n_heads >= 1, 1 <= n_rows <= 2^30, o0 >= 0, stride >= 0");
    if (o0 + (int64_t)(n_heads - 1) * stride + n_rows > W->O)
        return fail(COLI_EINVAL, "head rows run past the matrix: o0 + (n_heads-1)*stride + n_rows = %lld > O = %lld",
                    (long long)(o0 + (int64_t)(n_heads - 1) * stride + n_rows), (long long)W->O);
    if (int rc = injected()) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    const int fmt = W->fmt;
    const int N = fmt == 0 ? 2 : (fmt == 1 || fmt == 7) ? 8 : fmt == 3 ? 32 : 16;   // elements per 8-byte unit
    const int units = (int)((W->I + N - 1) / N);
    // grid y: 64-row blocks of a head (forward) or 32-unit column blocks (transposed)
    if ((transposed ? (units + 31) / 32 : (n_rows + 63) / 64) > 65535)
        return fail(COLI_EINVAL, "%s: %s too large for one launch",
                    transposed ? "coli_matmul_rows_t" : "coli_matmul_rows", transposed ? "I" : "n_rows");
    if (absorb_smem(fmt, transposed, units, (int)n_rows, S) > (size_t)ds->smem_optin)
        return fail(COLI_EINVAL, "%s: the shared-memory stage (%zu bytes) exceeds the device limit",
                    transposed ? "coli_matmul_rows_t" : "coli_matmul_rows",
                    absorb_smem(fmt, transposed, units, (int)n_rows, S));
    int nl = 0;
    cudaError_t e = launch_absorb(desc_of(W), fmt, (int)W->I, units, o0, stride, (int)n_rows, n_heads, S, x, y,
                                  transposed, (cudaStream_t)stream, &nl);
    if (e != cudaSuccess) return cuda_fail(e, transposed ? "coli_matmul_rows_t" : "coli_matmul_rows");
    count(nl, (uint64_t)n_heads * (uint64_t)n_rows * (uint64_t)W->rs);
    return COLI_OK;
}

int coli_matmul_rows(const coli_tensor *W, int64_t o0, int64_t stride, int64_t n_rows, int n_heads, const float *x,
                     float *y, int S, void *stream) {
    return run_rows(W, o0, stride, n_rows, n_heads, x, y, S, stream, false);
}

int coli_matmul_rows_t(const coli_tensor *W, int64_t o0, int64_t stride, int64_t n_rows, int n_heads, const float *x,
                       float *y, int S, void *stream) {
    return run_rows(W, o0, stride, n_rows, n_heads, x, y, S, stream, true);
}

// ------------------------------------------------------------------ routing
int coli_moe_route(const int32_t *ids, int S, int K, int n_experts, int32_t *offsets, int32_t *order,
                   void *stream) {
    g_msg[0] = 0;
    if (int rc = check_ptr(ids, "ids")) return rc;
    if (int rc = check_ptr(offsets, "offsets")) return rc;
    if (int rc = check_ptr(order, "order")) return rc;
    if (S < 1 || K < 1 || K > 64) return fail(COLI_EINVAL, "need S >= 1 and 1 <= K <= 64 (got S=%d K=%d)", S, K);
    if (n_experts < 1 || n_experts > 8192)
        return fail(COLI_EINVAL, "n_experts must be in 1..8192 (got %d)", n_experts);
    if ((long long)S * K > (1LL << 30)) return fail(COLI_EINVAL, "S*K too large");
    if (int rc = injected()) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    RouteArgs a;
    memset(&a, 0, sizeof a);
    a.ids = ids;
    a.S = S;
    a.K = K;
    a.E = n_experts;
    a.offsets = offsets;
    a.order = order;
    a.err = ds->err;
    a.tile_rows = kGemmBP;
    cudaError_t e = launch_route(a, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "routing launch");
    count(1, 0);
    return COLI_OK;
}

int coli_moe_topk(const float *logits, const float *bias, int S, int n_experts, int K, float top_p, int norm_topk,
                  float routed_scale, int32_t *ids, float *w, void *stream) {
    g_msg[0] = 0;
    if (int rc = check_ptr(logits, "logits")) return rc;
    if (bias && ((uintptr_t)bias & 3)) return fail(COLI_EINVAL, "bias is not 4-byte aligned");
    if (int rc = check_ptr(ids, "ids")) return rc;
    if (int rc = check_ptr(w, "w")) return rc;
    if (n_experts < 1 || n_experts > 16384)
        return fail(COLI_EINVAL, "n_experts must be in 1..16384 (got %d)", n_experts);
    if (S < 1 || K < 1 || K > 64 || K > n_experts)
        return fail(COLI_EINVAL, "need S >= 1 and 1 <= K <= min(64, n_experts) (got S=%d K=%d)", S, K);
    if (!(top_p == top_p) || !(routed_scale == routed_scale))
        return fail(COLI_EINVAL, "top_p and routed_scale must not be NaN");
    if (int rc = injected()) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    if (topk_smem(n_experts) > ds->smem_optin) return fail(COLI_EINVAL, "n_experts too large for one block");
    cudaError_t e = launch_topk(logits, bias, S, n_experts, K, top_p, norm_topk, routed_scale, ids, w,
                                (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "router top-K launch");
    count(1, 0);
    return COLI_OK;
}

int coli_moe_router(const float *x, int S, const coli_tensor *router, const float *bias, int K, float top_p,
                    int norm_topk, float routed_scale, int32_t *ids, float *w, void *stream) {
    g_msg[0] = 0;
    if (int rc = check_tensor(router, "router")) return rc;
    if (int rc = check_ptr(x, "x")) return rc;
    if (router->O > 16384) return fail(COLI_EINVAL, "the router has more than 16384 experts");
    if (S < 1) return fail(COLI_EINVAL, "S must be >= 1 (got %d)", S);
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    // logits go to a scratch buffer of their own (the stream's workspace is used by the matvec)
    float *logits = nullptr;
    if (int rc = router_scratch(ds, st, (size_t)S * router->O * sizeof(float), &logits)) return rc;
    float *ys[1] = {logits};
    const coli_tensor *Ws[1] = {router};
    if (int rc = coli_matmul_multi(1, Ws, x, ys, S, stream)) return rc;
    return coli_moe_topk(logits, bias, S, (int)router->O, K, top_p, norm_topk, routed_scale, ids, w, stream);
}

// ------------------------------------------------------------------ expert block
static int expert_table(DeviceState *ds, const coli_expert *ex, int n, cudaStream_t st, const ExpertDesc **out) {
    uint64_t key = 1469598103934665603ULL ^ (uint64_t)n;
    for (int e = 0; e < n; e++) {
        const coli_tensor *m[3] = {ex[e].gate, ex[e].up, ex[e].down};
        for (int k = 0; k < 3; k++) key = (key ^ m[k]->uid) * 1099511628211ULL;
    }
    std::lock_guard<std::mutex> lk(ds->mu);
    auto it = ds->tables.find(key);
    if (it != ds->tables.end() && it->second.n == n) {
        it->second.last_use = ++ds->tick;
        *out = it->second.d;
        return COLI_OK;
    }
    if (ds->tables.size() >= 16) {   // evict the least recently used table
        auto victim = ds->tables.begin();
        for (auto i = ds->tables.begin(); i != ds->tables.end(); ++i)
            if (i->second.last_use < victim->second.last_use) victim = i;
        CU(cudaDeviceSynchronize(), "cudaDeviceSynchronize(table eviction)");
        cudaFree(victim->second.d);
        ds->tables.erase(victim);
    }
    std::vector<ExpertDesc> h((size_t)n);
    for (int e = 0; e < n; e++) {
        h[e].m[0] = desc_of(ex[e].gate);
        h[e].m[1] = desc_of(ex[e].up);
        h[e].m[2] = desc_of(ex[e].down);
    }
    CachedTable ct;
    ct.n = n;
    ct.last_use = ++ds->tick;
    CU(cudaMalloc(&ct.d, sizeof(ExpertDesc) * (size_t)n), "cudaMalloc(expert table)");
    cudaError_t e = cudaMemcpyAsync(ct.d, h.data(), sizeof(ExpertDesc) * (size_t)n, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaFree(ct.d);
        return cuda_fail(e, "expert table upload");
    }
    ds->tables[key] = ct;
    *out = ct.d;
    return COLI_OK;
}

// What the expert block's dispatch needs to know about an expert table,
// found in one pass over it (coli_moe_block: on every call;
// coli_expert_table_create: once).
struct MoeInfo {
    int n, fmt, device;
    int64_t H, F;
    const coli_tensor *g0, *d0;   // expert 0's gate and down: the shapes and gs of every expert's
    bool host_any;                // some matrix lives in pinned host memory
    bool gs_ok;                   // fmt=4: every gs a multiple of 32
    bool gs_uniform;              // every gate/up gs equals g0's, every down gs d0's
    bool slab_gs;                 // every gs taken by the slab kernels
    bool tc_all;                  // every matrix taken by the tensor-core GEMM, with its TMA map
};

static int moe_info(const coli_expert *experts, int n_experts, MoeInfo *mi) {
    if (!experts) return fail(COLI_EINVAL, "experts is NULL");
    if (n_experts < 1 || n_experts > 8192)
        return fail(COLI_EINVAL, "n_experts must be in 1..8192 (got %d)", n_experts);
    int dev = 0;
    CU(cudaGetDevice(&dev), "cudaGetDevice");
    const coli_tensor *g0 = experts[0].gate, *d0 = experts[0].down;
    if (!g0) return fail(COLI_EINVAL, "experts[0].gate is NULL");
    if (!d0) return fail(COLI_EINVAL, "experts[0].down is NULL");
    const int64_t F = g0->O, H = g0->I;
    const int fmt = g0->fmt;
    if (F > (1 << 30) || H > (1 << 30)) return fail(COLI_EINVAL, "expert dimensions too large");
    MoeInfo r;
    r.n = n_experts;
    r.fmt = fmt;
    r.device = dev;
    r.H = H;
    r.F = F;
    r.g0 = g0;
    r.d0 = d0;
    r.host_any = false;
    r.gs_ok = r.gs_uniform = r.slab_gs = r.tc_all = true;
    const char *nm[3] = {"gate", "up", "down"};
    for (int e = 0; e < n_experts; e++) {
        const coli_tensor *m[3] = {experts[e].gate, experts[e].up, experts[e].down};
        for (int k = 0; k < 3; k++) {
            if (!m[k]) return fail(COLI_EINVAL, "expert %d %s is NULL", e, nm[k]);
            if (m[k]->device != dev)
                return fail(COLI_EDEVICE, "expert %d %s lives on device %d but device %d is current", e, nm[k],
                            m[k]->device, dev);
            if (m[k]->fmt != fmt)
                return fail(COLI_EFMT, "expert %d %s has fmt=%d but expert 0 gate has fmt=%d; one format per "
                                       "expert table is supported", e, nm[k], m[k]->fmt, fmt);
            r.host_any |= m[k]->host != 0;
            r.gs_ok &= fmt != 4 || m[k]->gs % 32 == 0;
            r.gs_uniform &= m[k]->gs == (k == 2 ? d0->gs : g0->gs);
            r.slab_gs &= slab_supported(fmt, m[k]->gs);
            r.tc_all &= tc_supported_fmt(fmt, m[k]->gs) && m[k]->tmap != nullptr;
        }
        if (m[0]->O != F || m[0]->I != H || m[1]->O != F || m[1]->I != H || m[2]->O != H || m[2]->I != F)
            return fail(COLI_EINVAL, "expert %d: gate/up must be [%lld][%lld] and down [%lld][%lld]", e,
                        (long long)F, (long long)H, (long long)H, (long long)F);
    }
    *mi = r;
    return COLI_OK;
}

// The tensor-core decode plan of a table for one K, kept by
// coli_expert_table_create's tables between calls.
struct MdPlanCache {
    int K = -1;
    bool ok = false;
    MdArgs a;
    size_t smem = 0;
};

static int moe_run(const MoeInfo &mi, const ExpertDesc *table, DeviceState *ds, const float *x, int S,
                   const int32_t *ids, const float *w, int K, float *y, cudaStream_t st, MdPlanCache *pc);

int coli_moe_block(const float *x, int S, const coli_expert *experts, int n_experts, const int32_t *ids,
                   const float *w, int K, float *y, void *stream) {
    g_msg[0] = 0;
    if (int rc = check_ptr(x, "x")) return rc;
    if (int rc = check_ptr(y, "y")) return rc;
    if (int rc = check_ptr(ids, "ids")) return rc;
    if (int rc = check_ptr(w, "w")) return rc;
    if (S < 1 || K < 1 || K > 64) return fail(COLI_EINVAL, "need S >= 1 and 1 <= K <= 64 (got S=%d K=%d)", S, K);
    MoeInfo mi;
    if (int rc = moe_info(experts, n_experts, &mi)) return rc;
    if (int rc = injected()) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const ExpertDesc *table = nullptr;
    if (int rc = expert_table(ds, experts, n_experts, st, &table)) return rc;
    return moe_run(mi, table, ds, x, S, ids, w, K, y, st, nullptr);
}

}  // extern "C"

// A table made once by coli_expert_table_create.
struct coli_expert_table {
    MoeInfo mi;
    ExpertDesc *d = nullptr;   // device copy of the descriptors
    std::mutex mu;             // guards pc
    MdPlanCache pc;
};

extern "C" {

int coli_expert_table_create(const coli_expert *experts, int n_experts, coli_expert_table **out) {
    g_msg[0] = 0;
    if (!out) return fail(COLI_EINVAL, "out is NULL");
    *out = nullptr;
    MoeInfo mi;
    if (int rc = moe_info(experts, n_experts, &mi)) return rc;
    std::vector<ExpertDesc> h((size_t)n_experts);
    for (int e = 0; e < n_experts; e++) {
        h[e].m[0] = desc_of(experts[e].gate);
        h[e].m[1] = desc_of(experts[e].up);
        h[e].m[2] = desc_of(experts[e].down);
    }
    coli_expert_table *t = new coli_expert_table();
    t->mi = mi;
    CU(cudaMalloc(&t->d, sizeof(ExpertDesc) * (size_t)n_experts), "cudaMalloc(expert table)");
    const cudaError_t e = cudaMemcpy(t->d, h.data(), sizeof(ExpertDesc) * (size_t)n_experts, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(t->d);
        delete t;
        return cuda_fail(e, "expert table upload");
    }
    *out = t;
    return COLI_OK;
}

void coli_expert_table_free(coli_expert_table *t) {
    if (!t) return;
    cudaFree(t->d);
    delete t;
}

int coli_moe_block_t(const float *x, int S, const coli_expert_table *table, const int32_t *ids, const float *w,
                     int K, float *y, void *stream) {
    g_msg[0] = 0;
    if (int rc = check_ptr(x, "x")) return rc;
    if (int rc = check_ptr(y, "y")) return rc;
    if (int rc = check_ptr(ids, "ids")) return rc;
    if (int rc = check_ptr(w, "w")) return rc;
    if (!table) return fail(COLI_EINVAL, "table is NULL");
    if (S < 1 || K < 1 || K > 64) return fail(COLI_EINVAL, "need S >= 1 and 1 <= K <= 64 (got S=%d K=%d)", S, K);
    int dev = 0;
    CU(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != table->mi.device)
        return fail(COLI_EDEVICE, "the table lives on device %d but device %d is current", table->mi.device, dev);
    if (int rc = injected()) return rc;
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    coli_expert_table *t = const_cast<coli_expert_table *>(table);
    std::lock_guard<std::mutex> lk(t->mu);
    return moe_run(t->mi, t->d, ds, x, S, ids, w, K, y, (cudaStream_t)stream, &t->pc);
}

static int moe_run(const MoeInfo &mi, const ExpertDesc *table, DeviceState *ds, const float *x, int S,
                   const int32_t *ids, const float *w, int K, float *y, cudaStream_t st, MdPlanCache *pc) {
    const int n_experts = mi.n, fmt = mi.fmt;
    const int64_t H = mi.H, F = mi.F;
    const coli_tensor *g0 = mi.g0;
    const int n_slots = S * K;
    const int cpr_gu = g0->cpr, cpr_d = mi.d0->cpr;
    const bool gs_ok = mi.gs_ok, host_any = mi.host_any;

    // ---------------- decode, S = 1, int4 tables (gs a power-of-two multiple of 64): weights streamed by
    // bulk copies, dot products on the tensor cores, one cooperative launch
    if (S == 1 && (fmt == 2 || fmt == 4) && n_slots <= kMaxDecodeSlots && !host_any) {
        const coli_tensor *d0 = mi.d0;
        const int gs_gu = g0->gs, gs_d = d0->gs;
        MdArgs a;
        size_t smem = 0;
        bool planned;
        if (pc && pc->K == K) {   // the table's plan for this K
            planned = pc->ok;
            a = pc->a;
            smem = pc->smem;
        } else {
            int per_sm = 0;
            planned = (fmt == 2 || mi.gs_uniform) &&
                      md_plan(fmt, (int)H, (int)F, K, (int)g0->rs, (int)d0->rs, g0->ng, d0->ng, gs_gu, gs_d, ds->n_sm,
                              (size_t)ds->smem_optin, &a, &smem) &&
                      md_occupancy(a, smem, &per_sm) == cudaSuccess && per_sm >= 1;
            if (pc) {
                pc->K = K;
                pc->ok = planned;
                pc->a = a;
                pc->smem = smem;
            }
        }
        if (planned) {
            unsigned *ctr = nullptr;
            if (int rc = decode_counters(ds, st, md_counter_words(a), &ctr)) return rc;
            a.x = x;
            a.ids = ids;
            a.w = w;
            a.y = y;
            a.table = table;
            a.n_experts = n_experts;
            a.ctr = ctr;
            a.err = ds->err;
            a.timeout_ns = 2000000000LL;
            cudaError_t e = launch_decode_mma(a, ds->n_sm, smem, st);
            if (e != cudaSuccess) return cuda_fail(e, "decode expert-block launch");
            count(1, 0);
            return COLI_OK;
        }
    }

    // ---------------- decode, S = 1, int4 / int8 tables: weights streamed by bulk copies, dp4a decode,
    // one cooperative launch
    if (S == 1 && (fmt == 1 || fmt == 2 || fmt == 4) && n_slots <= kMaxDecodeSlots && !host_any) {
        const coli_tensor *d0 = mi.d0;
        const int gs_gu = g0->gs, gs_d = d0->gs;
        // one gs per role, a power-of-two number of 16-byte chunks per group
        const bool ok = fmt != 4 || (slab_supported(4, gs_gu) && slab_supported(4, gs_d) && mi.gs_uniform);
        SdArgs a;
        size_t smem = 0;
        int per_sm = 0;
        if (ok && sd_plan(fmt, (int)H, (int)F, K, cpr_gu, cpr_d, (int)g0->rs, (int)d0->rs, g0->ng, d0->ng, ds->n_sm,
                          (size_t)ds->smem_optin, &a, &smem) &&
            sd_occupancy(a, smem, &per_sm) == cudaSuccess && per_sm >= 1) {
            Workspace *ws = nullptr;
            if (int rc = workspace(ds, st, sd_scratch_bytes(a), &ws)) return rc;
            unsigned *ctr = nullptr;
            if (int rc = decode_counters(ds, st, sd_counter_words(a), &ctr)) return rc;
            a.x = x;
            a.ids = ids;
            a.w = w;
            a.y = y;
            a.table = table;
            a.n_experts = n_experts;
            a.gshift_gu = fmt == 4 ? __builtin_ctz(gs_gu / 32) : 0;
            a.gshift_d = fmt == 4 ? __builtin_ctz(gs_d / 32) : 0;
            a.hbuf = (float *)ws->buf;
            a.ctr = ctr;
            a.err = ds->err;
            a.timeout_ns = 2000000000LL;
            cudaError_t e = launch_stream_decode(a, ds->n_sm, smem, st);
            if (e != cudaSuccess) return cuda_fail(e, "decode expert-block launch");
            count(1, 0);
            return COLI_OK;
        }
    }

    // ---------------- decode, S = 1: activation slab in registers, one cooperative launch
    const bool slab_ok = S == 1 && n_slots <= kMaxDecodeSlots && fmt != 3 && F % 32 == 0 && mi.slab_gs && mi.gs_uniform;
    if (slab_ok) {
        const int grid_min = ds->n_sm;
        int sb = std::min(n_slots, 8);
        size_t smem = slab_decode_smem(fmt, cpr_gu, cpr_d, (int)F, n_slots, grid_min, (int)H, sb);
        while (sb > 1 && smem > 110 * 1024) {
            sb--;
            smem = slab_decode_smem(fmt, cpr_gu, cpr_d, (int)F, n_slots, grid_min, (int)H, sb);
        }
        int per_sm = 0;
        if (smem <= ds->smem_optin && slab_decode_occupancy(fmt, smem, &per_sm) == cudaSuccess && per_sm >= 1) {
            Workspace *ws = nullptr;
            if (int rc = workspace(ds, st, (size_t)n_slots * F * sizeof(float), &ws)) return rc;
            const int grid = std::min(per_sm, 2) * ds->n_sm;
            MoeDecodeArgs a;
            memset(&a, 0, sizeof a);
            a.x = x;
            a.ids = ids;
            a.w = w;
            a.y = y;
            a.table = table;
            a.n_experts = n_experts;
            a.S = 1;
            a.K = K;
            a.H = (int)H;
            a.F = (int)F;
            a.cpr_gu = cpr_gu;
            a.cpr_d = cpr_d;
            a.hbuf = (float *)ws->buf;
            a.bar = ws->bar;
            a.err = ds->err;
            a.sb = sb;
            a.rpc = (int)((H + grid - 1) / grid);
            a.timeout_ns = 2000000000LL;
            cudaError_t e = launch_slab_decode(a, fmt, grid, smem, fmt == 4 ? g0->gs : 32,
                                               fmt == 4 ? mi.d0->gs : 32, st);
            if (e != cudaSuccess) return cuda_fail(e, "decode expert-block launch");
            count(1, 0);
            return COLI_OK;
        }
    }

    // ---------------- decode: one cooperative launch
    if (n_slots <= kMaxDecodeSlots && gs_ok) {
        const int xlen_gu = staged_len(fmt, cpr_gu), xlen_d = staged_len(fmt, cpr_d);
        const size_t budget = 110 * 1024 / 4;   // floats per CTA: two CTAs per SM
        const int rpc_alloc = (int)((H + ds->n_sm - 1) / ds->n_sm);
        const size_t fixed = (size_t)S * rpc_alloc;
        int sb = 0;
        if (budget > fixed + xlen_d + rpc_alloc)
            sb = (int)std::min<size_t>((size_t)n_slots, (budget - fixed) / (size_t)(xlen_d + rpc_alloc));
        const size_t stage = std::max((size_t)S * xlen_gu, (size_t)sb * xlen_d);
        const size_t smem = (stage + (size_t)sb * rpc_alloc + fixed) * sizeof(float);
        if (sb >= 1 && (size_t)S * xlen_gu <= budget && smem <= ds->smem_optin) {
            int per_sm = 0;
            cudaError_t e = moe_decode_occupancy(fmt, smem, &per_sm);
            if (e != cudaSuccess) return cuda_fail(e, "decode occupancy");
            if (per_sm >= 1) {
                Workspace *ws = nullptr;
                if (int rc = workspace(ds, st, (size_t)n_slots * F * sizeof(float), &ws)) return rc;
                const int grid = per_sm * ds->n_sm;
                MoeDecodeArgs a;
                memset(&a, 0, sizeof a);
                a.x = x;
                a.ids = ids;
                a.w = w;
                a.y = y;
                a.table = table;
                a.n_experts = n_experts;
                a.S = S;
                a.K = K;
                a.H = (int)H;
                a.F = (int)F;
                a.cpr_gu = cpr_gu;
                a.cpr_d = cpr_d;
                a.hbuf = (float *)ws->buf;
                a.bar = ws->bar;
                a.err = ds->err;
                a.sb = sb;
                a.rpc = (int)((H + grid - 1) / grid);
                a.timeout_ns = 2000000000LL;
                e = launch_moe_decode(a, fmt, grid, smem, st);
                if (e != cudaSuccess) return cuda_fail(e, "decode expert-block launch");
                count(1, 0);
                return COLI_OK;
            }
        }
    }

    // ---------------- prefill on the tensor cores (int4 formats with one gs per role)
    const bool tc_ok = (fmt == 2 || fmt == 4) && mi.tc_all && mi.gs_uniform;
    if (tc_ok) {
        const int TR = tc_block_rows();
        const int max_tiles = (n_slots + TR - 1) / TR + std::min(n_experts, n_slots);
        const int H_pad = (int)((H + 63) / 64 * 64), F_pad = (int)((F + 63) / 64 * 64);
        const int rows_alloc = std::max(n_slots, 64);
        auto al = [](size_t b) { return (b + 255) / 256 * 256; };
        const size_t sz_off = al((size_t)(n_experts + 1) * 4), sz_ord = al((size_t)n_slots * 4);
        const size_t sz_tile = al((size_t)max_tiles * 4);
        const size_t sz_px = al((size_t)3 * rows_alloc * H_pad * 2), sz_gu = al((size_t)n_slots * 2 * F * 4);
        const size_t sz_ph = al((size_t)3 * rows_alloc * F_pad * 2), sz_out = al((size_t)n_slots * H * 4);
        // experts with at most kSmallRows rows: groups of up to 4 rows on the mma.sync path (moe_small.cu)
        constexpr int kSmallRows = 12;
        SmArgs sgu, sdn;
        size_t smem_gu = 0, smem_dn = 0;
        const bool small = sm_plan(false, fmt, g0->gs, (int)H, (int)F, (int)g0->rs, g0->ng, (size_t)ds->smem_optin,
                                   &sgu, &smem_gu) &&
                           sm_plan(true, fmt, mi.d0->gs, (int)F, (int)H, (int)mi.d0->rs, mi.d0->ng,
                                   (size_t)ds->smem_optin, &sdn, &smem_dn);
        const size_t sz_sg = al((size_t)n_slots * 4);
        const size_t total =
            sz_off + 2 * sz_ord + 3 * sz_tile + 256 + sz_px + sz_gu + sz_ph + sz_out + 3 * sz_sg + al(n_slots);
        Workspace *ws = nullptr;
        if (int rc = workspace(ds, st, total, &ws)) return rc;
        char *p = (char *)ws->buf;
        int32_t *offsets = (int32_t *)p; p += sz_off;
        int32_t *order = (int32_t *)p; p += sz_ord;
        int32_t *inv = (int32_t *)p; p += sz_ord;
        int32_t *te = (int32_t *)p; p += sz_tile;
        int32_t *tp0 = (int32_t *)p; p += sz_tile;
        int32_t *tp1 = (int32_t *)p; p += sz_tile;
        int32_t *ntiles = (int32_t *)p;
        int *flags = (int *)(p + 64);
        p += 256;
        void *px = p; p += sz_px;
        float *gu = (float *)p; p += sz_gu;
        void *ph = p; p += sz_ph;
        float *slot_out = (float *)p; p += sz_out;
        int32_t *sg_e = (int32_t *)p; p += sz_sg;
        int32_t *sg_p0 = (int32_t *)p; p += sz_sg;
        int32_t *sg_n = (int32_t *)p; p += sz_sg;
        uint8_t *row_small = (uint8_t *)p;
        int32_t *n_sg = flags + 4;   // the small-group count, beside the plane flags (one zeroed block)
        CU(cudaMemsetAsync(flags, 0, 8 * sizeof(int), st), "cudaMemsetAsync(flags)");

        RouteArgs r;
        memset(&r, 0, sizeof r);
        r.ids = ids; r.S = S; r.K = K; r.E = n_experts;
        r.offsets = offsets; r.order = order; r.inv = inv;
        r.tile_e = te; r.tile_p0 = tp0; r.tile_p1 = tp1; r.n_tiles = ntiles;
        r.tile_rows = TR;
        r.small_rows = small ? kSmallRows : 0;
        r.sg_e = sg_e; r.sg_p0 = sg_p0; r.sg_n = sg_n; r.n_sg = n_sg;
        r.row_small = small ? row_small : nullptr;
        r.err = ds->err;
        cudaError_t e = launch_route(r, st);
        if (e != cudaSuccess) return cuda_fail(e, "routing launch");
        int n_launch = 6;
        if (small) {
            for (SmArgs *sa : {&sgu, &sdn}) {
                sa->table = table;
                sa->sg_e = sg_e; sa->sg_p0 = sg_p0; sa->sg_n = sg_n; sa->n_sg = n_sg;
                sa->err = ds->err;
            }
            sgu.x = x; sgu.ldx = H; sgu.order = order; sgu.K = K;
            sgu.out = gu; sgu.ldo = 2 * F;
            sdn.gu = gu;
            sdn.out = slot_out; sdn.ldo = H;
            e = launch_moe_small(sgu, ds->n_sm, smem_gu, st);
            if (e != cudaSuccess) return cuda_fail(e, "small-expert gate/up launch");
            n_launch++;
        }
        e = launch_gather_planes(x, H, order, K, offsets + n_experts, n_slots, (int)H, H_pad, px,
                                 (long long)rows_alloc * H_pad, &flags[0], st, small ? row_small : nullptr);
        if (e != cudaSuccess) return cuda_fail(e, "activation planes launch");
        PlaneMapSet mapx, maph;
        e = encode_plane_maps(px, H_pad, rows_alloc, &mapx);
        if (e != cudaSuccess) return cuda_fail(e, "activation tensor map");
        TcArgs a;
        memset(&a, 0, sizeof a);
        a.table = table;
        a.mi = 0;
        a.dual_mb = (int)((F + 127) / 128);
        a.fmt = fmt;
        a.O = (int)F;
        a.I = (int)H;
        a.nkb = H_pad / 64;
        a.gkb = fmt == 4 ? g0->gs / 64 : a.nkb;
        a.n_mblk = 2 * a.dual_mb;
        a.tile_e = te; a.tile_p0 = tp0; a.tile_p1 = tp1; a.n_tiles = ntiles;
        a.rows_alloc = rows_alloc;
        a.nterm_flag = &flags[0];
        a.out = gu;
        a.ldo = 2 * F;
        a.err = ds->err;
        a.timeout_ns = 2000000000LL;
        e = launch_gemm_tc(a, mapx, max_tiles, ds->n_sm, st);
        if (e != cudaSuccess) return cuda_fail(e, "gate/up tensor-core launch");
        e = launch_silu_planes(gu, (int)F, offsets + n_experts, n_slots, F_pad, ph, (long long)rows_alloc * F_pad,
                               &flags[1], st, small ? row_small : nullptr);
        if (e != cudaSuccess) return cuda_fail(e, "silu planes launch");
        e = encode_plane_maps(ph, F_pad, rows_alloc, &maph);
        if (e != cudaSuccess) return cuda_fail(e, "hidden tensor map");
        TcArgs d = a;
        d.mi = 2;
        d.dual_mb = 0;
        d.O = (int)H;
        d.I = (int)F;
        d.nkb = F_pad / 64;
        d.gkb = fmt == 4 ? mi.d0->gs / 64 : d.nkb;
        d.n_mblk = (int)((H + 127) / 128);
        d.nterm_flag = &flags[1];
        d.out = slot_out;
        d.ldo = H;
        e = launch_gemm_tc(d, maph, max_tiles, ds->n_sm, st);
        if (e != cudaSuccess) return cuda_fail(e, "down tensor-core launch");
        if (small) {
            e = launch_moe_small(sdn, ds->n_sm, smem_dn, st);
            if (e != cudaSuccess) return cuda_fail(e, "small-expert down launch");
            n_launch++;
        }
        e = launch_combine(slot_out, inv, w, S, K, (int)H, y, st);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
        count(n_launch, 0);
        return COLI_OK;
    }

    // ---------------- prefill pipeline on the CUDA cores (other formats / group sizes)
    const int max_tiles = (n_slots + kGemmBP - 1) / kGemmBP + std::min(n_experts, n_slots);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t sz_off = al((size_t)(n_experts + 1) * 4), sz_ord = al((size_t)n_slots * 4);
    const size_t sz_tile = al((size_t)max_tiles * 4), sz_h = al((size_t)n_slots * F * 4);
    const size_t sz_out = al((size_t)n_slots * H * 4);
    const size_t total = sz_off + 2 * sz_ord + 3 * sz_tile + 256 + sz_h + sz_out;
    Workspace *ws = nullptr;
    if (int rc = workspace(ds, st, total, &ws)) return rc;
    char *p = (char *)ws->buf;
    int32_t *offsets = (int32_t *)p; p += sz_off;
    int32_t *order = (int32_t *)p; p += sz_ord;
    int32_t *inv = (int32_t *)p; p += sz_ord;
    int32_t *te = (int32_t *)p; p += sz_tile;
    int32_t *tp0 = (int32_t *)p; p += sz_tile;
    int32_t *tp1 = (int32_t *)p; p += sz_tile;
    int32_t *ntiles = (int32_t *)p; p += 256;
    float *hbuf = (float *)p; p += sz_h;
    float *slot_out = (float *)p;

    RouteArgs r;
    memset(&r, 0, sizeof r);
    r.ids = ids;
    r.S = S;
    r.K = K;
    r.E = n_experts;
    r.offsets = offsets;
    r.order = order;
    r.inv = inv;
    r.tile_e = te;
    r.tile_p0 = tp0;
    r.tile_p1 = tp1;
    r.n_tiles = ntiles;
    r.tile_rows = kGemmBP;
    r.err = ds->err;
    cudaError_t e = launch_route(r, st);
    if (e != cudaSuccess) return cuda_fail(e, "routing launch");

    GemmArgs gu;
    memset(&gu, 0, sizeof gu);
    gu.table = table;
    gu.mi = 0;
    gu.fmt = fmt;
    gu.O = (int)F;
    gu.I = (int)H;
    gu.X = x;
    gu.ldx = H;
    gu.order = order;
    gu.kdiv = K;
    gu.tile_e = te;
    gu.tile_p0 = tp0;
    gu.tile_p1 = tp1;
    gu.n_tiles = ntiles;
    gu.out = hbuf;
    gu.ldo = F;
    e = launch_gemm_cc(gu, true, max_tiles, st);
    if (e != cudaSuccess) return cuda_fail(e, "gate/up launch");

    GemmArgs dn = gu;
    dn.mi = 2;
    dn.O = (int)H;
    dn.I = (int)F;
    dn.X = hbuf;
    dn.ldx = F;
    dn.order = nullptr;
    dn.kdiv = 1;
    dn.out = slot_out;
    dn.ldo = H;
    e = launch_gemm_cc(dn, false, max_tiles, st);
    if (e != cudaSuccess) return cuda_fail(e, "down launch");

    e = launch_combine(slot_out, inv, w, S, K, (int)H, y, st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    count(4, 0);
    return COLI_OK;
}

int coli_sync_check(void *stream) {
    g_msg[0] = 0;
    cudaStream_t st = (cudaStream_t)stream;
    CU(cudaStreamSynchronize(st), "cudaStreamSynchronize");
    DeviceState *ds = nullptr;
    if (int rc = device_state(&ds)) return rc;
    int word = 0;
    CU(cudaMemcpy(&word, ds->err, sizeof(int), cudaMemcpyDeviceToHost), "reading the device error word");
    if (word == DEV_ERR_NONE) return COLI_OK;
    CU(cudaMemset(ds->err, 0, sizeof(int)), "clearing the device error word");
    if (word == DEV_ERR_TIMEOUT) {
        std::lock_guard<std::mutex> lk(ds->mu);
        for (auto &kv : ds->ws)
            if (kv.second.bar) cudaMemset(kv.second.bar, 0, kBarrierBytes);
        return fail(COLI_ETIMEOUT, "a grid-wide wait in the expert block ran out of time");
    }
    if (word == DEV_ERR_BAD_ID) return fail(COLI_EINVAL, "a routing id was outside [-1, n_experts)");
    return fail(COLI_ECUDA, "device error word %d", word);
}

}  // extern "C"
