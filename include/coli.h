/*
 * coli.h -- C ABI of the GB300 (sm_103a) quantized-weight matvec / routed-expert
 * library.  Plain pointers and sizes only; no C++ or framework types.
 *
 * The operation (colibri project pages):
 *   - y[s][o] = sum_i w[o][i] * x[s][i] over a quantized weight matrix W [O][I]
 *     in one of seven formats (PR #298 page, commit message "metal: grouped-int4
 *     (fmt=4) GEMV support": mm_gemv handled "fmt 0-3", fmt=4 added with one f32
 *     scale per gs inputs folded into the accumulation per group; commit message
 *     "CUDA backend had no fmt=4 case": per-row scale for fmt 1/2/3, per-group
 *     for fmt=4, O*ceil(I/gs) scales).
 *   - the routed-expert block: per routed (row, expert) pair, gate/up matvecs,
 *     silu(gate)*up, the down matvec, and a weighted scatter-add of the expert
 *     outputs over ragged per-row routing (colibri-strix commit log, "metal:
 *     batched moe_block": "gate/up/silu/down for a whole expert block",
 *     "per-row ragged expert routing", "weighted scatter-add").
 *
 * Host byte layout accepted by coli_tensor_upload (rows contiguous, each row
 * starting on a byte boundary):
 *   fmt=0  f32 [O][I], no scales.
 *   fmt=1  int8 two's complement [O][I]; scales f32 [O].
 *   fmt=2  int4 offset binary, value = nibble - 8; rows of ceil(I/2) bytes;
 *          element 2j is the LOW nibble of byte j; scales f32 [O].
 *   fmt=3  int2 offset binary, value = crumb - 2; rows of ceil(I/4) bytes
 *          (PR #298 page, qt_addrow commit message: stride (I+3)/4); element
 *          4j+t is bits [2t, 2t+1] of byte j; scales f32 [O].
 *   fmt=4  int4 as fmt=2; scales f32 [O][ceil(I/gs)], group g covering inputs
 *          [g*gs, min((g+1)*gs, I)) (PR #298 page, test_i4_grouped commit: the
 *          partial last group and gs > I).
 *   fmt=5  int3 offset binary, value = code - 4; rows of 3*ceil(I/8) bytes;
 *          element 8j+t is bits [3t, 3t+2] of the little-endian 24-bit word in
 *          bytes 3j..3j+2; scales f32 [O][ceil(I/gs)] as for fmt=4, gs a
 *          multiple of 8 (PR #298 page: "int3 fmt=5" in the #377 retarget
 *          list; the Vulkan fmt=4 commit message skips the per-row scale "like
 *          fmt=5"; the bit layout is this library's reading, the pages print
 *          none).  The device copy holds each code c as the int4 nibble c + 4
 *          (the same value c - 4) with the same scales, so every int4 kernel
 *          serves int3; it is 4/3 of the int3 bytes.
 *   fmt=7  FP8 E4M3 (OCP: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *          exponent 0 subnormal, no infinities, S.1111.111 NaN), one byte per
 *          element, [O][I]; scales f32 [ceil(O/128)][ceil(I/128)], one per
 *          128 x 128 block, w[o][i] = e4m3(byte) * s[o/128][i/128] (PR #298
 *          page, qt_addrow / qt_matvec_rows commit message: fmt=7 keeps raw
 *          bytes like fmt=1 and ceil(O/128)*ceil(I/128) per-block scales; the
 *          E4M3 encoding is this library's reading of its "fp8 passthrough").
 * The int4 offset encoding and the extremes 0x00 -> -8, 0xFF -> +7 are printed
 * on the PR #298 page (test_i4_grouped commit message); the element order in a
 * byte, the int2, int3 and int8 encodings are this library's documented readings.
 *
 * Conventions for every entry point:
 *   - Return 0 (COLI_OK) or a negative COLI_E* code; coli_last_error() then
 *     gives a message for the calling thread.  No entry point ever falls back
 *     to another implementation or returns a partial result: an argument it
 *     cannot handle is refused with an error, before anything is launched.
 *   - "device" pointers are CUDA global-memory pointers on the current device;
 *     "host" pointers are ordinary host memory.  The caller owns every pointer
 *     it passes and the stream.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).
 *   - Compute calls are asynchronous on `stream`.  Their return code covers
 *     argument checks and launch errors.  Errors found on the device (a bounded
 *     wait that ran out) are reported by the next coli_sync_check(stream).
 *   - Each device has its own library state; tensors live on the device that
 *     was current at upload and must be used with that device current.
 */
#ifndef COLI_H
#define COLI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    COLI_OK = 0,
    COLI_EINVAL = -1,     /* bad size, pointer, stride or combination of arguments */
    COLI_EFMT = -2,       /* unknown format or invalid group size */
    COLI_ENOMEM = -3,     /* device allocation failed */
    COLI_ECUDA = -4,      /* a CUDA runtime call failed (message names it) */
    COLI_ETIMEOUT = -5,   /* a bounded device-side wait ran out (from coli_sync_check) */
    COLI_EINJECTED = -6,  /* failure injected by coli_set_fail_after / COLI_FAIL_AFTER */
    COLI_EDEVICE = -7     /* tensor used on a device other than the one it lives on */
};

/* Opaque uploaded weight matrix.  The library owns its device memory. */
typedef struct coli_tensor coli_tensor;

/* One routed expert: gate [F][H], up [F][H], down [H][F]. */
typedef struct {
    const coli_tensor *gate, *up, *down;
} coli_expert;

/* Library-wide counters (all threads, all devices). */
typedef struct {
    uint64_t calls;        /* compute entry points that launched work */
    uint64_t launches;     /* CUDA kernels launched by this library */
    uint64_t weight_bytes; /* algorithmic weight bytes (codes + scales) of launched work */
} coli_stats;

/*
 * Upload one weight matrix W [O][I] (PR #298 page, "CUDA backend had no fmt=4
 * case" commit message: coli_cuda_tensor_upload_grouped takes gs and stores
 * O*ceil(I/gs) scales; this entry point is that upload for every format).
 *   fmt     0..5 or 7 as in the layout above.
 *   gs      fmt=4: group size, even and >= 2 (gs >= I means one group per row).
 *           fmt=5: group size, a multiple of 8.
 *           Other formats: ignored (fmt=7 blocks are always 128 x 128).
 *   O, I    rows (outputs) and columns (inputs), each >= 1, I <= 2^30.
 *   data    HOST pointer to the packed codes in the host layout above.
 *   scales  HOST pointer to the f32 scales (NULL for fmt=0).
 *   stream  stream for the copies; the call returns after they completed, so
 *           data and scales may be freed or reused right away.
 *   out     receives the new tensor; on error *out is set to NULL.
 * The device copy is re-laid out for the kernels (rows padded to 16 bytes,
 * int8 stored offset binary); the padding never contributes to a result.
 * Errors: COLI_EFMT (fmt or gs), COLI_EINVAL (sizes, NULL data/scales/out),
 * COLI_ENOMEM, COLI_ECUDA.
 */
int coli_tensor_upload(int fmt, int gs, int64_t O, int64_t I, const void *data,
                       const float *scales, void *stream, coli_tensor **out);

/*
 * Upload one weight matrix that STAYS IN HOST MEMORY (colibri-strix commit log:
 * "metal: backend infrastructure" and "metal: batched moe_block + zero-copy
 * slab registry" read expert slabs zero-copy from unified memory; "metal:
 * overlap disk loads with GPU compute" computes resident experts while the
 * others arrive).  The codes and scales are written, in the same padded layout
 * the device copy uses, into pinned host memory mapped into the GPU's address
 * space; the kernels read them over the CPU-GPU link (NVLink-C2C on Grace)
 * every call, with plain loads, while device-resident matrices of the same
 * call stream from HBM.
 *   Arguments, layout and errors as coli_tensor_upload (no stream: nothing is
 *   queued on the GPU).  data and scales may be freed when the call returns.
 *   The tensor is used exactly like a device one (coli_matmul, expert tables,
 *   mixed with device tensors); calls that touch one avoid the bulk-copy
 *   kernels.  coli_tensor_info reports device_bytes = 0.
 */
int coli_tensor_upload_host(int fmt, int gs, int64_t O, int64_t I, const void *data,
                            const float *scales, coli_tensor **out);

/* Free a tensor (NULL is ignored).  The caller must make sure no queued work
 * still reads it (synchronize the streams that used it first). */
void coli_tensor_free(coli_tensor *t);

/* Shape and storage of a tensor.  Any output pointer may be NULL.
 * fmt is the format as uploaded; device_bytes = device memory held; alg_bytes =
 * host-layout codes + scales. */
int coli_tensor_info(const coli_tensor *t, int *fmt, int *gs, int64_t *O, int64_t *I,
                     int64_t *device_bytes, int64_t *alg_bytes);

/*
 * y[S][O] = x[S][I] * W^T   (the quantized matvec for S = 1, the small-S
 * matmul for S > 1; PR #298 page, "metal: grouped-int4 (fmt=4) GEMV support"
 * commit message, Shader paragraph).
 *   W       uploaded tensor.
 *   x       device f32 [S][I], row-major, 4-byte aligned (16-byte alignment
 *           lets the kernels use vector loads).
 *   y       device f32 [S][O], row-major, overwritten; must not overlap x.
 *   S       rows, >= 1.  S <= 8 (with the activations fitting shared memory)
 *           runs the bandwidth-bound CUDA-core matvec kernels, S = 1 the
 *           slab kernel for fmt 0/1/2/4; larger S runs the tensor-core GEMM
 *           for fmt=2 and for fmt=4 with gs % 64 == 0, the tiled CUDA-core
 *           GEMM otherwise (fmt 0, 1, 3, 7); fmt=5 runs the int4 kernels.
 * Errors: COLI_EINVAL (NULL/misaligned pointer, S < 1), COLI_EDEVICE, COLI_ECUDA.
 */
int coli_matmul(const coli_tensor *W, const float *x, float *y, int S, void *stream);

/*
 * y_m = x * W_m^T for m < n, several matrices that share one input x (e.g. the
 * attention projections that read the same activations, or a layer's set of
 * expert matrices), as ONE launch.
 *   n       1..16 matrices; all have the same fmt and I (O and gs may differ).
 *   W       HOST array of n tensor pointers.
 *   x       device f32 [S][I].
 *   y       HOST array of n device pointers, y[m] is f32 [S][O_m], overwritten.
 *   S       1..16.
 * Errors as coli_matmul, plus COLI_EINVAL when formats or I differ.
 */
int coli_matmul_multi(int n, const coli_tensor *const *W, const float *x, float *const *y, int S,
                      void *stream);

/*
 * The two quantized products of the kv_b MLA-absorption path, batched over
 * attention heads (PR #298 page, commit message on qt_addrow / qt_matvec_rows:
 * a matvec over a range of rows of one quantized matrix, and the accumulation
 * of coefficient times dequantized row).  Head h owns rows
 * o0 + h*stride + j, j < n_rows, of W [O][I]:
 *   coli_matmul_rows    y[s][h][j] = sum_i W[o0 + h*stride + j][i] * x[s][h][i]
 *                       x: device f32 [S][n_heads][I]; y: [S][n_heads][n_rows]
 *   coli_matmul_rows_t  y[s][h][i] = sum_j x[s][h][j] * W[o0 + h*stride + j][i]
 *                       x: device f32 [S][n_heads][n_rows]; y: [S][n_heads][I]
 *   W       any format (device or host resident); y overwritten, must not overlap x.
 *   o0, stride, n_rows, n_heads  o0 >= 0, stride >= 0 (heads may share rows),
 *           1 <= n_rows <= 2^30, n_heads >= 1, o0 + (n_heads-1)*stride + n_rows <= O.
 *   S       rows of activations, >= 1 (each weight row is read once per 4 of them).
 * Errors: COLI_EINVAL (pointers, ranges, a head's activations too long for the
 * shared-memory stage), COLI_EDEVICE, COLI_ECUDA.
 */
int coli_matmul_rows(const coli_tensor *W, int64_t o0, int64_t stride, int64_t n_rows, int n_heads,
                     const float *x, float *y, int S, void *stream);
int coli_matmul_rows_t(const coli_tensor *W, int64_t o0, int64_t stride, int64_t n_rows, int n_heads,
                       const float *x, float *y, int S, void *stream);

/*
 * Routing inversion: a stable counting sort of the slots (s, k), s < S, k < K,
 * by expert id ids[s*K+k] (colibri-strix commit log, "metal: batched
 * moe_block": per-row ragged routing; id -1 is an empty slot).
 *   ids      device int32 [S][K], each in [-1, n_experts).
 *   offsets  device int32 [n_experts+1]: expert e's slots are
 *            order[offsets[e] .. offsets[e+1]); offsets[n_experts] = valid slots.
 *   order    device int32 [S*K]: slot indices s*K+k, grouped by expert, each
 *            group in ascending slot order (deterministic).
 *   S >= 1, 1 <= K <= 64, 1 <= n_experts <= 65536.
 * An id out of range makes the kernel record COLI_EINVAL for the next
 * coli_sync_check(stream) and leaves offsets/order unspecified.
 */
int coli_moe_route(const int32_t *ids, int S, int K, int n_experts, int32_t *offsets, int32_t *order,
                   void *stream);

/*
 * Router top-K: the routing coli_moe_block consumes, computed on the device
 * (colibri-strix commit log, "metal: full decode layer in ONE command buffer":
 * sigmoid of the router logits, exact greedy top-K over sigmoid + bias with the
 * CPU tie order, --topp truncation, norm_topk, routed_scale).  Per row s:
 *   score_e = sigmoid(logits[s][e])        (double, rounded to f32)
 *   key_e   = score_e + bias[e]            (f32; bias NULL means 0)
 *   K rounds pick the largest remaining key, ties to the lower id;
 *   ids[s][k] = the k-th pick, w[s][k] = its score (the bias only steers).
 *   top_p in (0, 1): keep the leading picks while the f32 running sum of the
 *   scores before each is below top_p * (f32 sum of the K scores); the rest
 *   become empty slots (id -1, weight 0).  top_p <= 0 or >= 1 keeps all K.
 *   norm_topk != 0: divide the kept weights by their f32 sum.
 *   Then multiply the kept weights by routed_scale.
 * Every decision and weight is the f32 value of these steps (one rounding per
 * operation), so the result is the same on every run.
 *   logits   device f32 [S][n_experts] (finite values).
 *   bias     device f32 [n_experts] or NULL.
 *   ids, w   device int32 / f32 [S][K], overwritten.
 *   S >= 1, 1 <= n_experts <= 16384, 1 <= K <= min(64, n_experts).
 * Errors: COLI_EINVAL (NULL/misaligned pointer, sizes, NaN top_p or
 * routed_scale), COLI_EDEVICE, COLI_ECUDA.
 */
int coli_moe_topk(const float *logits, const float *bias, int S, int n_experts, int K, float top_p,
                  int norm_topk, float routed_scale, int32_t *ids, float *w, void *stream);

/*
 * The router of the pages' decode layer in one call: logits = x * router^T
 * (coli_matmul_multi with the uploaded router matrix, [n_experts][H], any
 * format; the pages' router is f32, fmt=0), then coli_moe_topk.  The logits
 * live in a library scratch buffer per stream.
 *   x        device f32 [S][H].
 *   Other arguments and errors as coli_moe_topk and coli_matmul.
 */
int coli_moe_router(const float *x, int S, const coli_tensor *router, const float *bias, int K, float top_p,
                    int norm_topk, float routed_scale, int32_t *ids, float *w, void *stream);

/*
 * The routed-expert block (colibri-strix commit log, "metal: batched
 * moe_block"; the shared expert is one more expert with weight 1 for every
 * row, "fuse shared expert into GPU block"):
 *   y[s][:] = sum over k with e = ids[s*K+k] >= 0 of
 *             w[s*K+k] * down_e( silu(gate_e x[s]) * up_e x[s] )
 *   x        device f32 [S][H].
 *   experts  HOST array of n_experts descriptors; every gate/up is [F][H] and
 *            every down is [H][F] with one F and H for the whole table; all
 *            gates and ups share one format, all downs share one format; gs may
 *            differ per matrix.  The table may be reused across calls; the
 *            library caches its device copy keyed by the tensors it names.
 *   ids      device int32 [S][K], each in [-1, n_experts).
 *   w        device f32 [S][K] routing weights, used as given.
 *   y        device f32 [S][H], overwritten; must not overlap x.
 *   S >= 1, 1 <= K <= 64.
 * S*K <= 64 runs a single-launch decode kernel (one cooperative grid, one CTA
 * per SM, weights streamed through shared memory with bulk copies): for S = 1
 * and int4 tables (fmt=2, or fmt=4 with gs 64 or 128; H, F <= 6144; at most
 * one routed expert per SM) the kernel whose dot products run on the tensor
 * cores; for other S = 1 int4 / int8 tables the one that decodes with dp4a;
 * otherwise the slab kernel (S = 1) or the general decode kernel.  Larger S*K
 * runs the prefill pipeline (routing, gather, grouped gate/up, grouped down,
 * combine) on the tensor cores for int4 tables with gs % 64 == 0, on the CUDA
 * cores otherwise; int3 (fmt=5) tables take the int4 paths.  Every call checks the whole table (shapes, formats,
 * device) on the host: for a table used over and over, create it once with
 * coli_expert_table_create and call coli_moe_block_t.  An id out of range is
 * recorded for coli_sync_check(stream) and y is then unspecified.
 * Errors: COLI_EINVAL, COLI_EFMT, COLI_EDEVICE, COLI_ENOMEM, COLI_ECUDA.
 */
int coli_moe_block(const float *x, int S, const coli_expert *experts, int n_experts,
                   const int32_t *ids, const float *w, int K, float *y, void *stream);

/*
 * An expert table checked and copied to the device once, for coli_moe_block_t
 * (the host work of a call is then independent of the number of experts).
 * The colibri pages have no counterpart of this entry point.
 *   experts, n_experts  as coli_moe_block; copied, so the array may be freed.
 *   out      receives the table; the tensors it names must stay alive until
 *            coli_expert_table_free.  The table belongs to the device current
 *            at creation.
 * Errors: COLI_EINVAL, COLI_EFMT, COLI_EDEVICE, COLI_ENOMEM, COLI_ECUDA.
 */
typedef struct coli_expert_table coli_expert_table;
int coli_expert_table_create(const coli_expert *experts, int n_experts, coli_expert_table **out);
void coli_expert_table_free(coli_expert_table *table);

/*
 * coli_moe_block on a table from coli_expert_table_create: the same result,
 * the same kernels.  The table's decode plan for the last K used is kept with
 * it.  The table may be used from several host threads.
 * Errors: COLI_EINVAL (NULL pointer, S or K out of range), COLI_EDEVICE (the
 * current device is not the table's), COLI_ENOMEM, COLI_ECUDA.
 */
int coli_moe_block_t(const float *x, int S, const coli_expert_table *table, const int32_t *ids,
                     const float *w, int K, float *y, void *stream);

/*
 * The decode expert block of coli_moe_block for callers that cannot allocate
 * device memory.  The colibri pages have no counterpart of this entry point.
 *
 * Some callers must not call cudaMalloc/cudaFree: latency-critical decode
 * loops (allocation synchronises the device), processes whose GPU memory is
 * owned by another allocator.  coli_moe_block allocates scratch and an
 * expert-table copy on first use; this entry point allocates nothing.  Its
 * scratch (expert descriptors, the h buffer, the grid barrier words) is one
 * file-scope device array of about 2.2 MB that every GPU loading the library
 * holds until the process exits.
 *   Arguments as coli_moe_block, plus:
 *   dev_error  device int32, an output: cleared by the call, then set by the
 *              kernel to 1 if its bounded grid-wide wait ran out or 2 if a
 *              routing id was outside [-1, n_experts) (y is then unspecified).
 *   Limits (refused with COLI_EINVAL, nothing launched): S*K <= 64,
 *   n_experts <= 1024, S*K*F <= 524288, and the activations must fit the
 *   single-launch decode kernel's shared memory; fmt=4 and fmt=5 need
 *   gs % 32 == 0 (COLI_EFMT).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress).  The expert descriptors go to the array through the
 * parameters of a small copy kernel, and only when they differ from the ones
 * the previous call on the device left there; no host memory is read by the
 * device.  Every call shares the array: calls that may overlap on the GPU
 * (unordered streams, several host threads) race and must be serialised by
 * the caller.  Counts as a compute call for coli_set_fail_after and
 * coli_get_stats.
 * Errors: COLI_EINVAL, COLI_EFMT, COLI_EDEVICE, COLI_ECUDA, COLI_EINJECTED.
 */
int coli_moe_block_noalloc(const float *x, int S, const coli_expert *experts, int n_experts,
                           const int32_t *ids, const float *w, int K, float *y, int32_t *dev_error,
                           void *stream);

/* Synchronize `stream`, then report (and clear) any error the library's
 * kernels recorded on this device: COLI_ETIMEOUT for a bounded wait that ran
 * out, COLI_EINVAL for an out-of-range routing id, COLI_ECUDA for a CUDA
 * error.  Returns COLI_OK otherwise. */
int coli_sync_check(void *stream);

/* Message for the last error on the calling thread ("" if none). */
const char *coli_last_error(void);

/* Counters since load or the last reset. */
void coli_get_stats(coli_stats *out);
void coli_reset_stats(void);

/* Host-side fault injection: after n more successful compute calls, every
 * compute call returns COLI_EINJECTED without launching anything.  n < 0
 * switches it off.  The environment variable COLI_FAIL_AFTER=n sets it at
 * load time. */
void coli_set_fail_after(int64_t n);

/* Library version string. */
const char *coli_version(void);

#ifdef __cplusplus
}
#endif
#endif /* COLI_H */
