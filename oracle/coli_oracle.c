/*
 * coli_oracle.c -- plain CPU oracle for the quantized-weight matvec and the
 * routed-expert block.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the CPU-baseline leg of the benchmark are the only callers.  The CUDA
 * library never links, loads or calls this file, and this file shares no code,
 * header, table or constant with it.
 *
 * Everything is scalar, element by element, with double accumulation, in the
 * order the definitions state.  The only parallelism is an OpenMP loop over
 * independent outputs, which does not change any arithmetic.
 *
 * Sources (colibri project pages):
 *   [T]  PR #298 page, commit message adding tests/test_i4_grouped.c: the
 *        reference "dequantizes nibble -> (v-8)*scale[i/gs] and accumulates in
 *        double"; nibble extremes 0x00/0xFF decode to -8/+7; partial last
 *        group ("glen clamp"); odd I; gs > I.
 *   [M]  PR #298 page, commit message "metal: grouped-int4 (fmt=4) GEMV
 *        support": fmt=4 has the nibble layout of fmt=2 with one f32 scale per
 *        gs inputs along I, folded into the accumulation per group; fmt 1-3
 *        apply one scale per output row after the dot product.
 *   [C]  PR #298 page, commit message "CUDA backend had no fmt=4 case":
 *        scale per row for fmt 1/2/3, per group for fmt=4, O*ceil(I/gs) scales.
 *   [Q]  PR #298 page, commit message on qt_addrow / qt_matvec_rows: int2 row
 *        stride (I+3)/4 bytes; int8 bytes "same convention as fmt=1".
 *   [B]  colibri-strix commit log, "metal: batched moe_block": gate/up ->
 *        silu -> down per expert with per-row ragged routing, weighted
 *        scatter-add of the expert outputs.
 *   [E]  colibri-strix commit log, "fuse shared expert into GPU block": the
 *        shared expert is one more expert with weight 1.0 over all rows.
 *   [R]  colibri-strix commit log, "metal: full decode layer in ONE command
 *        buffer": the router is an f32 matvec followed by a sigmoid, then an
 *        exact top-K selection -- greedy argmax over sigmoid + bias with the
 *        CPU's tie order -- with top-p truncation, norm_topk and routed_scale.
 *   [A]  PR #298 page, commit message on qt_addrow / qt_matvec_rows: the two
 *        functions serve the kv_b MLA-absorption path; qt_matvec_rows is a
 *        matvec over a range of rows of a quantized matrix, qt_addrow adds a
 *        coefficient times one dequantized row into an accumulator.
 *   [P]  PR #298 page, commit message on qt_addrow / qt_matvec_rows (fmt=7):
 *        an fp8 "passthrough" format holding one raw byte per element (the
 *        byte convention of fmt=1) and ceil(O/128) * ceil(I/128) per-block
 *        f32 scales; a [130,130] tensor has 4 blocks.
 *   [V]  PR #298 page, Vulkan fmt=4 commit message and the #377 retarget
 *        list: fmt=5 is int3 (#168); like fmt=4 it skips the per-row scale
 *        (its scales vary along the row) and has a group size
 *        (detect_group_size serves it); the fmt=4 shaders gate gs to
 *        multiples of 8 so that a packed word never straddles a group.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - element 2j of an int4 row is the LOW nibble of byte j;
 *   - element 4j+t of an int2 row is bits [2t, 2t+1] of byte j, value crumb-2;
 *   - int8 codes are two's complement;
 *   - every row starts on a byte boundary: int4 rows are ceil(I/2) bytes;
 *   - group g covers inputs [g*gs, min((g+1)*gs, I)), ng = ceil(I/gs);
 *   - silu(g) = g / (1 + exp(-g));
 *   - routing weights are used as given; id -1 is an empty slot; y is
 *     overwritten; routing order is a stable sort of slots (s asc, k asc);
 *   - router top-K ([R]): the score of expert e is sigmoid(logit_e), computed
 *     in double and rounded to f32; the selection key is score + bias in f32;
 *     the greedy argmax breaks ties toward the lower id; a selected expert's
 *     weight is its score (the bias only steers the choice); top-p keeps the
 *     leading experts (selection order) while the f32 running sum of scores
 *     before each is below top_p * (f32 sum of the K scores), top_p <= 0 or
 *     >= 1 keeps all K; the rest become empty slots (id -1, weight 0);
 *     norm_topk divides the kept weights by their f32 sum; routed_scale then
 *     multiplies them.  Every decision and every weight is taken in f32, one
 *     rounding per operation (this file is compiled without FMA contraction);
 *   - fmt=7 ([P]): the byte of element (o, i) is an OCP FP8 E4M3 number (sign,
 *     4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal;
 *     no infinities; S.1111.111 is NaN), multiplied by the scale of block
 *     (o / 128, i / 128); the scales are stored block-row major,
 *     s[(o / 128) * ceil(I / 128) + i / 128]; blocks at the right and bottom
 *     edges are partial.  The gs argument is ignored for fmt=7;
 *   - fmt=5 ([V]; the pages give no bit layout): element 8j+t of a row is
 *     bits [3t, 3t+2] of the 24-bit little-endian word made of bytes 3j,
 *     3j+1, 3j+2 of the row (low bits first, as int4 and int2 fill a byte),
 *     a row is 3*ceil(I/8) bytes, the value is code - 4 (offset binary, as
 *     int4's -8 and int2's -2), times the f32 scale of group i/gs stored as
 *     for fmt=4 (O*ceil(I/gs) scales); gs is a multiple of 8, so the 8 codes
 *     of a 3-byte unit share one group;
 *   - absorption ([A]): head h of n_heads owns rows o0 + h*stride + j,
 *     j < n_rows; the row-range matvec gives each head its own input vector,
 *     y[s][h][j] = sum_i w[o0+h*stride+j][i] x[s][h][i]; the transposed form
 *     accumulates addrow over the head's rows in ascending row order,
 *     y[s][h][i] = sum_j x[s][h][j] w[o0+h*stride+j][i]; y is overwritten.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

/* Planted-mistake switch used only by the mutation tests: a build with
 * -DORACLE_MUTATION=k carries exactly one deliberate error so the tests can
 * show that the pins catch it.  The normal build has ORACLE_MUTATION == 0. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

int oracle_mutation(void) { return ORACLE_MUTATION; }

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (timing only: every result is the
 * same at any thread count, each output element being one thread's ordered
 * sum).  Returns the previous count. */
int oracle_set_threads(int n)
{
    const int prev = oracle_threads();
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
    return prev;
}

/* Bytes of one packed row on the host, per the readings above ([Q] for int2). */
int64_t oracle_row_bytes(int fmt, int64_t I)
{
    switch (fmt) {
    case 0: return 4 * I;
    case 1: return I;
    case 2: return (I + 1) / 2;
    case 3: return (I + 3) / 4;
    case 4: return (I + 1) / 2;
    case 5: return 3 * ((I + 7) / 8);
    case 7: return I;
    default: return -1;
    }
}

/* Number of f32 scales: none for fmt=0, one per row for fmt 1-3, O*ceil(I/gs)
 * for fmt=4 ([C]) and fmt=5 ([V]), one per 128 x 128 block for fmt=7 ([P]). */
int64_t oracle_scale_count(int fmt, int gs, int64_t O, int64_t I)
{
    switch (fmt) {
    case 0: return 0;
    case 1: case 2: case 3: return O;
    case 4: case 5: return gs > 0 ? O * ((I + gs - 1) / gs) : -1;
    case 7: return ((O + 127) / 128) * ((I + 127) / 128);
    default: return -1;
    }
}

/* Decoded code value (integer part, before scaling) of element (o, i). */
static int oracle_code(int fmt, int64_t I, const uint8_t *q, int64_t o, int64_t i)
{
    const int64_t rb = oracle_row_bytes(fmt, I);
    const uint8_t *row = q + o * rb;
    switch (fmt) {
    case 1: {
        /* two's complement int8 */
        int v = row[i];
        return v >= 128 ? v - 256 : v;
    }
    case 2: case 4: {
        uint8_t b = row[i / 2];
#if ORACLE_MUTATION == 1
        int nib = (i % 2 == 0) ? (b >> 4) : (b & 0xF);     /* planted: swapped nibble order */
#else
        int nib = (i % 2 == 0) ? (b & 0xF) : (b >> 4);     /* even element = low nibble */
#endif
#if ORACLE_MUTATION == 2
        return nib >= 8 ? nib - 16 : nib;                  /* planted: two's complement */
#else
        return nib - 8;                                    /* offset binary [T] */
#endif
    }
    case 3: {
        uint8_t b = row[i / 4];
        int cr = (b >> (2 * (int)(i % 4))) & 3;
        return cr - 2;                                     /* offset binary crumb */
    }
    case 5: {
        /* the 3-byte unit of elements 8j .. 8j+7, as one little-endian word */
        const uint8_t *u = row + 3 * (i / 8);
        const uint32_t word = (uint32_t)u[0] | ((uint32_t)u[1] << 8) | ((uint32_t)u[2] << 16);
#if ORACLE_MUTATION == 13
        const int c = (int)((word >> (21 - 3 * (int)(i % 8))) & 7);   /* planted: high bits first */
#else
        const int c = (int)((word >> (3 * (int)(i % 8))) & 7);
#endif
#if ORACLE_MUTATION == 14
        return c - 3;                                      /* planted: wrong offset */
#else
        return c - 4;                                      /* offset binary 3-bit code */
#endif
    }
    default:
        return 0;
    }
}

/* Value of one OCP FP8 E4M3 byte, from the format's definition: normal
 * numbers (-1)^s 2^(e-7) (1 + m/8), subnormals (-1)^s 2^-6 (m/8), NaN for
 * exponent and mantissa all ones. */
double oracle_fp8_value(int byte)
{
    const int sgn = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
#if ORACLE_MUTATION == 11
    v = ldexp(1.0 + m / 8.0, e - 7);                        /* planted: subnormals read as normals */
#else
    if (e == 0)
        v = ldexp(m / 8.0, -6);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
#endif
    return sgn ? -v : v;
}

/* Scale of element (o, i). */
static double oracle_scale(int fmt, int gs, int64_t I, const float *s, int64_t o, int64_t i)
{
    switch (fmt) {
    case 1: case 2: case 3:
        return (double)s[o];
    case 4: case 5: {
        const int64_t ng = (I + gs - 1) / gs;
#if ORACLE_MUTATION == 3
        (void)ng; (void)i;
        return (double)s[o];                               /* planted: per-row scale on fmt=4 */
#elif ORACLE_MUTATION == 4
        return (double)s[o * ng + (i + 1) / gs];           /* planted: shifted group boundary */
#else
        return (double)s[o * ng + i / gs];
#endif
    }
    case 7: {
        const int64_t nbr = (I + 127) / 128;               /* blocks per block-row */
#if ORACLE_MUTATION == 10
        return (double)s[(i / 128) * nbr + o / 128];       /* planted: transposed block index */
#else
        return (double)s[(o / 128) * nbr + i / 128];
#endif
    }
    default:
        return 1.0;
    }
}

/* Dequantized weight w[o][i] in double: the definition in [T], generalised
 * to every format by [M] and [C]. */
static double oracle_weight(int fmt, int gs, int64_t I, const void *data, const float *s,
                            int64_t o, int64_t i)
{
    if (fmt == 0)
        return (double)((const float *)data)[o * I + i];
    if (fmt == 7)
        return oracle_fp8_value(((const uint8_t *)data)[o * I + i]) * oracle_scale(fmt, gs, I, s, o, i);
    return (double)oracle_code(fmt, I, (const uint8_t *)data, o, i) * oracle_scale(fmt, gs, I, s, o, i);
}

static int oracle_check(int fmt, int gs, int64_t O, int64_t I)
{
    if (fmt < 0 || fmt == 6 || fmt > 7 || O < 1 || I < 1)
        return ORACLE_EINVAL;
    if (fmt == 4 && (gs < 2 || (gs & 1)))
        return ORACLE_EINVAL;
    if (fmt == 5 && (gs < 8 || gs % 8 != 0))
        return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* One dequantized row as doubles (out has I entries). */
int oracle_dequant_row(int fmt, int gs, int64_t O, int64_t I, const void *data,
                       const float *scales, int64_t o, double *out)
{
    if (oracle_check(fmt, gs, O, I) || o < 0 || o >= O)
        return ORACLE_EINVAL;
    for (int64_t i = 0; i < I; i++)
        out[i] = oracle_weight(fmt, gs, I, data, scales, o, i);
    return ORACLE_OK;
}

/* y[s][o] = sum_i w[o][i] * x[s][i], dequantize-then-multiply, accumulated in
 * double over i in ascending order and rounded to f32 once at the end.
 * y64 (optional) receives the double result, yabs (optional) the sum of
 * |w[o][i] * x[s][i]| that the pages use to assess rounding ([T], tolerance
 * paragraph). */
int oracle_matmul(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                  int64_t S, const float *x, float *y, double *y64, double *yabs)
{
    if (oracle_check(fmt, gs, O, I) || S < 0)
        return ORACLE_EINVAL;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t s = 0; s < S; s++) {
        for (int64_t o = 0; o < O; o++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < I; i++) {
                const double t = oracle_weight(fmt, gs, I, data, scales, o, i) * (double)x[s * I + i];
#if ORACLE_MUTATION == 5
                if (i == I - 1) continue;                  /* planted: dropped last term */
#endif
                acc += t;
                mag += fabs(t);
            }
            if (y) y[s * O + o] = (float)acc;
            if (y64) y64[s * O + o] = acc;
            if (yabs) yabs[s * O + o] = mag;
        }
    }
    return ORACLE_OK;
}

/* The same product in the evaluation order the pages give for the kernels
 * ([M] Shader paragraph, [C]): fmt 1-3 multiply the row scale once after the
 * integer-code dot product; fmt=4 (and fmt=5, [V]) forms each group's code dot product and
 * folds the group scale in before summing over groups; fmt=7 does the same per
 * 128-input block with the scale of the row's block.  Mathematically equal
 * to oracle_matmul; used to pin that equality. */
int oracle_matmul_inline(int fmt, int gs, int64_t O, int64_t I, const void *data,
                         const float *scales, int64_t S, const float *x, double *y64)
{
    if (oracle_check(fmt, gs, O, I) || S < 0)
        return ORACLE_EINVAL;
    const uint8_t *q = (const uint8_t *)data;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t s = 0; s < S; s++) {
        for (int64_t o = 0; o < O; o++) {
            const float *xs = x + s * I;
            double acc = 0.0;
            if (fmt == 0) {
                for (int64_t i = 0; i < I; i++)
                    acc += (double)((const float *)data)[o * I + i] * (double)xs[i];
            } else if (fmt == 4 || fmt == 5) {
                const int64_t ng = (I + gs - 1) / gs;
                for (int64_t g = 0; g < ng; g++) {
                    const int64_t i0 = g * gs;
                    const int64_t i1 = (i0 + gs < I) ? i0 + gs : I;   /* glen clamp */
                    double part = 0.0;
                    for (int64_t i = i0; i < i1; i++)
                        part += (double)oracle_code(fmt, I, q, o, i) * (double)xs[i];
                    acc += (double)scales[o * ng + g] * part;
                }
            } else if (fmt == 7) {
                const int64_t nb = (I + 127) / 128;
                for (int64_t b = 0; b < nb; b++) {
                    const int64_t i1 = (b * 128 + 128 < I) ? b * 128 + 128 : I;
                    double part = 0.0;
                    for (int64_t i = b * 128; i < i1; i++)
                        part += oracle_fp8_value(q[o * I + i]) * (double)xs[i];
                    acc += (double)scales[(o / 128) * nb + b] * part;
                }
            } else {
                double part = 0.0;
                for (int64_t i = 0; i < I; i++)
                    part += (double)oracle_code(fmt, I, q, o, i) * (double)xs[i];
                acc = (double)scales[o] * part;
            }
            y64[s * O + o] = acc;
        }
    }
    return ORACLE_OK;
}

/* silu(g) = g * sigmoid(g) = g / (1 + exp(-g)), in double. */
double oracle_silu(double g)
{
#if ORACLE_MUTATION == 6
    return g / (1.0 + exp(g));                             /* planted: sign error */
#else
    return g / (1.0 + exp(-g));
#endif
}

/* Routing inversion: a stable counting sort of the slots (s, k) with
 * ids[s*K+k] >= 0 by expert id.  offsets has n_experts+1 entries; order
 * receives the slot indices s*K+k of each expert's group in (s asc, k asc)
 * order.  Returns the number of valid slots, or ORACLE_EINVAL for an id
 * outside [-1, n_experts). */
int64_t oracle_route(const int32_t *ids, int64_t S, int64_t K, int64_t n_experts,
                     int64_t *offsets, int64_t *order)
{
    if (S < 0 || K < 1 || n_experts < 1)
        return ORACLE_EINVAL;
    for (int64_t t = 0; t < S * K; t++)
        if (ids[t] < -1 || ids[t] >= n_experts)
            return ORACLE_EINVAL;
    for (int64_t e = 0; e <= n_experts; e++)
        offsets[e] = 0;
    for (int64_t t = 0; t < S * K; t++)            /* count */
        if (ids[t] >= 0)
            offsets[ids[t] + 1]++;
    for (int64_t e = 0; e < n_experts; e++)        /* exclusive prefix sum */
        offsets[e + 1] += offsets[e];
    int64_t *fill = (int64_t *)malloc(sizeof(int64_t) * (size_t)n_experts);
    if (!fill)
        return ORACLE_EINVAL;
    for (int64_t e = 0; e < n_experts; e++)
        fill[e] = offsets[e];
    for (int64_t t = 0; t < S * K; t++)            /* place, in slot order */
        if (ids[t] >= 0)
            order[fill[ids[t]]++] = t;
    free(fill);
    return offsets[n_experts];
}

/* One expert matrix as the oracle sees it. */
typedef struct {
    int fmt, gs;
    int64_t O, I;
    const void *data;
    const float *scales;
} oracle_mat;

/* Routed-expert block ([B], [E]):
 *   for each row s and slot k with e = ids[s*K+k] >= 0:
 *     g_j = sum_i G_e[j][i] x[s][i],  u_j = sum_i U_e[j][i] x[s][i]   (j < F)
 *     h_j = silu(g_j) * u_j
 *     y[s][o] += w[s*K+k] * sum_j D_e[o][j] h_j                         (o < H)
 *   with y starting at zero, all in double, rounded to f32 at the end.
 * gate/up/down hold n_experts matrices each: gate and up are [F][H], down is
 * [H][F].  y64 (optional) receives the double result. */
int oracle_moe_block(int64_t H, int64_t F, int64_t S, int64_t K, int64_t n_experts,
                     const oracle_mat *gate, const oracle_mat *up, const oracle_mat *down,
                     const float *x, const int32_t *ids, const float *w, float *y, double *y64)
{
    if (H < 1 || F < 1 || S < 0 || K < 1 || n_experts < 1)
        return ORACLE_EINVAL;
    for (int64_t e = 0; e < n_experts; e++) {
        if (oracle_check(gate[e].fmt, gate[e].gs, gate[e].O, gate[e].I) ||
            oracle_check(up[e].fmt, up[e].gs, up[e].O, up[e].I) ||
            oracle_check(down[e].fmt, down[e].gs, down[e].O, down[e].I))
            return ORACLE_EINVAL;
        if (gate[e].O != F || gate[e].I != H || up[e].O != F || up[e].I != H ||
            down[e].O != H || down[e].I != F)
            return ORACLE_EINVAL;
    }
    for (int64_t t = 0; t < S * K; t++)
        if (ids[t] < -1 || ids[t] >= n_experts)
            return ORACLE_EINVAL;

    double *acc = (double *)calloc((size_t)(S * H), sizeof(double));
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    if (!acc || !h) {
        free(acc);
        free(h);
        return ORACLE_EINVAL;
    }
    for (int64_t s = 0; s < S; s++) {
        const float *xs = x + s * H;
        for (int64_t k = 0; k < K; k++) {
            const int32_t e = ids[s * K + k];
            if (e < 0)
                continue;                                  /* empty slot */
            const oracle_mat *G = &gate[e], *U = &up[e], *D = &down[e];
#pragma omp parallel for schedule(static)
            for (int64_t j = 0; j < F; j++) {
                double g = 0.0, u = 0.0;
                for (int64_t i = 0; i < H; i++) {
                    g += oracle_weight(G->fmt, G->gs, H, G->data, G->scales, j, i) * (double)xs[i];
                    u += oracle_weight(U->fmt, U->gs, H, U->data, U->scales, j, i) * (double)xs[i];
                }
                h[j] = oracle_silu(g) * u;
            }
            const double wk = (double)w[s * K + k];
#pragma omp parallel for schedule(static)
            for (int64_t o = 0; o < H; o++) {
                double d = 0.0;
                for (int64_t j = 0; j < F; j++)
                    d += oracle_weight(D->fmt, D->gs, F, D->data, D->scales, o, j) * h[j];
#if ORACLE_MUTATION == 7
                acc[s * H + o] += d;                       /* planted: routing weight dropped */
#else
                acc[s * H + o] += wk * d;
#endif
            }
        }
    }
    for (int64_t t = 0; t < S * H; t++) {
        if (y) y[t] = (float)acc[t];
        if (y64) y64[t] = acc[t];
    }
    free(acc);
    free(h);
    return ORACLE_OK;
}

/* Router top-K ([R]) for S rows of n_experts logits (f32 [S][E]); bias is
 * f32 [E] or NULL.  ids/w receive [S][K].  See the reading in the header. */
int oracle_moe_topk(const float *logits, const float *bias, int64_t S, int64_t E, int64_t K,
                    float top_p, int norm_topk, float routed_scale, int32_t *ids, float *w)
{
    if (S < 0 || E < 1 || K < 1 || K > E)
        return ORACLE_EINVAL;
    float *score = (float *)malloc(sizeof(float) * (size_t)E);
    float *key = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!score || !key || !taken) {
        free(score); free(key); free(taken);
        return ORACLE_EINVAL;
    }
    for (int64_t s = 0; s < S; s++) {
        const float *l = logits + s * E;
        for (int64_t e = 0; e < E; e++) {
            score[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));
#if ORACLE_MUTATION == 9
            key[e] = score[e];                              /* planted: bias ignored */
#else
            key[e] = score[e] + (bias ? bias[e] : 0.0f);
#endif
            taken[e] = 0;
        }
        int32_t *id = ids + s * K;
        float *wt = w + s * K;
        for (int64_t k = 0; k < K; k++) {                 /* greedy argmax */
            int64_t best = -1;
            for (int64_t e = 0; e < E; e++) {
                if (taken[e])
                    continue;
#if ORACLE_MUTATION == 8
                if (best < 0 || key[e] >= key[best])        /* planted: ties go to the higher id */
#else
                if (best < 0 || key[e] > key[best])
#endif
                    best = e;
            }
            taken[best] = 1;
            id[k] = (int32_t)best;
            wt[k] = score[best];
        }
        int64_t keep = K;                                   /* top-p truncation */
        if (top_p > 0.0f && top_p < 1.0f) {
            float total = 0.0f;
            for (int64_t k = 0; k < K; k++)
                total = total + wt[k];
            const float limit = top_p * total;
            float cum = 0.0f;
            keep = 0;
            for (int64_t k = 0; k < K; k++) {
                if (!(cum < limit))
                    break;
                cum = cum + wt[k];
                keep++;
            }
        }
        for (int64_t k = keep; k < K; k++) {
            id[k] = -1;
            wt[k] = 0.0f;
        }
        if (norm_topk) {
            float sum = 0.0f;
            for (int64_t k = 0; k < keep; k++)
                sum = sum + wt[k];
            for (int64_t k = 0; k < keep; k++)
                wt[k] = wt[k] / sum;
        }
        for (int64_t k = 0; k < keep; k++)
            wt[k] = wt[k] * routed_scale;
    }
    free(score); free(key); free(taken);
    return 0;
}

/* Row-range matvec of the absorption path ([A], qt_matvec_rows), per head:
 * y[s][h][j] = sum_i w[o0 + h*stride + j][i] * x[s][h][i], double accumulation
 * in ascending i, rounded to f32 once.  x is [S][n_heads][I], y is
 * [S][n_heads][n_rows]. */
int oracle_matmul_rows(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                       int64_t o0, int64_t stride, int64_t n_rows, int64_t n_heads, int64_t S,
                       const float *x, float *y)
{
    if (oracle_check(fmt, gs, O, I) || o0 < 0 || n_rows < 1 || n_heads < 1 || stride < 0 || S < 0 ||
        o0 + (n_heads - 1) * stride + n_rows > O)
        return ORACLE_EINVAL;
#pragma omp parallel for collapse(3) schedule(static)
    for (int64_t s = 0; s < S; s++)
        for (int64_t h = 0; h < n_heads; h++)
            for (int64_t j = 0; j < n_rows; j++) {
                const int64_t o = o0 + h * stride + j;
                const float *xv = x + (s * n_heads + h) * I;
                double acc = 0.0;
                for (int64_t i = 0; i < I; i++)
                    acc += oracle_weight(fmt, gs, I, data, scales, o, i) * (double)xv[i];
                y[(s * n_heads + h) * n_rows + j] = (float)acc;
            }
    return ORACLE_OK;
}

/* Transposed row-range product of the absorption path ([A], qt_addrow summed
 * over a head's rows): y[s][h][i] = sum_j x[s][h][j] * w[o0 + h*stride + j][i],
 * each row added in ascending j in double, rounded to f32 once.  x is
 * [S][n_heads][n_rows], y is [S][n_heads][I]. */
int oracle_matmul_rows_t(int fmt, int gs, int64_t O, int64_t I, const void *data, const float *scales,
                         int64_t o0, int64_t stride, int64_t n_rows, int64_t n_heads, int64_t S,
                         const float *x, float *y)
{
    if (oracle_check(fmt, gs, O, I) || o0 < 0 || n_rows < 1 || n_heads < 1 || stride < 0 || S < 0 ||
        o0 + (n_heads - 1) * stride + n_rows > O)
        return ORACLE_EINVAL;
    int rc = ORACLE_OK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t s = 0; s < S; s++)
        for (int64_t h = 0; h < n_heads; h++) {
            double *acc = (double *)calloc((size_t)I, sizeof(double));
            const float *xv = x + (s * n_heads + h) * n_rows;
            if (!acc) {
                rc = ORACLE_EINVAL;
                continue;
            }
            for (int64_t j = 0; j < n_rows; j++) {
#if ORACLE_MUTATION == 12
                const int64_t o = o0 + h * n_rows + j;          /* planted: heads packed at n_rows, not stride */
#else
                const int64_t o = o0 + h * stride + j;
#endif
                const double c = (double)xv[j];
                for (int64_t i = 0; i < I; i++)
                    acc[i] += c * oracle_weight(fmt, gs, I, data, scales, o, i);   /* addrow */
            }
            for (int64_t i = 0; i < I; i++)
                y[(s * n_heads + h) * I + i] = (float)acc[i];
            free(acc);
        }
    return rc;
}
