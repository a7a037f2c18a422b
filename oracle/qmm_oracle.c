/*
 * Plain CPU oracle for MLX grouped affine quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * Everything here is written to be checked by eye against the pages:
 *
 *  - Packed format (nuvec_core quantized.rs, module doc; `quantize` doc):
 *    each row of a weight is a little-endian bit stream of `bits`-bit codes,
 *    stored as uint32 words; a row of `cols` codes takes cols*bits/32 words.
 *    Code j of a row occupies stream bits [j*bits, (j+1)*bits), least
 *    significant bit first (rlx-moshi src/mlx_dequant.rs, `dequantize_affine`
 *    doc: code s sits at bits [s*bits, (s+1)*bits) of its word).  Stream bit i
 *    is bit (i mod 32) of word floor(i/32).  The oracle reads a code one bit at
 *    a time, on purpose unlike any shift-and-mask unpacker.
 *
 *  - Groups (nuvec_core quantized.rs, module doc; spark_runtime
 *    weights/mlx_int8.rs, module doc): one scale and one bias per group of
 *    `group_size` consecutive codes along the last (stored) axis, stored as
 *    bf16 [rows, cols/group_size].
 *
 *  - Dequantization (rlx-moshi `dequantize_affine`; nuvec_core `dequantize`;
 *    spark_runtime module doc): w = scale * code + bias, bias added (it is
 *    the group minimum).  In fp32 the product of a bf16 scale and a code of
 *    at most 8 bits is exact, so fp32 `p = s*c; r = p + b` rounds once, at
 *    the add.  This file is compiled with -ffp-contract=off so that the two
 *    statements stay two operations.  bf16 output is the round-to-nearest-even
 *    bf16 of that fp32 value.
 *
 *  - quantized_matmul (nuvec_core `quantized_matmul` doc; maya2_mlx quant.py
 *    `mm`): y = x . dequant(W)^T when `transpose` (W stored [N, K], the
 *    [out, in] layout), else y = x . dequant(W) (W stored [K, N], groups and
 *    packing along N).  The oracle takes every weight exactly (s*c + b in
 *    fp64 is exact) and accumulates in fp64.  It also returns
 *    A[m,n] = sum_k |x[m,k] * w[k,n]|, the scale of the matmul tolerance.
 *
 *  - rows (maya2_mlx quant.py, `rows`): dequantize only the gathered rows
 *    w[idx].  An index outside the table gives a zero row (the pages say
 *    nothing about it; the library reports such an index through its device
 *    error word, and the oracle counts them).
 *
 *  - Other dtypes (nuvec_core quantized.rs, `quantize` doc: w may be
 *    float16, bfloat16 or float32 and the scales and biases keep w's dtype;
 *    `dequantize` doc: the result is in the scales' dtype; `quantized_matmul`:
 *    x, scales and biases are promoted to one floating-point type).  The
 *    typed functions take each buffer's type: ORACLE_F32, ORACLE_BF16 or
 *    ORACLE_F16 (IEEE binary16).  A dequantized element is scale * code +
 *    bias rounded once to fp32 (fmaf); for 16-bit scales the product is exact
 *    in fp32, so this is the same value as the multiply-then-add above.  A
 *    16-bit output is the round-to-nearest-even of that fp32 value.
 *
 * Threading: rows (or output elements) are independent, so they are split
 * across plain pthreads, the way rlx-moshi's `dequantize_affine` splits rows
 * across rayon workers.  Results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bits --- */

/* Stream bit i of one row. */
static inline uint32_t stream_bit(const uint32_t *row_words, int64_t i)
{
    return (row_words[i / 32] >> (uint32_t)(i % 32)) & 1u;
}

/* Code j of one row: bits [j*bits, (j+1)*bits), least significant first. */
uint32_t oracle_code(const uint32_t *row_words, int64_t j, int bits)
{
    uint32_t code = 0;
    for (int t = 0; t < bits; ++t)
        code |= stream_bit(row_words, j * (int64_t)bits + t) << t;
    return code;
}

int64_t oracle_words_per_row(int64_t cols, int bits)
{
    return cols * bits / 32;
}

/* codes[rows, cols] (one byte each) from packed[rows, cols*bits/32]. */
void oracle_unpack(const uint32_t *packed, int64_t rows, int64_t cols, int bits,
                   uint8_t *codes)
{
    int64_t wpr = oracle_words_per_row(cols, bits);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j)
            codes[r * cols + j] = (uint8_t)oracle_code(packed + r * wpr, j, bits);
}

/* The inverse, one bit at a time: the writer side of the same bit stream. */
void oracle_pack(const uint8_t *codes, int64_t rows, int64_t cols, int bits,
                 uint32_t *packed)
{
    int64_t wpr = oracle_words_per_row(cols, bits);
    memset(packed, 0, (size_t)(rows * wpr) * sizeof(uint32_t));
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t *row = packed + r * wpr;
        for (int64_t j = 0; j < cols; ++j)
            for (int t = 0; t < bits; ++t) {
                uint32_t bit = ((uint32_t)codes[r * cols + j] >> t) & 1u;
                int64_t i = j * (int64_t)bits + t;
                row[i / 32] |= bit << (uint32_t)(i % 32);
            }
    }
}

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the top half of an fp32 (rlx-moshi `bf16_to_f32`): exact. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even from fp32 to bf16.  Drop the low 16 bits after
 * adding half an ulp, where "half" is 0x7FFF plus the kept lsb so that an
 * exact tie rounds to the even neighbour.  NaN stays NaN (quiet bit set). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + kept_lsb;
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- fp16 --- */

/* IEEE 754 binary16: sign in bit 15, a 5-bit exponent field (bias 15) in
 * bits 10..14, a 10-bit fraction.  Field 0 holds zero and the subnormals
 * fraction * 2^-24; field 31 the infinities (fraction 0) and NaNs. */
double oracle_f16_to_f64(uint16_t h)
{
    int e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return (h & 0x8000u) ? -v : v;
}

/* Round-to-nearest-even from fp32 to binary16, from the definition: q is the
 * spacing of binary16 numbers at |v| (2^(e-10) for |v| in [2^e, 2^(e+1)),
 * 2^-24 below 2^-14), |v|/q (exact: q is a power of two) goes to the nearest
 * integer with ties to even, and the result is encoded.  Results of 2^16 or
 * more are past the largest finite value (65504) and become infinity. */
uint16_t oracle_f32_to_f16(float f)
{
    double v = (double)f, a = fabs(v);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return sign | 0x7E00u;
    if (isinf(v))
        return sign | 0x7C00u;
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int ex = e - 1 < -14 ? -14 : e - 1;
    double q = ldexp(1.0, ex - 10);
    double r = nearbyint(a / q) * q;
    if (r >= 65536.0)
        return sign | 0x7C00u;
    if (r < ldexp(1.0, -14))
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    int e2;
    double m = frexp(r, &e2); /* r = m * 2^e2, m in [0.5, 1) */
    return sign | (uint16_t)((e2 - 1 + 15) << 10) | (uint16_t)((m * 2.0 - 1.0) * 1024.0);
}

/* Element types of the typed functions. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* Element i of a buffer of the given type, exactly. */
static double load_elem(const void *p, int type, int64_t i)
{
    if (type == ORACLE_BF16)
        return (double)oracle_bf16_to_f32(((const uint16_t *)p)[i]);
    if (type == ORACLE_F16)
        return oracle_f16_to_f64(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

/* Store the fp32 value v as element i: as is, or rounded to nearest even. */
static void store_elem(void *p, int type, int64_t i, float v)
{
    if (type == ORACLE_BF16)
        ((uint16_t *)p)[i] = oracle_f32_to_bf16(v);
    else if (type == ORACLE_F16)
        ((uint16_t *)p)[i] = oracle_f32_to_f16(v);
    else
        ((float *)p)[i] = v;
}

/* One weight in fp32: scale * code + bias, rounded once (C99 fmaf). */
static inline float dequant_f32(float s, uint32_t code, float b)
{
    return fmaf(s, (float)code, b);
}

/* ------------------------------------------------------------- threads --- */

typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end);

typedef struct {
    range_fn fn;
    void *ctx;
    int64_t begin, end;
} range_job;

static void *run_range(void *arg)
{
    range_job *j = (range_job *)arg;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

/* Split [0, count) into nthreads contiguous ranges and run them. */
static void parallel_for(int64_t count, int nthreads, range_fn fn, void *ctx)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > count)
        nthreads = count > 0 ? (int)count : 1;
    if (nthreads == 1) {
        fn(ctx, 0, count);
        return;
    }
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    range_job *jobs = (range_job *)malloc(sizeof(range_job) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].begin = count * t / nthreads;
        jobs[t].end = count * (t + 1) / nthreads;
        pthread_create(&tids[t], NULL, run_range, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(tids[t], NULL);
    free(tids);
    free(jobs);
}

/* ----------------------------------------------------------- dequantize --- */

typedef struct {
    const uint32_t *packed;
    const void *scales, *biases;
    int sb_type;
    const uint32_t *idx; /* NULL: row r of the output is row r of the table */
    int64_t table_rows, cols;
    int group_size, bits, out_type;
    void *out;
    int64_t bad_index; /* rows gathered from outside the table */
} dequant_ctx;

static void dequant_range(void *arg, int64_t begin, int64_t end)
{
    dequant_ctx *c = (dequant_ctx *)arg;
    int64_t wpr = oracle_words_per_row(c->cols, c->bits);
    int64_t groups = c->cols / c->group_size;
    for (int64_t r = begin; r < end; ++r) {
        int64_t src = c->idx ? (int64_t)c->idx[r] : r;
        int in_table = src >= 0 && src < c->table_rows;
        if (!in_table)
            __atomic_add_fetch(&c->bad_index, 1, __ATOMIC_RELAXED);
        for (int64_t j = 0; j < c->cols; ++j) {
            float v = 0.0f;
            if (in_table) {
                int64_t g = j / c->group_size;
                float s = (float)load_elem(c->scales, c->sb_type, src * groups + g);
                float b = (float)load_elem(c->biases, c->sb_type, src * groups + g);
                uint32_t code = oracle_code(c->packed + src * wpr, j, c->bits);
                v = dequant_f32(s, code, b);
            }
            store_elem(c->out, c->out_type, r * c->cols + j, v);
        }
    }
}

/* out[rows, cols] = dequant(W).  Returns 0.  The oracle does not enforce the
 * library's parameter rules: any group size that divides cols and any bit
 * width 1..8 with cols*bits a multiple of 32 is computed as written. */
int oracle_dequantize_typed(const uint32_t *packed, const void *scales,
                            const void *biases, int sb_type, int64_t rows,
                            int64_t cols, int group_size, int bits, int out_type,
                            void *out, int nthreads)
{
    dequant_ctx c = {packed, scales, biases, sb_type, NULL, rows, cols,
                     group_size, bits, out_type, out, 0};
    parallel_for(rows, nthreads, dequant_range, &c);
    return 0;
}

/* bf16 scales and biases; fp32 output, or bf16 if out_bf16. */
int oracle_dequantize(const uint32_t *packed, const uint16_t *scales,
                      const uint16_t *biases, int64_t rows, int64_t cols,
                      int group_size, int bits, int out_bf16, void *out,
                      int nthreads)
{
    return oracle_dequantize_typed(packed, scales, biases, ORACLE_BF16, rows, cols,
                                   group_size, bits,
                                   out_bf16 ? ORACLE_BF16 : ORACLE_F32, out, nthreads);
}

/* out[n, cols] = dequant(W[idx[i]]).  Returns the number of indices outside
 * [0, table_rows); their output rows are zero. */
int64_t oracle_rows_typed(const uint32_t *packed, const void *scales,
                          const void *biases, int sb_type, int64_t table_rows,
                          int64_t cols, const uint32_t *idx, int64_t n,
                          int group_size, int bits, int out_type, void *out,
                          int nthreads)
{
    dequant_ctx c = {packed, scales, biases, sb_type, idx, table_rows, cols,
                     group_size, bits, out_type, out, 0};
    parallel_for(n, nthreads, dequant_range, &c);
    return c.bad_index;
}

int64_t oracle_rows(const uint32_t *packed, const uint16_t *scales,
                    const uint16_t *biases, int64_t table_rows, int64_t cols,
                    const uint32_t *idx, int64_t n, int group_size, int bits,
                    int out_bf16, void *out, int nthreads)
{
    return oracle_rows_typed(packed, scales, biases, ORACLE_BF16, table_rows, cols,
                             idx, n, group_size, bits,
                             out_bf16 ? ORACLE_BF16 : ORACLE_F32, out, nthreads);
}

/* ------------------------------------------------------- quantized matmul --- */

/* The exact weight at logical position (k, n) of the [K, N] right operand
 * (s*c + b in fp64 is exact for 16-bit scales and biases; for fp32 ones it is
 * the fp64 rounding of the exact value, far inside any matmul tolerance). */
static double weight_kn(const uint32_t *packed, const void *scales,
                        const void *biases, int sb_type, int64_t N, int64_t K,
                        int transpose, int group_size, int bits, int64_t k,
                        int64_t n)
{
    /* Stored row and column of the element: [N, K] when transposed. */
    int64_t row = transpose ? n : k;
    int64_t col = transpose ? k : n;
    int64_t cols = transpose ? K : N;
    int64_t wpr = oracle_words_per_row(cols, bits);
    int64_t groups = cols / group_size;
    double s = load_elem(scales, sb_type, row * groups + col / group_size);
    double b = load_elem(biases, sb_type, row * groups + col / group_size);
    uint32_t code = oracle_code(packed + row * wpr, col, bits);
    return s * (double)code + b;
}

typedef struct {
    const void *x;
    int x_type;
    int64_t M;
    const uint32_t *packed;
    const void *scales, *biases;
    int sb_type;
    int64_t N, K;
    int transpose, group_size, bits;
    const int64_t *ms, *ns; /* sampled outputs, or NULL for all of them */
    double *y, *absy;
} qmm_ctx;

/* One output column n for every m: decode the column of weights once. */
static void qmm_cols_range(void *arg, int64_t begin, int64_t end)
{
    qmm_ctx *c = (qmm_ctx *)arg;
    double *w = (double *)malloc(sizeof(double) * (size_t)c->K);
    for (int64_t n = begin; n < end; ++n) {
        for (int64_t k = 0; k < c->K; ++k)
            w[k] = weight_kn(c->packed, c->scales, c->biases, c->sb_type, c->N, c->K,
                             c->transpose, c->group_size, c->bits, k, n);
        for (int64_t m = 0; m < c->M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < c->K; ++k) {
                double t = load_elem(c->x, c->x_type, m * c->K + k) * w[k];
                acc += t;
                mag += fabs(t);
            }
            c->y[m * c->N + n] = acc;
            c->absy[m * c->N + n] = mag;
        }
    }
    free(w);
}

static void qmm_samples_range(void *arg, int64_t begin, int64_t end)
{
    qmm_ctx *c = (qmm_ctx *)arg;
    for (int64_t i = begin; i < end; ++i) {
        int64_t m = c->ms[i], n = c->ns[i];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < c->K; ++k) {
            double t = load_elem(c->x, c->x_type, m * c->K + k) *
                       weight_kn(c->packed, c->scales, c->biases, c->sb_type, c->N,
                                 c->K, c->transpose, c->group_size, c->bits, k, n);
            acc += t;
            mag += fabs(t);
        }
        c->y[i] = acc;
        c->absy[i] = mag;
    }
}

/* y[M, N] and absy[M, N] (fp64) for x [M, K] of x_type and scales/biases of
 * sb_type.  The promoted type changes nothing here: every operand value is
 * exact in fp64, and the result is the exact product up to fp64 rounding. */
int oracle_qmm_typed(const void *x, int x_type, int64_t M, const uint32_t *packed,
                     const void *scales, const void *biases, int sb_type, int64_t N,
                     int64_t K, int transpose, int group_size, int bits, double *y,
                     double *absy, int nthreads)
{
    qmm_ctx c = {x, x_type, M, packed, scales, biases, sb_type, N, K, transpose,
                 group_size, bits, NULL, NULL, y, absy};
    parallel_for(N, nthreads, qmm_cols_range, &c);
    return 0;
}

/* The same, at count sampled output positions (ms[i], ns[i]) only. */
int oracle_qmm_sampled_typed(const void *x, int x_type, int64_t M,
                             const uint32_t *packed, const void *scales,
                             const void *biases, int sb_type, int64_t N, int64_t K,
                             int transpose, int group_size, int bits,
                             const int64_t *ms, const int64_t *ns, int64_t count,
                             double *y, double *absy, int nthreads)
{
    qmm_ctx c = {x, x_type, M, packed, scales, biases, sb_type, N, K, transpose,
                 group_size, bits, ms, ns, y, absy};
    parallel_for(count, nthreads, qmm_samples_range, &c);
    return 0;
}

/* bf16 x, scales and biases. */
int oracle_qmm(const uint16_t *x, int64_t M, const uint32_t *packed,
               const uint16_t *scales, const uint16_t *biases, int64_t N,
               int64_t K, int transpose, int group_size, int bits, double *y,
               double *absy, int nthreads)
{
    return oracle_qmm_typed(x, ORACLE_BF16, M, packed, scales, biases, ORACLE_BF16, N, K,
                            transpose, group_size, bits, y, absy, nthreads);
}

int oracle_qmm_sampled(const uint16_t *x, int64_t M, const uint32_t *packed,
                       const uint16_t *scales, const uint16_t *biases,
                       int64_t N, int64_t K, int transpose, int group_size,
                       int bits, const int64_t *ms, const int64_t *ns,
                       int64_t count, double *y, double *absy, int nthreads)
{
    return oracle_qmm_sampled_typed(x, ORACLE_BF16, M, packed, scales, biases, ORACLE_BF16,
                                    N, K, transpose, group_size, bits, ms, ns, count, y,
                                    absy, nthreads);
}

/* ------------------------------------------------------------ quantize --- */
/*
 * quantize (nuvec_core quantized.rs, module doc: a value w is stored as
 * round((w - bias) / scale), clamped to [0, 2^bits - 1]; `dequantize` doc:
 * bias = the group minimum).  The pages do not give the scale; the reading
 * taken here is the plain min-max one: scale = (max - min) / (2^bits - 1),
 * in fp32, stored as its round-to-nearest-even bf16, and the codes come from
 * the stored (bf16) scale and bias, each step one IEEE fp32 operation, the
 * round half to even (rintf).  A zero scale (a constant group) gives every
 * code 0, so that the group dequantizes to its value exactly.
 * Input w [rows, cols] of w_type (fp32, bf16 or fp16); the scales and biases
 * are stored in w's type (nuvec_core `quantize` doc), the scale rounded to
 * nearest even from its fp32 value, the bias (a value of w) exactly.
 */
typedef struct {
    const void *w;
    int w_type;
    int64_t rows, cols;
    int group_size, bits;
    uint32_t *packed;
    void *scales, *biases;
} quant_ctx;

static void quant_rows_range(void *arg, int64_t begin, int64_t end)
{
    quant_ctx *c = (quant_ctx *)arg;
    int64_t groups = c->cols / c->group_size;
    uint32_t top = (1u << c->bits) - 1u;
    uint8_t *codes = (uint8_t *)malloc((size_t)c->cols);
    for (int64_t r = begin; r < end; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            int64_t v0 = r * c->cols + g * c->group_size; /* first element of the group */
            float lo = (float)load_elem(c->w, c->w_type, v0), hi = lo;
            for (int i = 1; i < c->group_size; ++i) {
                float f = (float)load_elem(c->w, c->w_type, v0 + i);
                if (f < lo)
                    lo = f;
                if (f > hi)
                    hi = f;
            }
            float range = hi - lo;
            float scale_f32 = range / (float)top;
            store_elem(c->scales, c->w_type, r * groups + g, scale_f32);
            store_elem(c->biases, c->w_type, r * groups + g, lo); /* exact: lo is a value of w */
            float s = (float)load_elem(c->scales, c->w_type, r * groups + g);
            float b = (float)load_elem(c->biases, c->w_type, r * groups + g);
            for (int i = 0; i < c->group_size; ++i) {
                uint32_t code = 0;
                if (s != 0.0f) {
                    float d = (float)load_elem(c->w, c->w_type, v0 + i) - b;
                    float q = rintf(d / s);
                    if (q < 0.0f)
                        q = 0.0f;
                    if (q > (float)top)
                        q = (float)top;
                    code = (uint32_t)q;
                }
                codes[g * c->group_size + i] = (uint8_t)code;
            }
        }
        oracle_pack(codes, 1, c->cols, c->bits,
                    c->packed + r * oracle_words_per_row(c->cols, c->bits));
    }
    free(codes);
}

void oracle_quantize_typed(const void *w, int w_type, int64_t rows, int64_t cols,
                           int group_size, int bits, uint32_t *packed, void *scales,
                           void *biases, int nthreads)
{
    quant_ctx c = {w, w_type, rows, cols, group_size, bits, packed, scales, biases};
    parallel_for(rows, nthreads, quant_rows_range, &c);
}

void oracle_quantize(const uint16_t *w, int64_t rows, int64_t cols, int group_size,
                     int bits, uint32_t *packed, uint16_t *scales, uint16_t *biases,
                     int nthreads)
{
    oracle_quantize_typed(w, ORACLE_BF16, rows, cols, group_size, bits, packed, scales,
                          biases, nthreads);
}
