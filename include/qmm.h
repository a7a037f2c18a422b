/*
 * qmm.h -- C ABI of the GB300 (sm_103a) library for MLX grouped affine
 * quantization: dequantize, quantized_matmul and the rows gather-dequant.
 *
 * Packed format (nuvec_core quantized.rs, module doc; rlx-moshi
 * src/mlx_dequant.rs, `dequantize_affine` doc; spark_runtime
 * weights/mlx_int8.rs, module doc):
 *   - A weight [rows, cols] stores `bits`-bit codes (bits in 1..6 or 8), each
 *     row a little-endian bit stream packed into uint32 words: code j of a row
 *     sits at stream bits [j*bits, (j+1)*bits), least significant bit first,
 *     and stream bit i is bit (i mod 32) of word floor(i/32).  A row takes
 *     cols*bits/32 words; rows are contiguous (row pitch cols*bits/8 bytes).
 *     At 8 bits the low byte of a word is the first column.
 *   - One bf16 scale and one bf16 bias per group of `group_size` (32, 64 or
 *     128) consecutive codes of a row: scales and biases are bf16
 *     [rows, cols/group_size], row-major.
 *   - w = scale * code + bias.
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller (the library never
 *     frees caller memory, as spark_runtime's `MlxInt8Weight` leaves buffers
 *     to their owner).  Every pointer must be 16-byte aligned.  bf16 values
 *     are passed as their 16-bit patterns (uint16_t).
 *   - The only memory the library takes is stream-ordered scratch, from the
 *     current device's default memory pool, returned on the same stream by
 *     the same call: the split-K workspace of qmm_quantized_matmul (and of its
 *     fp32 form in qmm_quantized_matmul_typed) and the plan of
 *     qmm_gather_qmm's tensor-core form (see there).  Every other path
 *     allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and run on the current CUDA device.  Results follow
 *     stream order.
 *   - Arguments are checked on the host before anything is launched.  A bad
 *     argument returns QMM_ERR_INVALID_ARG, an unsupported dtype
 *     QMM_ERR_UNSUPPORTED, and nothing runs.  A failed launch returns
 *     QMM_ERR_CUDA.  qmm_last_error() then describes the failure.
 *   - An empty output (zero rows, M == 0, N == 0 or n == 0) is a valid no-op.
 *   - Outputs: QMM_F32 or QMM_BF16 (round to nearest even).
 *   - Other dtypes: the calls above take bf16 x, scales and biases (the
 *     pages' checkpoint format).  The *_typed calls at the end of this file
 *     take fp16 and fp32 as well, with MLX's promotion of x, scales and
 *     biases to one type (see qmm_promote_types).
 *
 * Thread safety: calls may come from several host threads; the last-error
 * message is per host thread.
 */
#ifndef QMM_H
#define QMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *qmm_stream_t;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1, /* shape, parameter, pointer or alignment rule broken */
    QMM_ERR_UNSUPPORTED = 2, /* output dtype not supported */
    QMM_ERR_CUDA = 3,        /* a CUDA call or launch failed */
    QMM_ERR_INDEX = 4,       /* qmm_rows met an index outside the table */
    QMM_ERR_TIMEOUT = 5      /* a bounded wait inside a kernel ran out */
} qmm_status;

/* Element types.  bf16 and fp16 values are passed as their 16-bit patterns. */
typedef enum { QMM_F32 = 0, QMM_BF16 = 1, QMM_F16 = 2 } qmm_dtype;

/*
 * qmm_dequantize -- out = dequant(W), contiguous [rows, cols].
 * (nuvec_core quantized.rs, `dequantize`: code * scale + bias; rlx-moshi
 *  src/mlx_dequant.rs, `dequantize_affine`; spark_runtime
 *  weights/mlx_int8.rs, `dequantize_to`.)
 *
 *   w       uint32 [rows, cols*bits/32]
 *   scales  bf16   [rows, cols/group_size]
 *   biases  bf16   [rows, cols/group_size]
 *   out     [rows, cols] of out_dtype
 *
 * Each element is fp32 scale*code + bias (the product is exact, one rounding
 * at the add); QMM_F32 stores it as is, QMM_BF16 rounds it to nearest even.
 * Rules: bits in {1,2,3,4,5,6,8}; group_size in {32,64,128}; cols > 0 and a
 * multiple of group_size; rows >= 0.
 */
qmm_status qmm_dequantize(const uint32_t *w, const uint16_t *scales,
                          const uint16_t *biases, int64_t rows, int64_t cols,
                          int group_size, int bits, void *out,
                          qmm_dtype out_dtype, qmm_stream_t stream);

/*
 * qmm_quantize -- packed codes, scales and biases of a bf16 weight, in the
 * format above.  (nuvec_core quantized.rs, module doc: a value w is stored as
 * round((w - bias) / scale), clamped to [0, 2^bits - 1]; `dequantize` doc:
 * bias = the group minimum.)
 *
 *   w       bf16 [rows, cols]
 *   packed  uint32 [rows, cols*bits/32]
 *   scales  bf16   [rows, cols/group_size]
 *   biases  bf16   [rows, cols/group_size]
 *
 * Per group: bias = the minimum (exact); scale = (max - min) / (2^bits - 1)
 * in fp32, rounded to nearest even bf16 (the pages do not give the scale:
 * this is the plain min-max reading, not a claim of MLX's exact rounding);
 * code = round half to even of (w - bias) / scale with the stored bf16 scale
 * and bias, each step one IEEE fp32 operation, clamped.  A zero scale gives
 * every code 0.  Rules: bits and group_size as above; cols > 0 and a multiple
 * of group_size; rows >= 0.
 */
qmm_status qmm_quantize(const uint16_t *w, int64_t rows, int64_t cols, int group_size, int bits,
                        uint32_t *packed, uint16_t *scales, uint16_t *biases,
                        qmm_stream_t stream);

/*
 * qmm_quantized_matmul -- y = x . dequant(W)^T (transpose = 1) or
 * y = x . dequant(W) (transpose = 0), without materialising dequant(W).
 * (nuvec_core quantized.rs, `quantized_matmul`; maya2_mlx quant.py, `mm`,
 *  which always passes transpose=True for an [out, in] weight; spark_runtime
 *  weights/mlx_int8.rs, `gemv` and `gemm`.)
 *
 *   x       bf16 [M, K]   (a 1-D x is M = 1; flatten batch dims into M)
 *   transpose = 1: w uint32 [N, K*bits/32], scales/biases bf16 [N, K/group_size]
 *   transpose = 0: w uint32 [K, N*bits/32], scales/biases bf16 [K, N/group_size]
 *   y       [M, N] of y_dtype
 *
 * Accumulation is fp32 over weights rounded once to bf16; every output is
 * within 8e-3 * sum_k |x[m,k] * w[k,n]| + 1e-6 of the exact product.
 * Rules: bits and group_size as above; K > 0; the packed (last) axis of W a
 * multiple of group_size (K when transpose, N otherwise); M, N >= 0;
 * transpose in {0, 1}.  M <= 16 runs the decode kernel, larger M the
 * tensor-core (tcgen05) kernel.
 *
 * Split-K: when M > 16 gives fewer 256 x 256 output tiles than half the SMs,
 * the K range of each tile is split over several blocks; their fp32 partials
 * go to a workspace of splits * M * N * 4 bytes (never more than one tile
 * per SM, about 40 MB on a GB300) and a second kernel adds them in a fixed
 * order, so results repeat bit for bit.  The workspace comes from
 * cudaMallocAsync on `stream` and goes back with cudaFreeAsync on `stream`
 * (under stream capture, as graph allocation and free nodes).  If it cannot
 * be had, the call runs without split-K.
 */
qmm_status qmm_quantized_matmul(const uint16_t *x, int64_t M, const uint32_t *w,
                                const uint16_t *scales, const uint16_t *biases,
                                int64_t N, int64_t K, int transpose,
                                int group_size, int bits, void *y,
                                qmm_dtype y_dtype, qmm_stream_t stream);

/*
 * qmm_gather_qmm -- quantized matmuls of gathered batches (mixture-of-experts
 * layers): output batch b is x[lhs_indices[b]] . dequant(w[rhs_indices[b]])^T
 * (transpose = 1) or without the transpose.
 * (nuvec_core quantized.rs, `gather_qmm`: the indices address the flattened
 *  batch dimensions of x and w; either defaults to every batch of its operand
 *  in order; sorted_indices promises sorted rhs_indices, so that each weight
 *  batch can be walked once.)
 *
 *   x            bf16 [x_batches, M, K]
 *   w, scales, biases  w_batches weights one after another, each laid out
 *                as qmm_quantized_matmul's (transpose = 1: w [N, K*bits/32],
 *                scales/biases [N, K/group_size]; transpose = 0:
 *                [K, N*bits/32] and [K, N/group_size])
 *   lhs_indices  uint32 [batches] on the device, or NULL: batch b uses x[b]
 *   rhs_indices  uint32 [batches] on the device, or NULL: batch b uses w[b]
 *   y            [batches, M, N] of y_dtype
 *
 * The index arrays are the broadcast of the caller's index shapes, flattened
 * (the caller broadcasts).  NULL indices need x_batches (resp. w_batches)
 * equal to batches.  An index past its operand gives a batch of zeros and is
 * reported by qmm_get_device_error as QMM_ERR_INDEX.  sorted_indices = 1
 * with M == 1, NULL lhs_indices and non-decreasing rhs_indices lets one block
 * stream each weight tile once for all the batches that use it; if the
 * promise is false the results are wrong (nothing is read out of bounds).
 * Same tolerance as qmm_quantized_matmul.  The kernels are the decode ones
 * (M is walked in 8- or 16-row passes), launched without programmatic
 * dependent launch: the indices may come from the previous kernel.  With
 * sorted indices as above, transpose = 1 and 32 or more batches per weight
 * batch on average (prefill-sized runs), the call instead runs a small
 * planning kernel (each weight batch's run of rows, cut into 256-row tiles)
 * and the tensor-core GEMM over those tiles; it then takes a stream-ordered
 * allocation of 4 * (3 * tiles + 1) bytes for the plan, as the split-K
 * workspace of qmm_quantized_matmul does.
 */
qmm_status qmm_gather_qmm(const uint16_t *x, int64_t x_batches, int64_t M, const uint32_t *w,
                          const uint16_t *scales, const uint16_t *biases, int64_t w_batches,
                          int64_t N, int64_t K, const uint32_t *lhs_indices,
                          const uint32_t *rhs_indices, int64_t batches, int transpose,
                          int group_size, int bits, int sorted_indices, void *y,
                          qmm_dtype y_dtype, qmm_stream_t stream);

/*
 * qmm_gemv_gate_up -- the two projections of a gated feed-forward block from
 * one x in one launch: y_gate = x . dequant(W_gate)^T, y_up = x . dequant(W_up)^T.
 * (spark_runtime weights/mlx_int8.rs, `gemv_gate_up`: both weights share
 *  out and in features and group size, and x is read for both.)
 *
 *   x                 bf16 [M, K], 1 <= M <= 16
 *   w_gate, w_up      uint32 [N, K*bits/32] each (transposed layout)
 *   scales_gate, biases_gate, scales_up, biases_up  bf16 [N, K/group_size]
 *   y_gate, y_up      [M, N] of y_dtype
 *
 * Rules: as qmm_quantized_matmul with transpose = 1, and K a multiple of 128.
 * Same tolerance.  Launched like the decode kernel (programmatic dependent
 * launch when QMM_LAUNCH_PDL is set).
 */
qmm_status qmm_gemv_gate_up(const uint16_t *x, int64_t M, const uint32_t *w_gate,
                            const uint16_t *scales_gate, const uint16_t *biases_gate,
                            const uint32_t *w_up, const uint16_t *scales_up,
                            const uint16_t *biases_up, int64_t N, int64_t K, int group_size,
                            int bits, void *y_gate, void *y_up, qmm_dtype y_dtype,
                            qmm_stream_t stream);

/*
 * qmm_gemv_silu_gate -- y = dequant(W) . (silu(gate) * up) (+ resid), the
 * down projection of a gated feed-forward block with its input formed inside
 * the kernel: no intermediate [M, K] buffer and no separate launch.
 * (spark_runtime weights/mlx_int8.rs, `gemv_silu_gate` and
 *  `gemv_silu_gate_resid`: y[n] = x_resid[n] + sum_k W[n, k] *
 *  (silu(gate[k]) * up[k]).)
 *
 *   gate, up  bf16 [M, K], 1 <= M <= 8
 *   w         uint32 [N, K*bits/32], scales/biases bf16 [N, K/group_size]
 *   resid     bf16 [M, N] added to y before its rounding, or NULL
 *   y         [M, N] of y_dtype
 *
 * silu(g) = g / (1 + exp(-g)) and its product with up are formed in fp32 and
 * rounded once to bf16 before the contraction (fp32 accumulation, as
 * qmm_quantized_matmul).  Every output is within
 * 8e-3 * (sum_k |x[m,k] * w[n,k]| + |resid[m,n]|) + 1e-6 of the exact value,
 * x being the exact silu(gate) * up.  Rules: as qmm_gemv_gate_up for the
 * weight; K a multiple of 128.
 */
qmm_status qmm_gemv_silu_gate(const uint16_t *gate, const uint16_t *up, int64_t M,
                              const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                              int64_t N, int64_t K, int group_size, int bits,
                              const uint16_t *resid, void *y, qmm_dtype y_dtype,
                              qmm_stream_t stream);

/*
 * qmm_quantized_matmul_noalloc -- qmm_quantized_matmul for callers that cannot
 * allocate device memory while they run: code that owns every byte of the
 * device through its own allocator, or that records work where no allocation
 * call may appear.  (The pages have no counterpart: MLX allocates its
 * outputs and scratch through its own allocator.)
 *
 * Same arguments, checks and kernels as qmm_quantized_matmul, and results
 * within the same tolerance.  The only difference: the split-K partials
 * (M > 16 with few output tiles) go to a fixed 24 MiB scratch array inside
 * the library instead of a stream-ordered allocation, so the call allocates
 * and frees nothing.  Every GPU that loads the library holds that array until
 * the process exits.
 *   - When the usual split would need more than 24 MiB of partials
 *     (splits * M * N * 4 bytes), K is split fewer ways, as many as fit, or
 *     not at all; the sums then run in another order than
 *     qmm_quantized_matmul's (same tolerance, not the same bits).
 *   - The first call on each device looks up the array's device address
 *     (set-up, once per device, with that device current); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind (nothing in it needs to start at zero).  Calls whose kernels
 *     overlap on the GPU -- on different streams without ordering between
 *     them -- race on it and give wrong results; keep them ordered.
 */
qmm_status qmm_quantized_matmul_noalloc(const uint16_t *x, int64_t M, const uint32_t *w,
                                        const uint16_t *scales, const uint16_t *biases,
                                        int64_t N, int64_t K, int transpose,
                                        int group_size, int bits, void *y,
                                        qmm_dtype y_dtype, qmm_stream_t stream);

/*
 * qmm_rows -- out[i, :] = dequant(W[idx[i], :]) for i < n: an embedding
 * lookup that dequantizes only the gathered rows in one pass.
 * (maya2_mlx quant.py, `rows`: dequantize(q[idx], scales[idx], biases[idx]).)
 *
 *   w, scales, biases  the table [table_rows, cols], laid out as for
 *                      qmm_dequantize
 *   idx     uint32 [n] device array of row indices (duplicates allowed)
 *   out     [n, cols] of out_dtype
 *
 * An index >= table_rows gives a zero output row and records QMM_ERR_INDEX in
 * the device error word (read by qmm_get_device_error); nothing faults.
 */
qmm_status qmm_rows(const uint32_t *w, const uint16_t *scales,
                    const uint16_t *biases, int64_t table_rows, int64_t cols,
                    const uint32_t *idx, int64_t n, int group_size, int bits,
                    void *out, qmm_dtype out_dtype, qmm_stream_t stream);

/*
 * Launch options for the calls this host thread makes from now on (the pages
 * have no counterpart: this is a property of how kernels are launched on
 * this GPU).  Returns the previous flags.
 *
 *   QMM_LAUNCH_PDL  Launch the decode kernels (qmm_quantized_matmul with
 *                   M <= 16) with programmatic dependent launch: a kernel may
 *                   start, and begin streaming its packed weight, scales and
 *                   biases, before the previous kernel in the stream has
 *                   finished; it reads x and writes y only after that kernel
 *                   has completed.  Only use it when the weights are not
 *                   written by the kernel immediately before the call in the
 *                   same stream (model weights normally are not).  Default
 *                   off.
 * Unknown bits return QMM_ERR_INVALID_ARG through qmm_last_error and are
 * ignored; the previous flags are still returned.
 */
#define QMM_LAUNCH_PDL 1u
unsigned qmm_set_launch_flags(unsigned flags);

/*
 * qmm_set_wait_limit -- after how many unsuccessful polls of one of its own
 * barriers a kernel gives up (the pages have no counterpart: it bounds the
 * waits of this library's kernels on their own copies and stages).  Applies
 * to the calls this host thread makes from now on; returns the previous
 * setting.  0 restores the default (2^24 polls, each suspended for at most a
 * few hundred nanoseconds: seconds in all); 1 gives up at the first poll that
 * finds the barrier incomplete.
 *
 * A wait that runs out makes the kernel stop early: it records
 * QMM_ERR_TIMEOUT in the device error word (qmm_get_device_error), waits
 * for the copies it has in flight, frees what it holds and returns; the
 * outputs of that call are then undefined (the split-K matmul writes NaN).
 * A small limit makes waits run out on purpose, which is how the timeout
 * path is tested; nothing faults or hangs.
 */
uint32_t qmm_set_wait_limit(uint32_t polls);

/* The message for the last non-OK status returned on this host thread
 * (empty string if none).  The pointer stays valid until the next call. */
const char *qmm_last_error(void);

/*
 * Synchronizes `stream`, then reads and clears the current device's error
 * word: QMM_ERR_INDEX if a qmm_rows index was outside its table,
 * QMM_ERR_TIMEOUT if a bounded wait in a kernel ran out (the kernel then
 * stops early and its output is incomplete), QMM_ERR_CUDA if the
 * synchronization itself failed, else QMM_OK.
 */
qmm_status qmm_get_device_error(qmm_stream_t stream);

/* ------------------------------------------------------------- dtypes ----
 * (nuvec_core quantized.rs: `quantize` takes float16, bfloat16 or float32
 * weights and returns scales and biases in the weights' dtype; `dequantize`
 * returns the scales' dtype; `quantized_matmul` promotes x, scales and biases
 * to one floating-point type and computes in it.)  These calls take the same
 * pointers as the bf16 calls above, typed by a qmm_dtype argument; an fp32
 * buffer holds 4-byte values, the others 16-bit patterns.  Scales and biases
 * share one dtype. */

/*
 * qmm_promote_types -- *out = the type that a and b promote to: the
 * narrowest of bf16, f16 and f32 that holds every value of both exactly
 * (a itself when a == b; f32 otherwise, since bf16 and f16 each hold values
 * the other lacks).  QMM_ERR_UNSUPPORTED for an unknown dtype.
 */
qmm_status qmm_promote_types(qmm_dtype a, qmm_dtype b, qmm_dtype *out);

/*
 * qmm_dequantize_typed / qmm_rows_typed -- qmm_dequantize and qmm_rows with
 * scales and biases of sb_dtype.  Each element is scale * code + bias
 * rounded once to fp32 (for 16-bit scales the product is exact), stored as
 * is (out_dtype QMM_F32) or rounded to nearest even in the scales' dtype
 * (out_dtype == sb_dtype); other output dtypes give QMM_ERR_UNSUPPORTED.
 * Rules, ownership and errors as qmm_dequantize / qmm_rows.
 */
qmm_status qmm_dequantize_typed(const uint32_t *w, const void *scales, const void *biases,
                                qmm_dtype sb_dtype, int64_t rows, int64_t cols, int group_size,
                                int bits, void *out, qmm_dtype out_dtype, qmm_stream_t stream);

qmm_status qmm_rows_typed(const uint32_t *w, const void *scales, const void *biases,
                          qmm_dtype sb_dtype, int64_t table_rows, int64_t cols,
                          const uint32_t *idx, int64_t n, int group_size, int bits, void *out,
                          qmm_dtype out_dtype, qmm_stream_t stream);

/*
 * qmm_quantize_typed -- qmm_quantize of a weight of w_dtype; scales and
 * biases [rows, cols/group_size] are written in w_dtype: the bias (the group
 * minimum) exactly, the scale (max - min) / (2^bits - 1) computed in fp32 and
 * rounded to nearest even for the 16-bit types.  Codes, rules and errors as
 * qmm_quantize.
 */
qmm_status qmm_quantize_typed(const void *w, qmm_dtype w_dtype, int64_t rows, int64_t cols,
                              int group_size, int bits, uint32_t *packed, void *scales,
                              void *biases, qmm_stream_t stream);

/*
 * qmm_quantized_matmul_typed -- qmm_quantized_matmul with x of x_dtype and
 * scales and biases of sb_dtype, computed in D = the promotion of the two:
 *   D = bf16: the bf16 kernels of qmm_quantized_matmul;
 *   D = f16:  the same kernels in fp16 (weights rounded once to fp16, fp16
 *             tensor-core products, fp32 accumulation);
 *   D = f32:  fp32 on the CUDA cores (weights fp32 fma(scale, code, bias),
 *             x widened exactly, fp32 products and sums), for any mix that
 *             promotes to f32; x rows at most 65535 * 128.
 * y_dtype is QMM_F32 or D.  Every output is within 8e-3 * sum_k |x w| + 1e-6
 * of the exact product (D = f32 is far inside it: the sums' own rounding).
 * Shapes, rules and errors as qmm_quantized_matmul; the D = f32 path splits K
 * over blocks with a stream-ordered workspace the same way.
 */
qmm_status qmm_quantized_matmul_typed(const void *x, qmm_dtype x_dtype, int64_t M,
                                      const uint32_t *w, const void *scales, const void *biases,
                                      qmm_dtype sb_dtype, int64_t N, int64_t K, int transpose,
                                      int group_size, int bits, void *y, qmm_dtype y_dtype,
                                      qmm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
