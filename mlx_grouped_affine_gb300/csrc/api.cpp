// The C ABI: argument checks, dispatch to the kernels, status codes and the
// per-thread last-error message.
//
// The checks mirror the pages' rules: group size 32, 64 or 128 and bit width
// 1-6 or 8 (nuvec_core quantized.rs, `check_params`); the grouped axis a
// multiple of the group size and the packed axis equal to cols*bits/32
// (rlx-moshi src/mlx_dequant.rs, `dequantize_affine`; spark_runtime
// weights/mlx_int8.rs, `load`).  The library owns no buffer: every pointer is
// the caller's (spark_runtime `MlxInt8Weight`, `release`).
#include "qmm.h"
#include "internal.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>

namespace {

thread_local char g_last_error[512] = "";
thread_local unsigned g_launch_flags = 0;
thread_local uint32_t g_wait_limit = 0;  // 0: the default

qmm_status fail(qmm_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

qmm_status cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return QMM_OK;
  return fail(QMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qmm_status check_params(const char *op, int group_size, int bits) {
  if (group_size != 32 && group_size != 64 && group_size != 128)
    return fail(QMM_ERR_INVALID_ARG, "%s: group size %d is not supported (32, 64 or 128)", op,
                group_size);
  if (bits < 1 || bits > 8 || bits == 7)
    return fail(QMM_ERR_INVALID_ARG, "%s: %d bits are not supported (1, 2, 3, 4, 5, 6 or 8)",
                op, bits);
  return QMM_OK;
}

qmm_status check_dtype(const char *op, qmm_dtype d) {
  if (d != QMM_F32 && d != QMM_BF16)
    return fail(QMM_ERR_UNSUPPORTED, "%s: output dtype %d is not supported (QMM_F32, QMM_BF16)",
                op, static_cast<int>(d));
  return QMM_OK;
}

bool known_dtype(qmm_dtype d) { return d == QMM_F32 || d == QMM_BF16 || d == QMM_F16; }

const char *dtype_name(qmm_dtype d) {
  return d == QMM_F32 ? "f32" : d == QMM_BF16 ? "bf16" : d == QMM_F16 ? "f16" : "unknown";
}

// An output of a typed call: fp32, or the type the call computes in.
qmm_status check_out_dtype(const char *op, qmm_dtype out, qmm_dtype compute) {
  if (!known_dtype(out) || (out != QMM_F32 && out != compute))
    return fail(QMM_ERR_UNSUPPORTED, "%s: output dtype %d is not supported here (QMM_F32 or %s)",
                op, static_cast<int>(out), dtype_name(compute));
  return QMM_OK;
}

// The narrowest of bf16, f16 and f32 that holds every value of a and of b
// (bf16 and f16 each hold values the other lacks, so together they need f32).
qmm_dtype promote(qmm_dtype a, qmm_dtype b) {
  if (a == b) return a;
  return QMM_F32;
}

// The packed weight [rows, cols]: grouped axis, pointers, alignment.
qmm_status check_weight(const char *op, const uint32_t *w, const uint16_t *scales,
                        const uint16_t *biases, int64_t rows, int64_t cols, int group_size) {
  if (rows < 0) return fail(QMM_ERR_INVALID_ARG, "%s: negative row count %lld", op, (long long)rows);
  if (cols <= 0 || cols % group_size != 0)
    return fail(QMM_ERR_INVALID_ARG,
                "%s: the grouped axis (%lld) must be positive and a multiple of group size %d", op,
                (long long)cols, group_size);
  if (cols > (int64_t(1) << 40) || rows > (int64_t(1) << 40))
    return fail(QMM_ERR_INVALID_ARG, "%s: weight [%lld, %lld] is too large", op, (long long)rows,
                (long long)cols);
  if (!w || !scales || !biases)
    return fail(QMM_ERR_INVALID_ARG, "%s: null weight, scales or biases pointer", op);
  if (!aligned16(w) || !aligned16(scales) || !aligned16(biases))
    return fail(QMM_ERR_INVALID_ARG, "%s: weight, scales and biases must be 16-byte aligned", op);
  return QMM_OK;
}

// ------------------------------------------------ shared implementations ----
// The bf16 entry points are the typed ones with bf16 operands; `op` names the
// entry point the caller used, for the last-error message.

// dequantize (gather false) or rows (gather true: n rows at indices idx).
qmm_status dequantize_impl(const char *op, const uint32_t *w, const void *scales,
                           const void *biases, qmm_dtype sb_dtype, int64_t rows, int64_t cols,
                           bool gather, const uint32_t *idx, int64_t n, int group_size, int bits,
                           void *out, qmm_dtype out_dtype, qmm_stream_t stream) {
  qmm_status st;
  if ((st = check_params(op, group_size, bits)) != QMM_OK) return st;
  if (!known_dtype(sb_dtype))
    return fail(QMM_ERR_UNSUPPORTED, "%s: unknown scale dtype %d", op, static_cast<int>(sb_dtype));
  if ((st = check_out_dtype(op, out_dtype, sb_dtype)) != QMM_OK) return st;
  const uint16_t *s16 = static_cast<const uint16_t *>(scales);
  const uint16_t *b16 = static_cast<const uint16_t *>(biases);
  if ((st = check_weight(op, w, s16, b16, rows, cols, group_size)) != QMM_OK) return st;
  const int64_t out_rows = gather ? n : rows;
  if (gather && n < 0) return fail(QMM_ERR_INVALID_ARG, "%s: negative index count %lld", op, (long long)n);
  if (out_rows == 0) return QMM_OK;
  if (gather && (!idx || !aligned16(idx)))
    return fail(QMM_ERR_INVALID_ARG, "%s: indices must be a non-null 16-byte aligned pointer", op);
  if (!out || !aligned16(out))
    return fail(QMM_ERR_INVALID_ARG, "%s: output must be a non-null 16-byte aligned pointer", op);
  qmm::PackedWeight pw{w, s16, b16, rows, cols, group_size, bits, static_cast<int>(sb_dtype)};
  return cuda_status(qmm::launch_dequantize(pw, gather ? idx : nullptr, out_rows, out,
                                            static_cast<int>(out_dtype),
                                            reinterpret_cast<cudaStream_t>(stream)),
                     op);
}

qmm_status quantize_impl(const char *op, const void *w, qmm_dtype w_dtype, int64_t rows,
                         int64_t cols, int group_size, int bits, uint32_t *packed, void *scales,
                         void *biases, qmm_stream_t stream) {
  qmm_status st;
  if ((st = check_params(op, group_size, bits)) != QMM_OK) return st;
  if (!known_dtype(w_dtype))
    return fail(QMM_ERR_UNSUPPORTED, "%s: unknown weight dtype %d", op, static_cast<int>(w_dtype));
  if (rows < 0) return fail(QMM_ERR_INVALID_ARG, "%s: negative row count %lld", op, (long long)rows);
  if (cols <= 0 || cols % group_size != 0)
    return fail(QMM_ERR_INVALID_ARG, "%s: cols (%lld) must be a positive multiple of group_size %d",
                op, (long long)cols, group_size);
  if (rows == 0) return QMM_OK;
  if (!w || !aligned16(w) || !packed || !aligned16(packed) || !scales || !aligned16(scales) ||
      !biases || !aligned16(biases))
    return fail(QMM_ERR_INVALID_ARG, "%s: every pointer must be non-null and 16-byte aligned", op);
  return cuda_status(qmm::launch_quantize(w, static_cast<int>(w_dtype), rows, cols, group_size,
                                          bits, packed, scales, biases,
                                          reinterpret_cast<cudaStream_t>(stream)),
                     op);
}

// The checks of a quantized matmul, shared with the no-allocation entry
// point.  On QMM_OK, *work is false for an empty product (nothing to launch).
qmm_status check_matmul(const char *op, const void *x, qmm_dtype x_dtype, int64_t M,
                        const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                        qmm_dtype sb_dtype, int64_t N, int64_t K, int transpose, int group_size,
                        int bits, const void *y, qmm_dtype y_dtype, bool *work) {
  qmm_status st;
  *work = false;
  if ((st = check_params(op, group_size, bits)) != QMM_OK) return st;
  if (!known_dtype(x_dtype) || !known_dtype(sb_dtype))
    return fail(QMM_ERR_UNSUPPORTED, "%s: unknown x or scale dtype (%d, %d)", op,
                static_cast<int>(x_dtype), static_cast<int>(sb_dtype));
  if ((st = check_out_dtype(op, y_dtype, promote(x_dtype, sb_dtype))) != QMM_OK) return st;
  if (transpose != 0 && transpose != 1)
    return fail(QMM_ERR_INVALID_ARG, "%s: transpose must be 0 or 1, got %d", op, transpose);
  if (M < 0 || N < 0) return fail(QMM_ERR_INVALID_ARG, "%s: negative M or N", op);
  if (K <= 0) return fail(QMM_ERR_INVALID_ARG, "%s: K must be positive, got %lld", op, (long long)K);
  // Stored weight: [N, K] when transposed, [K, N] otherwise; the packed,
  // grouped axis is the stored last one.
  const int64_t rows = transpose ? N : K, cols = transpose ? K : N;
  if (transpose || N > 0) {
    if ((st = check_weight(op, w, scales, biases, rows, cols, group_size)) != QMM_OK) return st;
  }
  if (M == 0 || N == 0) return QMM_OK;
  if (!x || !aligned16(x))
    return fail(QMM_ERR_INVALID_ARG, "%s: x must be a non-null 16-byte aligned pointer", op);
  if (!y || !aligned16(y))
    return fail(QMM_ERR_INVALID_ARG, "%s: y must be a non-null 16-byte aligned pointer", op);
  if (M > (int64_t(1) << 31) || K > (int64_t(1) << 31) || N > (int64_t(1) << 31))
    return fail(QMM_ERR_INVALID_ARG, "%s: M, N and K must each be below 2^31", op);
  if (promote(x_dtype, sb_dtype) == QMM_F32 && M > int64_t(65535) * 128)
    return fail(QMM_ERR_INVALID_ARG, "%s: the fp32 path takes at most %lld rows of x", op,
                (long long)(int64_t(65535) * 128));
  *work = true;
  return QMM_OK;
}

qmm_status matmul_impl(const char *op, const void *x, qmm_dtype x_dtype, int64_t M,
                       const uint32_t *w, const void *scales, const void *biases,
                       qmm_dtype sb_dtype, int64_t N, int64_t K, int transpose, int group_size,
                       int bits, void *y, qmm_dtype y_dtype, qmm_stream_t stream) {
  const uint16_t *s16 = static_cast<const uint16_t *>(scales);
  const uint16_t *b16 = static_cast<const uint16_t *>(biases);
  bool work = false;
  const qmm_status st = check_matmul(op, x, x_dtype, M, w, s16, b16, sb_dtype, N, K, transpose,
                                     group_size, bits, y, y_dtype, &work);
  if (st != QMM_OK || !work) return st;
  const int64_t rows = transpose ? N : K, cols = transpose ? K : N;
  qmm::PackedWeight pw{w, s16, b16, rows, cols, group_size, bits, static_cast<int>(sb_dtype)};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const qmm_dtype d = promote(x_dtype, sb_dtype);
  const bool y16 = y_dtype != QMM_F32;
  const uint16_t *x16 = static_cast<const uint16_t *>(x);
  cudaError_t e;
  if (d == QMM_BF16)
    e = M <= 16 ? qmm::launch_gemv(x16, M, pw, transpose != 0, y, y16, s)
                : qmm::launch_gemm(x16, M, pw, transpose != 0, y, y16, s);
  else if (d == QMM_F16)
    e = M <= 16 ? qmm::launch_gemv_f16(x16, M, pw, transpose != 0, y, y16, s)
                : qmm::launch_gemm_f16(x16, M, pw, transpose != 0, y, y16, s);
  else
    e = qmm::launch_mm_f32(x, static_cast<int>(x_dtype), M, pw, transpose != 0,
                           static_cast<float *>(y), s);
  return cuda_status(e, op);
}

}  // namespace

namespace qmm {
unsigned launch_flags() { return g_launch_flags; }
uint32_t wait_limit() { return g_wait_limit ? g_wait_limit : kDefaultWaitLimit; }
}  // namespace qmm

extern "C" {

const char *qmm_last_error(void) { return g_last_error; }

uint32_t qmm_set_wait_limit(uint32_t polls) {
  const uint32_t prev = g_wait_limit;
  g_wait_limit = polls;
  return prev;
}

unsigned qmm_set_launch_flags(unsigned flags) {
  const unsigned prev = g_launch_flags;
  if (flags & ~QMM_LAUNCH_PDL) {
    fail(QMM_ERR_INVALID_ARG, "qmm_set_launch_flags: unknown flag bits 0x%x ignored",
         flags & ~QMM_LAUNCH_PDL);
    flags &= QMM_LAUNCH_PDL;
  }
  g_launch_flags = flags;
  return prev;
}

qmm_status qmm_dequantize(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                          int64_t rows, int64_t cols, int group_size, int bits, void *out,
                          qmm_dtype out_dtype, qmm_stream_t stream) {
  return dequantize_impl("qmm_dequantize", w, scales, biases, QMM_BF16, rows, cols, false, nullptr,
                         0, group_size, bits, out, out_dtype, stream);
}

qmm_status qmm_rows(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                    int64_t table_rows, int64_t cols, const uint32_t *idx, int64_t n,
                    int group_size, int bits, void *out, qmm_dtype out_dtype,
                    qmm_stream_t stream) {
  return dequantize_impl("qmm_rows", w, scales, biases, QMM_BF16, table_rows, cols, true, idx, n,
                         group_size, bits, out, out_dtype, stream);
}

qmm_status qmm_quantized_matmul(const uint16_t *x, int64_t M, const uint32_t *w,
                                const uint16_t *scales, const uint16_t *biases, int64_t N,
                                int64_t K, int transpose, int group_size, int bits, void *y,
                                qmm_dtype y_dtype, qmm_stream_t stream) {
  return matmul_impl("qmm_quantized_matmul", x, QMM_BF16, M, w, scales, biases, QMM_BF16, N, K,
                     transpose, group_size, bits, y, y_dtype, stream);
}

qmm_status qmm_gather_qmm(const uint16_t *x, int64_t x_batches, int64_t M, const uint32_t *w,
                          const uint16_t *scales, const uint16_t *biases, int64_t w_batches,
                          int64_t N, int64_t K, const uint32_t *lhs_indices,
                          const uint32_t *rhs_indices, int64_t batches, int transpose,
                          int group_size, int bits, int sorted_indices, void *y,
                          qmm_dtype y_dtype, qmm_stream_t stream) {
  const char *op = "qmm_gather_qmm";
  qmm_status st;
  if ((st = check_params(op, group_size, bits)) != QMM_OK) return st;
  if ((st = check_dtype(op, y_dtype)) != QMM_OK) return st;
  if (transpose != 0 && transpose != 1)
    return fail(QMM_ERR_INVALID_ARG, "%s: transpose must be 0 or 1, got %d", op, transpose);
  if (sorted_indices != 0 && sorted_indices != 1)
    return fail(QMM_ERR_INVALID_ARG, "%s: sorted_indices must be 0 or 1, got %d", op, sorted_indices);
  if (M < 0 || N < 0 || batches < 0)
    return fail(QMM_ERR_INVALID_ARG, "%s: negative M, N or batch count", op);
  if (K <= 0) return fail(QMM_ERR_INVALID_ARG, "%s: K must be positive, got %lld", op, (long long)K);
  if (x_batches < 1 || w_batches < 1)
    return fail(QMM_ERR_INVALID_ARG, "%s: x and w need at least one batch each", op);
  if (!lhs_indices && x_batches != batches)
    return fail(QMM_ERR_INVALID_ARG,
                "%s: without lhs_indices x must hold one batch per output batch (%lld, not %lld)",
                op, (long long)batches, (long long)x_batches);
  if (!rhs_indices && w_batches != batches)
    return fail(QMM_ERR_INVALID_ARG,
                "%s: without rhs_indices w must hold one batch per output batch (%lld, not %lld)",
                op, (long long)batches, (long long)w_batches);
  const int64_t rows = transpose ? N : K, cols = transpose ? K : N;
  if (transpose || N > 0) {
    // One weight batch is [rows, cols]; all of them are checked as one table.
    if ((st = check_weight(op, w, scales, biases, rows, cols, group_size)) != QMM_OK) return st;
  }
  if (M == 0 || N == 0 || batches == 0) return QMM_OK;
  if (!x || !aligned16(x))
    return fail(QMM_ERR_INVALID_ARG, "%s: x must be a non-null 16-byte aligned pointer", op);
  if (!y || !aligned16(y))
    return fail(QMM_ERR_INVALID_ARG, "%s: y must be a non-null 16-byte aligned pointer", op);
  if ((lhs_indices && !aligned16(lhs_indices)) || (rhs_indices && !aligned16(rhs_indices)))
    return fail(QMM_ERR_INVALID_ARG, "%s: index arrays must be 16-byte aligned", op);
  const int64_t lim = int64_t(1) << 31;
  if (M >= lim || K >= lim || N >= lim || batches >= lim || x_batches >= lim || w_batches >= lim ||
      x_batches * M * K >= (int64_t(1) << 62) || w_batches * rows >= lim)
    return fail(QMM_ERR_INVALID_ARG, "%s: sizes out of range (each below 2^31, w_batches*rows too)", op);
  qmm::PackedWeight pw{w, scales, biases, rows, cols, group_size, bits};
  cudaError_t e = qmm::launch_gather(x, x_batches, M, pw, w_batches, lhs_indices, rhs_indices,
                                     batches, transpose != 0, sorted_indices != 0, y,
                                     y_dtype == QMM_BF16, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(e, op);
}

qmm_status qmm_quantize(const uint16_t *w, int64_t rows, int64_t cols, int group_size, int bits,
                        uint32_t *packed, uint16_t *scales, uint16_t *biases,
                        qmm_stream_t stream) {
  return quantize_impl("qmm_quantize", w, QMM_BF16, rows, cols, group_size, bits, packed, scales,
                       biases, stream);
}

// Checks shared by the fused decode GEMVs: a transposed weight [N, K] with K
// a multiple of 128, 1 <= M <= max_m.
static qmm_status check_fused(const char *op, int64_t M, int64_t max_m, const uint32_t *w,
                              const uint16_t *scales, const uint16_t *biases, int64_t N,
                              int64_t K, int group_size, int bits, qmm_dtype y_dtype) {
  qmm_status st;
  if ((st = check_params(op, group_size, bits)) != QMM_OK) return st;
  if ((st = check_dtype(op, y_dtype)) != QMM_OK) return st;
  if (M < 0 || N < 0) return fail(QMM_ERR_INVALID_ARG, "%s: negative M or N", op);
  if (M > max_m)
    return fail(QMM_ERR_INVALID_ARG, "%s: M is at most %lld, got %lld", op, (long long)max_m,
                (long long)M);
  if (K <= 0 || K % 128 != 0 || K >= (int64_t(1) << 31))
    return fail(QMM_ERR_INVALID_ARG, "%s: K must be a positive multiple of 128, got %lld", op,
                (long long)K);
  if (N >= (int64_t(1) << 31)) return fail(QMM_ERR_INVALID_ARG, "%s: N must be below 2^31", op);
  return check_weight(op, w, scales, biases, N, K, group_size);
}

qmm_status qmm_gemv_gate_up(const uint16_t *x, int64_t M, const uint32_t *w_gate,
                            const uint16_t *scales_gate, const uint16_t *biases_gate,
                            const uint32_t *w_up, const uint16_t *scales_up,
                            const uint16_t *biases_up, int64_t N, int64_t K, int group_size,
                            int bits, void *y_gate, void *y_up, qmm_dtype y_dtype,
                            qmm_stream_t stream) {
  const char *op = "qmm_gemv_gate_up";
  qmm_status st;
  if ((st = check_fused(op, M, 16, w_gate, scales_gate, biases_gate, N, K, group_size, bits,
                        y_dtype)) != QMM_OK)
    return st;
  if ((st = check_weight(op, w_up, scales_up, biases_up, N, K, group_size)) != QMM_OK) return st;
  if (M == 0 || N == 0) return QMM_OK;
  if (!x || !aligned16(x))
    return fail(QMM_ERR_INVALID_ARG, "%s: x must be a non-null 16-byte aligned pointer", op);
  if (!y_gate || !aligned16(y_gate) || !y_up || !aligned16(y_up))
    return fail(QMM_ERR_INVALID_ARG, "%s: y_gate and y_up must be non-null 16-byte aligned pointers", op);
  qmm::PackedWeight g{w_gate, scales_gate, biases_gate, N, K, group_size, bits};
  qmm::PackedWeight u{w_up, scales_up, biases_up, N, K, group_size, bits};
  return cuda_status(qmm::launch_gate_up(x, M, g, u, y_gate, y_up, y_dtype == QMM_BF16,
                                         reinterpret_cast<cudaStream_t>(stream)),
                     op);
}

qmm_status qmm_gemv_silu_gate(const uint16_t *gate, const uint16_t *up, int64_t M,
                              const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                              int64_t N, int64_t K, int group_size, int bits,
                              const uint16_t *resid, void *y, qmm_dtype y_dtype,
                              qmm_stream_t stream) {
  const char *op = "qmm_gemv_silu_gate";
  qmm_status st;
  if ((st = check_fused(op, M, 8, w, scales, biases, N, K, group_size, bits, y_dtype)) != QMM_OK)
    return st;
  if (M == 0 || N == 0) return QMM_OK;
  if (!gate || !aligned16(gate) || !up || !aligned16(up))
    return fail(QMM_ERR_INVALID_ARG, "%s: gate and up must be non-null 16-byte aligned pointers", op);
  if (resid && !aligned16(resid))
    return fail(QMM_ERR_INVALID_ARG, "%s: resid must be 16-byte aligned", op);
  if (!y || !aligned16(y))
    return fail(QMM_ERR_INVALID_ARG, "%s: y must be a non-null 16-byte aligned pointer", op);
  qmm::PackedWeight pw{w, scales, biases, N, K, group_size, bits};
  return cuda_status(qmm::launch_silu_gate(gate, up, M, pw, resid, y, y_dtype == QMM_BF16,
                                           reinterpret_cast<cudaStream_t>(stream)),
                     op);
}

// For callers that cannot allocate device memory: the checks and kernels of
// qmm_quantized_matmul, with split-K partials in the library's static scratch.
qmm_status qmm_quantized_matmul_noalloc(const uint16_t *x, int64_t M, const uint32_t *w,
                                        const uint16_t *scales, const uint16_t *biases,
                                        int64_t N, int64_t K, int transpose, int group_size,
                                        int bits, void *y, qmm_dtype y_dtype,
                                        qmm_stream_t stream) {
  const char *op = "qmm_quantized_matmul_noalloc";
  bool work = false;
  const qmm_status st = check_matmul(op, x, QMM_BF16, M, w, scales, biases, QMM_BF16, N, K,
                                     transpose, group_size, bits, y, y_dtype, &work);
  if (st != QMM_OK || !work) return st;
  const int64_t rows = transpose ? N : K, cols = transpose ? K : N;
  // Set-up on the first call on this device: the scratch's device address.
  float *scratch = qmm::static_scratch();
  if (!scratch)
    return fail(QMM_ERR_CUDA, "%s: cannot look up the static scratch on the current device", op);
  qmm::PackedWeight pw{w, scales, biases, rows, cols, group_size, bits};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = y_dtype == QMM_BF16;
  if (M <= 16) return cuda_status(qmm::launch_gemv(x, M, pw, transpose != 0, y, bf16, s), op);
  size_t needed = 0;
  const cudaError_t e =
      qmm::launch_gemm_static_scratch(x, M, pw, transpose != 0, y, bf16, scratch, s, &needed);
  if (e == cudaErrorInvalidValue && needed > qmm::static_scratch_bytes())
    return fail(QMM_ERR_INVALID_ARG,
                "%s: M=%lld N=%lld K=%lld needs %zu bytes of split-K scratch, more than the "
                "%zu this entry point holds (qmm_quantized_matmul has no such limit)",
                op, (long long)M, (long long)N, (long long)K, needed, qmm::static_scratch_bytes());
  return cuda_status(e, op);
}

// ------------------------------------------------------------- dtypes ----

qmm_status qmm_promote_types(qmm_dtype a, qmm_dtype b, qmm_dtype *out) {
  if (!out) return fail(QMM_ERR_INVALID_ARG, "qmm_promote_types: null output pointer");
  if (!known_dtype(a) || !known_dtype(b))
    return fail(QMM_ERR_UNSUPPORTED, "qmm_promote_types: unknown dtype %d or %d",
                static_cast<int>(a), static_cast<int>(b));
  *out = promote(a, b);
  return QMM_OK;
}

qmm_status qmm_dequantize_typed(const uint32_t *w, const void *scales, const void *biases,
                                qmm_dtype sb_dtype, int64_t rows, int64_t cols, int group_size,
                                int bits, void *out, qmm_dtype out_dtype, qmm_stream_t stream) {
  return dequantize_impl("qmm_dequantize_typed", w, scales, biases, sb_dtype, rows, cols, false,
                         nullptr, 0, group_size, bits, out, out_dtype, stream);
}

qmm_status qmm_rows_typed(const uint32_t *w, const void *scales, const void *biases,
                          qmm_dtype sb_dtype, int64_t table_rows, int64_t cols,
                          const uint32_t *idx, int64_t n, int group_size, int bits, void *out,
                          qmm_dtype out_dtype, qmm_stream_t stream) {
  return dequantize_impl("qmm_rows_typed", w, scales, biases, sb_dtype, table_rows, cols, true, idx,
                         n, group_size, bits, out, out_dtype, stream);
}

qmm_status qmm_quantize_typed(const void *w, qmm_dtype w_dtype, int64_t rows, int64_t cols,
                              int group_size, int bits, uint32_t *packed, void *scales,
                              void *biases, qmm_stream_t stream) {
  return quantize_impl("qmm_quantize_typed", w, w_dtype, rows, cols, group_size, bits, packed,
                       scales, biases, stream);
}

qmm_status qmm_quantized_matmul_typed(const void *x, qmm_dtype x_dtype, int64_t M,
                                      const uint32_t *w, const void *scales, const void *biases,
                                      qmm_dtype sb_dtype, int64_t N, int64_t K, int transpose,
                                      int group_size, int bits, void *y, qmm_dtype y_dtype,
                                      qmm_stream_t stream) {
  return matmul_impl("qmm_quantized_matmul_typed", x, x_dtype, M, w, scales, biases, sb_dtype, N,
                     K, transpose, group_size, bits, y, y_dtype, stream);
}

qmm_status qmm_get_device_error(qmm_stream_t stream) {
  unsigned bits = 0;
  cudaError_t e = qmm::take_device_error(reinterpret_cast<cudaStream_t>(stream), &bits);
  if (e != cudaSuccess) return cuda_status(e, "qmm_get_device_error");
  if (bits & qmm::kErrTimeoutBit)
    return fail(QMM_ERR_TIMEOUT, "qmm_get_device_error: a bounded wait inside a kernel ran out");
  if (bits & qmm::kErrIndexBit)
    return fail(QMM_ERR_INDEX, "qmm_get_device_error: a qmm_rows index was outside its table");
  return QMM_OK;
}

}  // extern "C"
