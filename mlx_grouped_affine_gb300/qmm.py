"""Thin Python binding of the C ABI in include/qmm.h (argument marshalling only).

Every function here has the name of the C entry point it calls and passes the
device pointers of torch tensors straight through; all computation happens in
the CUDA kernels of libqmm.so.  There is no fallback: if the library cannot be
built or loaded, or a call returns an error status, a QmmError is raised.
"""
import ctypes

from . import build as _build

QMM_OK, QMM_ERR_INVALID_ARG, QMM_ERR_UNSUPPORTED, QMM_ERR_CUDA, QMM_ERR_INDEX, QMM_ERR_TIMEOUT = range(6)
QMM_F32, QMM_BF16, QMM_F16 = 0, 1, 2
STATUS_NAMES = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED",
                3: "QMM_ERR_CUDA", 4: "QMM_ERR_INDEX", 5: "QMM_ERR_TIMEOUT"}
QMM_LAUNCH_PDL = 1
EXPORTS = ("qmm_quantize", "qmm_dequantize", "qmm_quantized_matmul", "qmm_quantized_matmul_noalloc",
           "qmm_gather_qmm", "qmm_gemv_gate_up", "qmm_gemv_silu_gate", "qmm_rows",
           "qmm_last_error", "qmm_get_device_error", "qmm_set_launch_flags", "qmm_set_wait_limit",
           "qmm_promote_types", "qmm_dequantize_typed", "qmm_rows_typed", "qmm_quantize_typed",
           "qmm_quantized_matmul_typed")

_lib = None


class QmmError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


def lib():
    """The loaded libqmm.so (built first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.qmm_dequantize.argtypes = [P, P, P, I64, I64, I, I, P, I, P]
        L.qmm_quantize.argtypes = [P, I64, I64, I, I, P, P, P, P]
        L.qmm_quantized_matmul.argtypes = [P, I64, P, P, P, I64, I64, I, I, I, P, I, P]
        L.qmm_quantized_matmul_noalloc.argtypes = [P, I64, P, P, P, I64, I64, I, I, I, P, I, P]
        L.qmm_gather_qmm.argtypes = [P, I64, I64, P, P, P, I64, I64, I64, P, P, I64, I, I, I, I, P, I, P]
        L.qmm_gemv_gate_up.argtypes = [P, I64, P, P, P, P, P, P, I64, I64, I, I, P, P, I, P]
        L.qmm_gemv_silu_gate.argtypes = [P, P, I64, P, P, P, I64, I64, I, I, P, P, I, P]
        L.qmm_rows.argtypes = [P, P, P, I64, I64, P, I64, I, I, P, I, P]
        L.qmm_get_device_error.argtypes = [P]
        L.qmm_promote_types.argtypes = [I, I, ctypes.POINTER(I)]
        L.qmm_dequantize_typed.argtypes = [P, P, P, I, I64, I64, I, I, P, I, P]
        L.qmm_rows_typed.argtypes = [P, P, P, I, I64, I64, P, I64, I, I, P, I, P]
        L.qmm_quantize_typed.argtypes = [P, I, I64, I64, I, I, P, P, P, P]
        L.qmm_quantized_matmul_typed.argtypes = [P, I, I64, P, P, P, I, I64, I64, I, I, I, P, I, P]
        for f in ("qmm_quantize", "qmm_dequantize", "qmm_quantized_matmul", "qmm_quantized_matmul_noalloc",
                  "qmm_gather_qmm", "qmm_gemv_gate_up", "qmm_gemv_silu_gate", "qmm_rows",
                  "qmm_get_device_error", "qmm_promote_types", "qmm_dequantize_typed",
                  "qmm_rows_typed", "qmm_quantize_typed", "qmm_quantized_matmul_typed"):
            getattr(L, f).restype = I
        L.qmm_set_launch_flags.argtypes = [ctypes.c_uint]
        L.qmm_set_launch_flags.restype = ctypes.c_uint
        L.qmm_set_wait_limit.argtypes = [ctypes.c_uint32]
        L.qmm_set_wait_limit.restype = ctypes.c_uint32
        L.qmm_last_error.argtypes = []
        L.qmm_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(t):
    """Device address of a tensor (or an int address, or None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status):
    if status != QMM_OK:
        raise QmmError(status, qmm_last_error())


def qmm_last_error():
    return lib().qmm_last_error().decode()


def qmm_quantize(w, rows, cols, group_size, bits, packed, scales, biases, stream=None):
    _check(lib().qmm_quantize(_ptr(w), rows, cols, group_size, bits, _ptr(packed), _ptr(scales),
                              _ptr(biases), _stream(stream)))


def qmm_dequantize(w, scales, biases, rows, cols, group_size, bits, out, out_dtype,
                   stream=None):
    _check(lib().qmm_dequantize(_ptr(w), _ptr(scales), _ptr(biases), rows, cols, group_size,
                                bits, _ptr(out), out_dtype, _stream(stream)))


def qmm_quantized_matmul(x, M, w, scales, biases, N, K, transpose, group_size, bits, y,
                         y_dtype, stream=None):
    _check(lib().qmm_quantized_matmul(_ptr(x), M, _ptr(w), _ptr(scales), _ptr(biases), N, K,
                                      int(transpose), group_size, bits, _ptr(y), y_dtype,
                                      _stream(stream)))


def qmm_quantized_matmul_noalloc(x, M, w, scales, biases, N, K, transpose, group_size, bits, y,
                                 y_dtype, stream=None):
    """qmm_quantized_matmul for callers that cannot allocate device memory:
    split-K partials go to the library's fixed 24 MiB scratch (see qmm.h)."""
    _check(lib().qmm_quantized_matmul_noalloc(_ptr(x), M, _ptr(w), _ptr(scales), _ptr(biases), N,
                                              K, int(transpose), group_size, bits, _ptr(y),
                                              y_dtype, _stream(stream)))


def qmm_gather_qmm(x, x_batches, M, w, scales, biases, w_batches, N, K, lhs_indices, rhs_indices,
                   batches, transpose, group_size, bits, sorted_indices, y, y_dtype, stream=None):
    _check(lib().qmm_gather_qmm(_ptr(x), x_batches, M, _ptr(w), _ptr(scales), _ptr(biases),
                                w_batches, N, K, _ptr(lhs_indices), _ptr(rhs_indices), batches,
                                int(transpose), group_size, bits, int(sorted_indices), _ptr(y),
                                y_dtype, _stream(stream)))


def qmm_gemv_gate_up(x, M, w_gate, scales_gate, biases_gate, w_up, scales_up, biases_up, N, K,
                     group_size, bits, y_gate, y_up, y_dtype, stream=None):
    _check(lib().qmm_gemv_gate_up(_ptr(x), M, _ptr(w_gate), _ptr(scales_gate), _ptr(biases_gate),
                                  _ptr(w_up), _ptr(scales_up), _ptr(biases_up), N, K, group_size,
                                  bits, _ptr(y_gate), _ptr(y_up), y_dtype, _stream(stream)))


def qmm_gemv_silu_gate(gate, up, M, w, scales, biases, N, K, group_size, bits, resid, y, y_dtype,
                       stream=None):
    _check(lib().qmm_gemv_silu_gate(_ptr(gate), _ptr(up), M, _ptr(w), _ptr(scales), _ptr(biases),
                                    N, K, group_size, bits, _ptr(resid), _ptr(y), y_dtype,
                                    _stream(stream)))


def qmm_rows(w, scales, biases, table_rows, cols, idx, n, group_size, bits, out, out_dtype,
             stream=None):
    _check(lib().qmm_rows(_ptr(w), _ptr(scales), _ptr(biases), table_rows, cols, _ptr(idx), n,
                          group_size, bits, _ptr(out), out_dtype, _stream(stream)))


def qmm_get_device_error(stream=None):
    """The status qmm_get_device_error returns (does not raise)."""
    return lib().qmm_get_device_error(_stream(stream))


def qmm_set_launch_flags(flags):
    """Set this host thread's launch flags (QMM_LAUNCH_PDL); returns the previous ones."""
    return int(lib().qmm_set_launch_flags(flags))


def qmm_set_wait_limit(polls):
    """Polls a bounded wait in this host thread's kernels makes before it
    gives up (0: the default); returns the previous limit."""
    return int(lib().qmm_set_wait_limit(polls))


def qmm_promote_types(a, b):
    """The dtype that a and b promote to (host-only: no GPU needed)."""
    out = ctypes.c_int(-1)
    _check(lib().qmm_promote_types(a, b, ctypes.byref(out)))
    return out.value


def qmm_dequantize_typed(w, scales, biases, sb_dtype, rows, cols, group_size, bits, out,
                         out_dtype, stream=None):
    """qmm_dequantize with scales and biases of sb_dtype (QMM_BF16, QMM_F16 or
    QMM_F32); out_dtype is QMM_F32 or sb_dtype."""
    _check(lib().qmm_dequantize_typed(_ptr(w), _ptr(scales), _ptr(biases), sb_dtype, rows, cols,
                                      group_size, bits, _ptr(out), out_dtype, _stream(stream)))


def qmm_rows_typed(w, scales, biases, sb_dtype, table_rows, cols, idx, n, group_size, bits, out,
                   out_dtype, stream=None):
    """qmm_rows with scales and biases of sb_dtype; out_dtype QMM_F32 or sb_dtype."""
    _check(lib().qmm_rows_typed(_ptr(w), _ptr(scales), _ptr(biases), sb_dtype, table_rows, cols,
                                _ptr(idx), n, group_size, bits, _ptr(out), out_dtype,
                                _stream(stream)))


def qmm_quantize_typed(w, w_dtype, rows, cols, group_size, bits, packed, scales, biases,
                       stream=None):
    """qmm_quantize of a weight of w_dtype; scales and biases are written in w_dtype."""
    _check(lib().qmm_quantize_typed(_ptr(w), w_dtype, rows, cols, group_size, bits, _ptr(packed),
                                    _ptr(scales), _ptr(biases), _stream(stream)))


def qmm_quantized_matmul_typed(x, x_dtype, M, w, scales, biases, sb_dtype, N, K, transpose,
                               group_size, bits, y, y_dtype, stream=None):
    """qmm_quantized_matmul computed in qmm_promote_types(x_dtype, sb_dtype):
    bf16 and fp16 on the tensor cores, fp32 on the CUDA cores; y_dtype is
    QMM_F32 or that type."""
    _check(lib().qmm_quantized_matmul_typed(_ptr(x), x_dtype, M, _ptr(w), _ptr(scales),
                                            _ptr(biases), sb_dtype, N, K, int(transpose),
                                            group_size, bits, _ptr(y), y_dtype, _stream(stream)))
