"""Plain CPU oracle for MLX grouped affine quantization (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it, and the two share no code: the oracle is
the C file ``qmm_oracle.c`` next to this module, compiled with gcc and loaded
through ctypes.  The arithmetic it follows is described, with the passages of
the pages it restates, at the top of that file.

All arrays are numpy arrays on the host:
  packed  uint32 [rows, cols*bits/32]   scales/biases uint16 (bf16 bits) [rows, cols/G]
  x       uint16 (bf16 bits) [M, K]     idx uint32 [n]
The typed variants take a dtype name per buffer: "bf16" and "f16" buffers
hold 16-bit patterns (uint16), "f32" buffers float32 values.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile the oracle with gcc (plain C99, no fast-math, no contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=gnu99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_code.argtypes = [P, I64, I]
        lib.oracle_code.restype = ctypes.c_uint32
        lib.oracle_unpack.argtypes = [P, I64, I64, I, P]
        lib.oracle_pack.argtypes = [P, I64, I64, I, P]
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_dequantize.argtypes = [P, P, P, I64, I64, I, I, I, P, I]
        lib.oracle_rows.argtypes = [P, P, P, I64, I64, P, I64, I, I, I, P, I]
        lib.oracle_rows.restype = I64
        lib.oracle_qmm.argtypes = [P, I64, P, P, P, I64, I64, I, I, I, P, P, I]
        lib.oracle_qmm_sampled.argtypes = [P, I64, P, P, P, I64, I64, I, I, I,
                                           P, P, I64, P, P, I]
        lib.oracle_quantize.argtypes = [P, I64, I64, I, I, P, P, P, I]
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_dequantize_typed.argtypes = [P, P, P, I, I64, I64, I, I, I, P, I]
        lib.oracle_rows_typed.argtypes = [P, P, P, I, I64, I64, P, I64, I, I, I, P, I]
        lib.oracle_rows_typed.restype = I64
        lib.oracle_qmm_typed.argtypes = [P, I, I64, P, P, P, I, I64, I64, I, I, I, P, P, I]
        lib.oracle_qmm_sampled_typed.argtypes = [P, I, I64, P, P, P, I, I64, I64, I, I, I,
                                                 P, P, I64, P, P, I]
        lib.oracle_quantize_typed.argtypes = [P, I, I64, I64, I, I, P, P, P, I]
        _lib = lib
    return _lib


# The oracle's own numbering of element types (qmm_oracle.c, ORACLE_*).
_TYPE = {"f32": 0, "bf16": 1, "f16": 2}
# numpy storage of each type: 16-bit types as their bit patterns.
_STORE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}

# (exponent bits, fraction bits) of each floating-point format.
_FORMAT = {"bf16": (8, 7), "f16": (5, 10), "f32": (8, 23)}


def promote_types(a, b):
    """The type x, scales and biases are promoted to (nuvec_core quantized.rs,
    `quantized_matmul`: promote_types over the three, floating point only):
    the narrowest of bf16, f16 and f32 whose exponent and fraction fields are
    both at least as wide as each operand's, so that it holds every value of
    both exactly.  bf16 with f16 has no 16-bit answer: f32."""
    ea, fa = _FORMAT[a]
    eb, fb = _FORMAT[b]
    fits = [t for t, (e, f) in _FORMAT.items() if e >= max(ea, eb) and f >= max(fa, fb)]
    return min(fits, key=lambda t: sum(_FORMAT[t]))


def default_threads():
    return os.cpu_count() or 1


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def code(row_words, j, bits):
    w, p = _c(row_words, np.uint32)
    return int(_load().oracle_code(p, j, bits))


def unpack(packed, cols, bits):
    """codes uint8 [rows, cols] from packed uint32 [rows, cols*bits/32]."""
    packed, p = _c(packed, np.uint32)
    rows = packed.shape[0] if packed.ndim == 2 else 1
    out = np.empty((rows, cols), dtype=np.uint8)
    _load().oracle_unpack(p, rows, cols, bits, out.ctypes.data_as(ctypes.c_void_p))
    return out


def pack(codes, bits):
    """packed uint32 [rows, cols*bits/32] from codes [rows, cols]."""
    codes, p = _c(np.atleast_2d(codes), np.uint8)
    rows, cols = codes.shape
    out = np.empty((rows, cols * bits // 32), dtype=np.uint32)
    _load().oracle_pack(p, rows, cols, bits, out.ctypes.data_as(ctypes.c_void_p))
    return out


def f16_to_f64(h):
    return float(_load().oracle_f16_to_f64(int(h)))


def f32_to_f16(f):
    return int(_load().oracle_f32_to_f16(float(f)))


def bf16_to_f32(h):
    return float(_load().oracle_bf16_to_f32(int(h)))


def f32_to_bf16(f):
    return int(_load().oracle_f32_to_bf16(float(f)))


def f32_to_bf16_array(a):
    lib = _load()
    flat = np.asarray(a, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(a))


def dequantize(packed, scales, biases, rows, cols, group_size, bits,
               out_dtype="f32", nthreads=None, sb_dtype="bf16"):
    """dequant(W) [rows, cols] in out_dtype: float32 values for "f32", 16-bit
    patterns (uint16) for "bf16" and "f16"; scales and biases of sb_dtype."""
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, _STORE[sb_dtype])
    biases, pb = _c(biases, _STORE[sb_dtype])
    out = np.empty((rows, cols), dtype=_STORE[out_dtype])
    _load().oracle_dequantize_typed(pp, ps, pb, _TYPE[sb_dtype], rows, cols, group_size, bits,
                                    _TYPE[out_dtype], out.ctypes.data_as(ctypes.c_void_p),
                                    nthreads or default_threads())
    return out


def rows(packed, scales, biases, table_rows, cols, idx, group_size, bits,
         out_dtype="bf16", nthreads=None, sb_dtype="bf16"):
    """(out [n, cols], number of out-of-table indices)."""
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, _STORE[sb_dtype])
    biases, pb = _c(biases, _STORE[sb_dtype])
    idx, pi = _c(idx, np.uint32)
    out = np.empty((idx.size, cols), dtype=_STORE[out_dtype])
    bad = _load().oracle_rows_typed(pp, ps, pb, _TYPE[sb_dtype], table_rows, cols, pi,
                                    idx.size, group_size, bits, _TYPE[out_dtype],
                                    out.ctypes.data_as(ctypes.c_void_p),
                                    nthreads or default_threads())
    return out, int(bad)


def qmm(x, M, packed, scales, biases, N, K, transpose, group_size, bits, nthreads=None,
        x_dtype="bf16", sb_dtype="bf16"):
    """(y, absy): fp64 [M, N] each; absy = sum_k |x*w|, the tolerance scale."""
    x, px = _c(x, _STORE[x_dtype])
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, _STORE[sb_dtype])
    biases, pb = _c(biases, _STORE[sb_dtype])
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    _load().oracle_qmm_typed(px, _TYPE[x_dtype], M, pp, ps, pb, _TYPE[sb_dtype], N, K,
                             int(bool(transpose)), group_size, bits,
                             y.ctypes.data_as(ctypes.c_void_p), a.ctypes.data_as(ctypes.c_void_p),
                             nthreads or default_threads())
    return y, a


def gather_qmm(x, x_batches, M, packed, scales, biases, w_batches, N, K, lhs, rhs, transpose,
               group_size, bits, nthreads=None):
    """(y, absy): fp64 [B, M, N] each.  Output batch i is x[lhs[i]] times
    dequant(w[rhs[i]]) transposed (or not), each batch an ordinary
    quantized_matmul (nuvec_core quantized.rs, `gather_qmm` doc: the indices
    address the flattened batch dimensions of x [..., M, K] and of w, scales,
    biases; either index array defaults to every batch of its operand in
    order).  lhs, rhs: uint32 [B] (already broadcast) or None.  An index past
    its operand gives a batch of zeros (the pages are silent; as rows)."""
    rows, cols = (N, K) if transpose else (K, N)
    xs = np.asarray(x).reshape(x_batches, M, K)
    pk = np.asarray(packed).reshape(w_batches, rows, -1)
    sc = np.asarray(scales).reshape(w_batches, rows, -1)
    bi = np.asarray(biases).reshape(w_batches, rows, -1)
    B = len(lhs) if lhs is not None else len(rhs) if rhs is not None else x_batches
    y = np.zeros((B, M, N), dtype=np.float64)
    a = np.zeros((B, M, N), dtype=np.float64)
    for i in range(B):
        xi = int(lhs[i]) if lhs is not None else i
        wi = int(rhs[i]) if rhs is not None else i
        if xi >= x_batches or wi >= w_batches:
            continue
        y[i], a[i] = qmm(xs[xi], M, pk[wi], sc[wi], bi[wi], N, K, transpose, group_size, bits,
                         nthreads)
    return y, a


def silu_gate_qmm(gate, up, M, packed, scales, biases, N, K, group_size, bits, resid=None):
    """(y, scale): fp64 [M, N] each.  y = dequant(W) (silu(gate) * up), plus
    resid when given (spark_runtime weights/mlx_int8.rs, `gemv_silu_gate` and
    `gemv_silu_gate_resid` docs: y[n] = x_resid[n] + sum_k W[n, k] *
    (silu(gate[k]) * up[k])), for each of the M rows; silu(g) = g / (1 + e^-g).
    Everything in fp64 from the bf16 inputs (W transposed: [N, K]).  scale =
    sum_k |x w| + |resid|, the tolerance scale."""
    g = _bf16_f64(gate).reshape(M, K)
    u = _bf16_f64(up).reshape(M, K)
    with np.errstate(over="ignore"):
        x = g / (1.0 + np.exp(-g)) * u
    codes = unpack(packed, K, bits).astype(np.float64)
    rep = np.repeat(np.arange(K // group_size), group_size)
    w = _bf16_f64(scales)[:, rep] * codes + _bf16_f64(biases)[:, rep]
    y = x @ w.T
    a = np.abs(x) @ np.abs(w).T
    if resid is not None:
        r = _bf16_f64(resid).reshape(M, N)
        y = y + r
        a = a + np.abs(r)
    return y, a


def _bf16_f64(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def quantize(w, rows, cols, group_size, bits, nthreads=None, w_dtype="bf16"):
    """(packed, scales, biases) of w [rows, cols] of w_dtype, the scales and
    biases in w_dtype; see oracle_quantize_typed in qmm_oracle.c for the rule
    and its readings."""
    w, pw = _c(w, _STORE[w_dtype])
    packed = np.empty((rows, cols * bits // 32), dtype=np.uint32)
    scales = np.empty((rows, cols // group_size), dtype=_STORE[w_dtype])
    biases = np.empty((rows, cols // group_size), dtype=_STORE[w_dtype])
    _load().oracle_quantize_typed(pw, _TYPE[w_dtype], rows, cols, group_size, bits,
                                  packed.ctypes.data_as(ctypes.c_void_p),
                                  scales.ctypes.data_as(ctypes.c_void_p),
                                  biases.ctypes.data_as(ctypes.c_void_p),
                                  nthreads or default_threads())
    return packed, scales, biases


def qmm_sampled(x, M, packed, scales, biases, N, K, transpose, group_size, bits,
                ms, ns, nthreads=None, x_dtype="bf16", sb_dtype="bf16"):
    """(y, absy) at the sampled positions (ms[i], ns[i])."""
    x, px = _c(x, _STORE[x_dtype])
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, _STORE[sb_dtype])
    biases, pb = _c(biases, _STORE[sb_dtype])
    ms, pm = _c(ms, np.int64)
    ns, pn = _c(ns, np.int64)
    y = np.empty(ms.size, dtype=np.float64)
    a = np.empty(ms.size, dtype=np.float64)
    _load().oracle_qmm_sampled_typed(px, _TYPE[x_dtype], M, pp, ps, pb, _TYPE[sb_dtype], N, K,
                                     int(bool(transpose)), group_size, bits, pm, pn, ms.size,
                                     y.ctypes.data_as(ctypes.c_void_p),
                                     a.ctypes.data_as(ctypes.c_void_p),
                                     nthreads or default_threads())
    return y, a
