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
        _lib = lib
    return _lib


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
               out_dtype="f32", nthreads=None):
    """dequant(W) as float32 [rows, cols], or bf16 bits (uint16) if out_dtype='bf16'."""
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, np.uint16)
    biases, pb = _c(biases, np.uint16)
    bf16 = out_dtype == "bf16"
    out = np.empty((rows, cols), dtype=np.uint16 if bf16 else np.float32)
    _load().oracle_dequantize(pp, ps, pb, rows, cols, group_size, bits, int(bf16),
                              out.ctypes.data_as(ctypes.c_void_p),
                              nthreads or default_threads())
    return out


def rows(packed, scales, biases, table_rows, cols, idx, group_size, bits,
         out_dtype="bf16", nthreads=None):
    """(out [n, cols], number of out-of-table indices)."""
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, np.uint16)
    biases, pb = _c(biases, np.uint16)
    idx, pi = _c(idx, np.uint32)
    bf16 = out_dtype == "bf16"
    out = np.empty((idx.size, cols), dtype=np.uint16 if bf16 else np.float32)
    bad = _load().oracle_rows(pp, ps, pb, table_rows, cols, pi, idx.size, group_size,
                              bits, int(bf16), out.ctypes.data_as(ctypes.c_void_p),
                              nthreads or default_threads())
    return out, int(bad)


def qmm(x, M, packed, scales, biases, N, K, transpose, group_size, bits, nthreads=None):
    """(y, absy): fp64 [M, N] each; absy = sum_k |x*w|, the tolerance scale."""
    x, px = _c(x, np.uint16)
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, np.uint16)
    biases, pb = _c(biases, np.uint16)
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    _load().oracle_qmm(px, M, pp, ps, pb, N, K, int(bool(transpose)), group_size, bits,
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


def quantize(w, rows, cols, group_size, bits, nthreads=None):
    """(packed, scales, biases) of bf16 w [rows, cols]; see oracle_quantize in
    qmm_oracle.c for the rule and its readings."""
    w, pw = _c(w, np.uint16)
    packed = np.empty((rows, cols * bits // 32), dtype=np.uint32)
    scales = np.empty((rows, cols // group_size), dtype=np.uint16)
    biases = np.empty((rows, cols // group_size), dtype=np.uint16)
    _load().oracle_quantize(pw, rows, cols, group_size, bits,
                            packed.ctypes.data_as(ctypes.c_void_p),
                            scales.ctypes.data_as(ctypes.c_void_p),
                            biases.ctypes.data_as(ctypes.c_void_p), nthreads or default_threads())
    return packed, scales, biases


def qmm_sampled(x, M, packed, scales, biases, N, K, transpose, group_size, bits,
                ms, ns, nthreads=None):
    """(y, absy) at the sampled positions (ms[i], ns[i])."""
    x, px = _c(x, np.uint16)
    packed, pp = _c(packed, np.uint32)
    scales, ps = _c(scales, np.uint16)
    biases, pb = _c(biases, np.uint16)
    ms, pm = _c(ms, np.int64)
    ns, pn = _c(ns, np.int64)
    y = np.empty(ms.size, dtype=np.float64)
    a = np.empty(ms.size, dtype=np.float64)
    _load().oracle_qmm_sampled(px, M, pp, ps, pb, N, K, int(bool(transpose)), group_size,
                               bits, pm, pn, ms.size, y.ctypes.data_as(ctypes.c_void_p),
                               a.ctypes.data_as(ctypes.c_void_p),
                               nthreads or default_threads())
    return y, a
