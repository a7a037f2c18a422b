"""qmm_quantized_matmul_noalloc, the entry point for callers that cannot
allocate device memory while they run (their own allocator owns the device,
or they record work where no allocation call may appear): called through the
C ABI, its results must match qmm_quantized_matmul's within the matmul
tolerance, 8e-3 * sum_k |x w| + 1e-6, on two calls in a row -- the second
finds the shared scratch holding the first call's partials.  This file is
collected last on purpose."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import TOL_ABS, TOL_REL, dev, empty_out, host_f64, weight  # noqa: E402


def both(x, M, w, N, K, transpose, y_dtype):
    pw, ps, pb = weight(w)
    dx = dev(x)
    y_ref = empty_out((M, N), y_dtype)
    qmm.qmm_quantized_matmul(dx, M, pw, ps, pb, N, K, transpose, w.group_size, w.bits, y_ref, y_dtype)
    outs = []
    for _ in range(2):
        y = empty_out((M, N), y_dtype)
        qmm.qmm_quantized_matmul_noalloc(dx, M, pw, ps, pb, N, K, transpose, w.group_size, w.bits,
                                         y, y_dtype)
        torch.cuda.synchronize()
        outs.append(host_f64(y))
    return host_f64(y_ref), outs


def absy_sampled(x, M, w, N, K, transpose, ms, ns):
    _, absy = oracle.qmm_sampled(x, M, w.packed, w.scales, w.biases, N, K, transpose,
                                 w.group_size, w.bits, ms, ns)
    return absy


@pytest.mark.parametrize("M,N,K,bits,transpose", [
    (128, 4096, 4096, 4, 1),   # split-K: 16 tiles, K split 9 ways, 18.9 MB of partials
    (64, 1024, 2048, 8, 1),    # split-K over 4 tiles
    (40, 512, 1024, 3, 0),     # split-K with W stored [K, N]
    (2048, 14336, 4096, 4, 1), # enough tiles: no split, no scratch
    (1, 4096, 4096, 4, 1),     # decode kernel
])
def test_noalloc_matches_quantized_matmul_twice(M, N, K, bits, transpose):
    rows, cols = (N, K) if transpose else (K, N)
    w = synth.quant_weight(700 + M + bits, rows, cols, bits, 64)
    x = synth.x_bf16(701 + M, M, K)
    ref, outs = both(x, M, w, N, K, transpose, qmm.QMM_BF16)
    g = np.random.default_rng(M + N)
    ms = np.concatenate([g.integers(0, M, 4000), np.full(N, M - 1)]).astype(np.int64)
    ns = np.concatenate([g.integers(0, N, 4000), np.arange(N)]).astype(np.int64)
    bound = TOL_REL * absy_sampled(x, M, w, N, K, transpose, ms, ns) + TOL_ABS
    for call, y in enumerate(outs):
        err = np.abs(y[ms, ns] - ref[ms, ns])
        assert (err <= bound).all(), "call %d: %d of %d sampled outputs differ beyond tolerance" % (
            call + 1, (err > bound).sum(), err.size)


@pytest.mark.parametrize("M,N,K", [
    (2048, 1024, 4096),  # 32 tiles: the usual 4-way split needs 33.5 MB; 3 ways fit 24 MiB
    (2048, 2048, 4096),  # 64 tiles: even a 2-way split needs 33.5 MB; runs unsplit
])
def test_noalloc_splits_fewer_ways_when_its_scratch_is_short(M, N, K):
    """Partials that would not fit the fixed array: K is split fewer ways (or
    not at all) instead of the call failing; results stay within tolerance
    of qmm_quantized_matmul's on two calls in a row."""
    w = synth.quant_weight(710 + N // 1024, N, K, 4, 64)
    x = synth.x_bf16(711, M, K)
    ref, outs = both(x, M, w, N, K, 1, qmm.QMM_BF16)
    g = np.random.default_rng(M + N + 1)
    ms = np.concatenate([g.integers(0, M, 4000), np.full(N, M - 1)]).astype(np.int64)
    ns = np.concatenate([g.integers(0, N, 4000), np.arange(N)]).astype(np.int64)
    bound = TOL_REL * absy_sampled(x, M, w, N, K, 1, ms, ns) + TOL_ABS
    for call, y in enumerate(outs):
        err = np.abs(y[ms, ns] - ref[ms, ns])
        assert (err <= bound).all(), "call %d: %d of %d sampled outputs differ beyond tolerance" % (
            call + 1, (err > bound).sum(), err.size)


def _cudart():
    """The CUDA runtime library, for reading the device's default memory
    pool (where stream-ordered allocations come from), or None."""
    import ctypes
    import glob
    import os
    names = []
    for d in [os.path.join(os.path.dirname(torch.__file__), "lib"), "/usr/local/cuda/lib64",
              "/usr/local/cuda/targets/sbsa-linux/lib", "/usr/local/cuda/targets/x86_64-linux/lib"]:
        names += sorted(glob.glob(os.path.join(d, "libcudart.so*")))
    names += ["libcudart.so.13", "libcudart.so"]
    for n in names:
        try:
            return ctypes.CDLL(n)
        except OSError:
            continue
    return None


def test_noalloc_takes_no_memory_from_the_pool():
    """The no-allocation entry point draws nothing from the device's default
    memory pool, where qmm_quantized_matmul takes its split-K workspace: the
    pool's used-memory high-water mark, reset before the call, stays at zero
    for the no-allocation call and rises for the allocating one (the check's
    positive control)."""
    import ctypes
    rt = _cudart()
    if rt is None:
        pytest.skip("no CUDA runtime library to read the memory pool with")
    kUsedMemHigh = 8  # cudaMemPoolAttrUsedMemHigh
    dev_id = ctypes.c_int(0)
    assert rt.cudaGetDevice(ctypes.byref(dev_id)) == 0
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), dev_id) == 0

    def high():
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, kUsedMemHigh, ctypes.byref(v)) == 0
        return v.value

    def reset():
        z = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, kUsedMemHigh, ctypes.byref(z)) == 0

    M, N, K = 128, 4096, 4096   # split-K: 18.9 MB of partials
    w = synth.quant_weight(720, N, K, 4, 64)
    pw, ps, pb = weight(w)
    dx = dev(synth.x_bf16(721, M, K))
    y = empty_out((M, N), qmm.QMM_BF16)
    torch.cuda.synchronize()
    reset()
    for _ in range(2):
        qmm.qmm_quantized_matmul_noalloc(dx, M, pw, ps, pb, N, K, 1, 64, 4, y, qmm.QMM_BF16)
    torch.cuda.synchronize()
    assert high() == 0
    qmm.qmm_quantized_matmul(dx, M, pw, ps, pb, N, K, 1, 64, 4, y, qmm.QMM_BF16)
    torch.cuda.synchronize()
    assert high() > 0
