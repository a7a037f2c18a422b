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


def test_noalloc_rejects_partials_beyond_its_scratch():
    # M = 2048 over a [1024, 4096] weight: 32 tiles, K split 4 ways, 33.5 MB of
    # partials -- more than the 24 MiB the entry point holds.
    M, N, K = 2048, 1024, 4096
    w = synth.quant_weight(710, N, K, 4, 64)
    x = synth.x_bf16(711, M, K)
    pw, ps, pb = weight(w)
    y = empty_out((M, N), qmm.QMM_BF16)
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_quantized_matmul_noalloc(dev(x), M, pw, ps, pb, N, K, 1, 64, 4, y, qmm.QMM_BF16)
    assert e.value.status == qmm.QMM_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
