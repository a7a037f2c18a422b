"""The bounded waits inside the kernels, made to run out on purpose.

Every wait of a kernel on its own barriers gives up after a number of polls
(qmm_set_wait_limit; seconds by default).  A wait that runs out records
QMM_ERR_TIMEOUT in the device error word, the kernel stops early, waits for
the copies it has in flight, frees its tensor memory and returns: nothing
faults or hangs, and the next call on the same stream is correct.  With the
limit at one poll, the tensor-core GEMM's consumer waits (for x tiles and for
dequantized weight stages that cannot be ready yet) run out at once.  (The
pages' own error model is a returned error: nuvec_core quantized.rs,
`check_params`; rlx-moshi src/mlx_dequant.rs, `dequantize_affine`.)"""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import assert_within_tolerance, dev, empty_out, host_f64, weight  # noqa: E402


def matmul(x, M, w, N, K, y_dtype):
    pw, ps, pb = weight(w)
    y = empty_out((M, N), y_dtype)
    qmm.qmm_quantized_matmul(dev(x), M, pw, ps, pb, N, K, 1, w.group_size, w.bits, y, y_dtype)
    return y


@pytest.mark.parametrize("M,N,K", [
    (256, 512, 4096),    # two 256-row tiles: no split
    (128, 1024, 4096),   # 4 tiles: split-K, partials added by a second kernel
])
def test_gemm_wait_runs_out_then_next_call_is_correct(M, N, K):
    w = synth.quant_weight(800 + M, N, K, 4, 64)
    x = synth.x_bf16(801 + M, M, K)
    qmm.qmm_get_device_error()  # read and clear what earlier calls left (an index test's bit)
    prev = qmm.qmm_set_wait_limit(1)
    try:
        y = matmul(x, M, w, N, K, qmm.QMM_F32)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_wait_limit(prev)
    assert qmm.qmm_get_device_error() == qmm.QMM_ERR_TIMEOUT
    if M == 128:
        # split-K: the finalize kernel saw the timeout and wrote NaN, not a
        # plausible sum of incomplete partials
        assert np.isnan(host_f64(y)).all()
    # The error word was read and cleared; the same call now runs to the end.
    y2 = matmul(x, M, w, N, K, qmm.QMM_BF16)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == qmm.QMM_OK
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, 64, 4)
    assert_within_tolerance(y2, ref, absy, "after the timeout")


def test_decode_wait_limit_then_next_call_is_correct():
    """The decode kernel with the one-poll limit: whether a chunk wait finds
    its copy still in flight depends on timing, so the status is OK or
    TIMEOUT; either way the kernel returns, and with the default limit back the
    next call is correct."""
    N, K = 4096, 4096
    w = synth.quant_weight(810, N, K, 4, 64)
    x = synth.x_bf16(811, 1, K)
    qmm.qmm_get_device_error()
    prev = qmm.qmm_set_wait_limit(1)
    try:
        for _ in range(8):
            matmul(x, 1, w, N, K, qmm.QMM_BF16)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_wait_limit(prev)
    assert qmm.qmm_get_device_error() in (qmm.QMM_OK, qmm.QMM_ERR_TIMEOUT)
    y = matmul(x, 1, w, N, K, qmm.QMM_BF16)
    torch.cuda.synchronize()
    assert qmm.qmm_get_device_error() == qmm.QMM_OK
    ref, absy = oracle.qmm(x, 1, w.packed, w.scales, w.biases, N, K, True, 64, 4)
    assert_within_tolerance(y, ref, absy, "decode after the one-poll limit")
