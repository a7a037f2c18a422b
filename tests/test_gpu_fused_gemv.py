"""GPU parity of the fused decode GEMVs against the oracle: gate_up against two
oracle matmuls (8e-3 * sum_k |x w| + 1e-6), silu_gate against the oracle's
fp64 silu(gate) * up product (8e-3 * (sum_k |x w| + |resid|) + 1e-6)."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import assert_within_tolerance, dev, empty_out, weight  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M", (1, 5, 9, 16))
def test_gate_up(bits, M):
    N, K, gs = 200, 1024, 64   # ragged last 16-row tile
    wg = synth.quant_weight(40 + bits, N, K, bits, gs)
    wu = synth.quant_weight(41 + bits, N, K, bits, gs)
    x = synth.x_bf16(42 + M, M, K)
    yg, yu = empty_out((M, N), qmm.QMM_BF16), empty_out((M, N), qmm.QMM_BF16)
    qmm.qmm_gemv_gate_up(dev(x), M, *weight(wg), *weight(wu), N, K, gs, bits, yg, yu, qmm.QMM_BF16)
    torch.cuda.synchronize()
    for y, w, what in ((yg, wg, "gate"), (yu, wu, "up")):
        ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, gs, bits)
        assert_within_tolerance(y, ref, absy, "gate_up %s bits=%d M=%d" % (what, bits, M))


@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("M", (1, 8))
def test_gate_up_many_row_tiles(bits, M):
    # 2 x 157 row tiles, more than two 16-warp blocks an SM: the 8-warp form
    # below 6 bits.
    N, K, gs = 2500, 1024, 64
    wg = synth.quant_weight(70 + bits, N, K, bits, gs)
    wu = synth.quant_weight(71 + bits, N, K, bits, gs)
    x = synth.x_bf16(72 + M, M, K)
    yg, yu = empty_out((M, N), qmm.QMM_BF16), empty_out((M, N), qmm.QMM_BF16)
    qmm.qmm_gemv_gate_up(dev(x), M, *weight(wg), *weight(wu), N, K, gs, bits, yg, yu, qmm.QMM_BF16)
    for y, w in ((yg, wg), (yu, wu)):
        ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, gs, bits)
        assert_within_tolerance(y, ref, absy, "gate_up many tiles b%d M%d" % (bits, M))


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M", (1, 3, 8))
@pytest.mark.parametrize("with_resid", (False, True))
def test_silu_gate(bits, M, with_resid):
    N, K, gs = 200, 1024, 32
    w = synth.quant_weight(50 + bits, N, K, bits, gs)
    gate = synth.x_bf16(51 + M, M, K)
    up = synth.x_bf16(52 + M, M, K)
    resid = synth.x_bf16(53 + M, M, N) if with_resid else None
    y = empty_out((M, N), qmm.QMM_F32)
    qmm.qmm_gemv_silu_gate(dev(gate), dev(up), M, *weight(w), N, K, gs, bits,
                           None if resid is None else dev(resid), y, qmm.QMM_F32)
    torch.cuda.synchronize()
    ref, scale = oracle.silu_gate_qmm(gate, up, M, w.packed, w.scales, w.biases, N, K, gs, bits,
                                      resid)
    assert_within_tolerance(y, ref, scale, "silu_gate bits=%d M=%d resid=%s" % (bits, M, with_resid))


def test_silu_gate_full_size_down_projection():
    # The down projection of an 8B-class block: W [4096, 14336], 4-bit g64, bf16 out.
    N, K = 4096, 14336
    w = synth.quant_weight(60, N, K, 4, 64)
    gate, up, resid = synth.x_bf16(61, 1, K), synth.x_bf16(62, 1, K), synth.x_bf16(63, 1, N)
    y = empty_out((1, N), qmm.QMM_BF16)
    qmm.qmm_gemv_silu_gate(dev(gate), dev(up), 1, *weight(w), N, K, 64, 4, dev(resid), y,
                           qmm.QMM_BF16)
    torch.cuda.synchronize()
    ref, scale = oracle.silu_gate_qmm(gate, up, 1, w.packed, w.scales, w.biases, N, K, 64, 4, resid)
    assert_within_tolerance(y, ref, scale, "silu_gate down projection")


def test_fused_reject_what_they_do_not_cover():
    w = synth.quant_weight(70, 64, 320, 4, 64)          # K = 320: not a multiple of 128
    x = dev(synth.x_bf16(71, 1, 320))
    y = empty_out((1, 64), qmm.QMM_BF16)
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_gemv_silu_gate(x, x, 1, *weight(w), 64, 320, 64, 4, None, y, qmm.QMM_BF16)
    assert e.value.status == qmm.QMM_ERR_INVALID_ARG
    w2 = synth.quant_weight(72, 64, 256, 4, 64)
    x2 = dev(synth.x_bf16(73, 9, 256))
    y2 = empty_out((9, 64), qmm.QMM_BF16)
    with pytest.raises(qmm.QmmError) as e:            # silu_gate takes M <= 8
        qmm.qmm_gemv_silu_gate(x2, x2, 9, *weight(w2), 64, 256, 64, 4, None, y2, qmm.QMM_BF16)
    assert e.value.status == qmm.QMM_ERR_INVALID_ARG
