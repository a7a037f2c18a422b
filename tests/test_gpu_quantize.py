"""GPU quantize against the oracle: packed words, scales and biases bit for
bit (integer and byte work), at every width and group size, on ragged shapes,
constant groups and a full-size weight."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import dev  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)


def run(w, rows, cols, gs, bits):
    packed = torch.empty((rows, cols * bits // 32), dtype=torch.int32, device="cuda")
    s = torch.empty((rows, cols // gs), dtype=torch.int16, device="cuda")
    b = torch.empty_like(s)
    qmm.qmm_quantize(dev(w), rows, cols, gs, bits, packed, s, b)
    torch.cuda.synchronize()
    return (packed.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
            b.cpu().numpy().view(np.uint16))


def check(w, rows, cols, gs, bits, what):
    got = run(w, rows, cols, gs, bits)
    want = oracle.quantize(w, rows, cols, gs, bits)
    for name, g, o in zip(("packed", "scales", "biases"), got, want):
        bad = g != o
        assert not bad.any(), "%s: %s differ at %d of %d places, first %s" % (
            what, name, bad.sum(), bad.size, tuple(np.argwhere(bad)[0]))


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("gs", (32, 64, 128))
def test_quantize_matches_oracle(bits, gs):
    rows, cols = 37, 384      # rows not a multiple of anything; 3 to 12 groups a row
    w = synth.x_bf16(80 + bits + gs, rows, cols)
    check(w, rows, cols, gs, bits, "bits=%d gs=%d" % (bits, gs))


@pytest.mark.parametrize("bits", (3, 4, 8))
def test_quantize_constant_and_mixed_groups(bits):
    rows, cols, gs = 4, 256, 64
    w = synth.x_bf16(90 + bits, rows, cols)
    w[1, :64] = w[1, 0]                  # a constant group: scale 0, codes 0
    w[2, 64:128] = 0                     # all zero
    w[3, :] = np.abs(w[3, :].view(np.int16)).astype(np.uint16)  # positive values only
    check(w, rows, cols, gs, bits, "constant/mixed bits=%d" % bits)


@pytest.mark.parametrize("bits", (2, 4, 8))
def test_quantize_signed_zero_minimum(bits):
    # Groups whose minimum is zero with both signs present: the minimum is
    # compared in the group's order, so the stored bias keeps the sign of the
    # first zero, and every code follows from it.  Row 0: -0 before +0; row 1:
    # +0 before -0; row 2: all zeros of mixed sign (a constant group).
    rows, cols, gs = 3, 128, 64
    w = synth.x_bf16(97 + bits, rows, cols) & np.uint16(0x7FFF)  # |x|: non-negative
    w[0, 3], w[0, 9] = 0x8000, 0x0000
    w[0, 64 + 1], w[0, 64 + 2] = 0x8000, 0x0000
    w[1, 5], w[1, 6] = 0x0000, 0x8000
    w[1, 64 + 0], w[1, 64 + 40] = 0x0000, 0x8000
    w[2, :] = np.where(np.arange(cols) % 3 == 0, 0x8000, 0x0000).astype(np.uint16)
    check(w, rows, cols, gs, bits, "signed zeros bits=%d" % bits)


def test_quantize_full_size_weight():
    rows, cols = 4096, 4096
    w = synth.x_bf16(95, rows, cols)
    check(w, rows, cols, 64, 4, "[4096, 4096] 4-bit")


def test_quantize_then_dequantize_round_trip():
    rows, cols, gs, bits = 64, 512, 32, 6
    w = synth.x_bf16(96, rows, cols)
    p, s, b = (t for t in run(w, rows, cols, gs, bits))
    out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    qmm.qmm_dequantize(dev(p), dev(s), dev(b), rows, cols, gs, bits, out, qmm.QMM_F32)
    torch.cuda.synchronize()
    back = out.cpu().numpy().astype(np.float64)
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    step = np.repeat((s.astype(np.uint32) << 16).view(np.float32).astype(np.float64), gs, axis=1)
    top = (1 << bits) - 1
    assert (np.abs(back - wf) <= 0.5 * step * (1 + 1e-3) + top * 2.0 ** -9 * step + 1e-6).all()


@pytest.mark.parametrize("bits", (2, 4, 8))
def test_quantize_exact_half_way_quotients(bits):
    """Groups built so that (w - bias) / scale is exactly n + 1/2 for many w:
    bias 0, maximum 2^bits - 1, so the scale is exactly 1, and the other values
    are half-integers (exact in bf16 below 128).  Ties go to the even code on
    both sides; the kernel must take its exact route for them."""
    rows, cols, gs = 3, 128, 64
    top = (1 << bits) - 1
    g = np.random.default_rng(97 + bits)
    halves = (g.integers(0, min(top, 127), size=(rows, cols)) + 0.5).astype(np.float32)
    halves[:, ::gs] = 0.0
    halves[:, 1::gs] = float(min(top, 127)) if bits < 8 else 127.0
    w = (halves.view(np.uint32) >> 16).astype(np.uint16)
    check(w, rows, cols, gs, bits, "half-way quotients bits=%d" % bits)
