"""The weights inside quantized_matmul, one element at a time.

With x rows that are one-hot (1.0 at column k_m, zero elsewhere) and fp32
output, every sum holds a single nonzero product, so y[m, n] is the matmul's
own dequantized weight w[n, k_m] with no accumulation error.  Each must be
the bf16 rounding of scale * code + bias: rounded once from the exact value,
or (the fp32 route) first to fp32 and then to bf16, as the standalone
dequantize does.  Scale laws cover both dequantization forms the kernels
choose between per chunk: normal scales below 2^-5, larger scales, a mix of
the two in one tile, and subnormal and zero scales."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import dev, empty_out, host_f64, weight  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)
ONE = 0x3F80  # bf16 1.0


def bf16_bits_of(f32):
    return (np.asarray(f32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_f64_to_bf16(v):
    """Round-to-nearest-even of float64 values to bf16 (8 significant bits);
    the values here are far from the bf16 subnormal and overflow ranges."""
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def with_scale_law(w, law, seed):
    """The weight w with its scales (and biases, by the same law as
    synth.quant_weight: -scale * 2^(bits-1) + N(0, 1e-3)) redrawn."""
    g = np.random.default_rng(seed)
    s = bf16_value(w.scales).astype(np.float32)
    if law == "large":
        s = g.uniform(0.05, 4.0, size=s.shape).astype(np.float32)
    elif law == "mixed":
        pick = g.random(size=s.shape) < 0.1
        s = np.where(pick, g.uniform(0.05, 4.0, size=s.shape), s).astype(np.float32)
    sb = bf16_bits_of(s)
    if law == "tiny":
        # subnormal bf16 scales (exponent field 0), some exactly zero
        sb = g.integers(1, 128, size=s.shape).astype(np.uint16)
        sb[g.random(size=s.shape) < 0.2] = 0
        s = bf16_value(sb).astype(np.float32)
    b = -s * np.float32(2 ** (w.bits - 1)) + g.normal(0.0, 1e-3, size=s.shape).astype(np.float32)
    return synth.QuantWeight(w.packed, sb, bf16_bits_of(b), w.rows, w.cols, w.bits, w.group_size)


def expected(w, transpose):
    """Stored-layout weights: exact-then-bf16 and the dequantize output."""
    codes = oracle.unpack(w.packed, w.cols, w.bits).astype(np.float64)
    rep = np.repeat(np.arange(w.cols // w.group_size), w.group_size)
    s = bf16_value(w.scales)[:, rep]
    b = bf16_value(w.biases)[:, rep]
    once = round_f64_to_bf16(s * codes + b)
    dq = bf16_value(oracle.dequantize(w.packed, w.scales, w.biases, w.rows, w.cols,
                                      w.group_size, w.bits, out_dtype="bf16"))
    return once, dq


@pytest.mark.parametrize("law", ("small", "large", "mixed", "tiny"))
@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M,transpose", ((1, True), (8, True), (16, True), (16, False), (40, True)))
def test_matmul_weights_are_rounded_dequantized_values(law, bits, M, transpose):
    # Stored [200, 1024] (a ragged 16-row tile) or, for W stored [K, N],
    # [1024, 256]; group 32.
    rows, cols, gs = (200, 1024, 32) if transpose else (1024, 256, 32)
    w = with_scale_law(synth.quant_weight(1000 + bits, rows, cols, bits, gs), law, 7 * bits + M)
    N, K = (rows, cols) if transpose else (cols, rows)
    ks = np.random.default_rng(M + bits).choice(K, size=M, replace=False)
    x = np.zeros((M, K), dtype=np.uint16)
    x[np.arange(M), ks] = ONE
    pw, ps, pb = weight(w)
    y = empty_out((M, N), qmm.QMM_F32)
    qmm.qmm_quantized_matmul(dev(x), M, pw, ps, pb, N, K, transpose, gs, bits, y, qmm.QMM_F32)
    torch.cuda.synchronize()
    got = host_f64(y)
    once, dq = expected(w, transpose)
    want_once = once[:, ks].T if transpose else once[ks, :]
    want_dq = dq[:, ks].T if transpose else dq[ks, :]
    ok = (got == want_once) | (got == want_dq)
    if not ok.all():
        m, n = np.argwhere(~ok)[0]
        raise AssertionError("%d of %d weights differ; first (m=%d, n=%d): got %r, rounded once %r, "
                             "dequantize %r" % ((~ok).sum(), ok.size, m, n, got[m, n],
                                                 want_once[m, n], want_dq[m, n]))
