"""GPU parity of qmm_quantized_matmul on the decode path (M <= 16) against the
fp64 oracle: every output within 8e-3 * sum_k |x w| + 1e-6."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import assert_within_tolerance, dev, empty_out, weight  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)


def run_qmm(x, M, w, N, K, transpose, y_dtype=qmm.QMM_BF16):
    pw, ps, pb = weight(w)
    dx = dev(x)
    y = empty_out((M, N), y_dtype)
    qmm.qmm_quantized_matmul(dx, M, pw, ps, pb, N, K, transpose, w.group_size, w.bits, y, y_dtype)
    torch.cuda.synchronize()
    return y


def check(x, M, w, N, K, transpose, y_dtype=qmm.QMM_BF16, what=""):
    y = run_qmm(x, M, w, N, K, transpose, y_dtype)
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, w.group_size, w.bits)
    return assert_within_tolerance(y, ref, absy, what)


def test_small_reference_case():
    """x [1, 512] . W[256, 512]^T at 4 bits, group 64, fp32 output."""
    w = synth.pr1_weight(0)
    x = synth.x_bf16(0, 1, 512)
    check(x, 1, w, 256, 512, True, qmm.QMM_F32, "pr1")


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("gs", (32, 128))
@pytest.mark.parametrize("M", (1, 3, 8, 9, 16))
def test_transposed_all_widths(bits, gs, M):
    # N = 200: a ragged last 16-row tile; K = 640 = five 128-code chunks.
    N, K = 200, 640
    w = synth.quant_weight(10 * bits + gs + M, N, K, bits, gs)
    x = synth.x_bf16(M + bits, M, K)
    check(x, M, w, N, K, True, what="bits=%d gs=%d M=%d" % (bits, gs, M))


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M", (1, 8, 16))
def test_transposed_many_tiles_ragged(bits, M):
    # N = 3000: 188 tiles of 16 rows, more than a GB300 has SMs and fewer than
    # two per SM; the last tile is ragged.  K = 640 = five chunks, fewer than
    # a block has warps.
    N, K = 3000, 640
    w = synth.quant_weight(300 + bits, N, K, bits, 64)
    x = synth.x_bf16(301 + M, M, K)
    check(x, M, w, N, K, True, qmm.QMM_F32, "many tiles bits=%d M=%d" % (bits, M))


@pytest.mark.parametrize("bits", (3, 4, 8))
def test_transposed_partial_chunk(bits):
    # K = 608 = 4 full 128-code chunks and 96 codes.
    N, K = 48, 608
    w = synth.quant_weight(71 + bits, N, K, bits, 32)
    x = synth.x_bf16(72, 2, K)
    check(x, 2, w, N, K, True, qmm.QMM_F32, "partial chunk")


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M", (1, 5, 16))
def test_not_transposed_all_widths(bits, M):
    # W stored [K, N], packed and grouped along N; K = 77 is odd.
    K, N = 77, 192
    w = synth.quant_weight(500 + bits + M, K, N, bits, 64)
    x = synth.x_bf16(600 + M, M, K)
    check(x, M, w, N, K, False, what="transpose=0 bits=%d M=%d" % (bits, M))


@pytest.mark.parametrize("bits", (4, 8))
@pytest.mark.parametrize("M", synth.DECODE_M)
def test_decode_full_size(bits, M):
    """x [M, 4096] . W[4096, 4096]^T at group 64: every output checked."""
    N, K = synth.DECODE_SHAPE
    w = synth.quant_weight(bits, N, K, bits, 64)
    x = synth.x_bf16(100 + M, M, K)
    check(x, M, w, N, K, True, what="decode b%d M%d" % (bits, M))


@pytest.mark.parametrize("bits", synth.ODD_BITS)
@pytest.mark.parametrize("gs", synth.ODD_GROUPS)
def test_odd_widths_full_size(bits, gs):
    """x [1, 4096] . W[11008, 4096]^T: every output checked."""
    N, K = synth.ODD_SHAPE
    w = synth.quant_weight(200 + bits + gs, N, K, bits, gs)
    x = synth.x_bf16(201, 1, K)
    check(x, 1, w, N, K, True, what="odd b%d g%d" % (bits, gs))


# Weights with more 16-row tiles than two 16-warp blocks per SM cover (N >
# 2 * 16 * 152) take 8-warp blocks: a ragged last tile, M up to 8, both output
# types, both dequantization forms (scales up to 0.2 leave the fast form's
# range); 6 and 8 bits keep 16-warp blocks.
@pytest.mark.parametrize("bits", (1, 2, 3, 4, 6, 8))
@pytest.mark.parametrize("M,gs,K,y_dtype,scale_hi", [
    (1, 32, 4096, qmm.QMM_BF16, 0.02),
    (5, 64, 4096, qmm.QMM_F32, 0.02),
    (8, 128, 2048, qmm.QMM_BF16, 0.2),
    (3, 64, 1024, qmm.QMM_F32, 0.2),
])
def test_many_row_tiles(bits, M, gs, K, y_dtype, scale_hi):
    N = 5003
    w = synth.quant_weight(300 + bits + M, N, K, bits, gs, scale_hi=scale_hi)
    x = synth.x_bf16(301 + M, M, K)
    check(x, M, w, N, K, True, y_dtype, what="many tiles b%d M%d g%d K%d" % (bits, M, gs, K))


@pytest.mark.parametrize("shape", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("transpose", (True, False))
def test_sweep_shapes_m16(shape, transpose):
    N, K = shape
    rows, cols = (N, K) if transpose else (K, N)
    w = synth.quant_weight(N + K + int(transpose), rows, cols, 4, 64)
    x = synth.x_bf16(7, 16, K)
    check(x, 16, w, N, K, transpose, what="sweep %s t=%d" % (shape, transpose))


@pytest.mark.parametrize("bits", (1, 4, 6, 8))
def test_weights_that_are_exactly_zero(bits):
    """Codes 2^(bits-1) with bias -scale * 2^(bits-1): every weight is exactly 0,
    so y must be 0 within the absolute 1e-6."""
    N, K = 64, 256
    w = synth.quant_weight(9, N, K, bits, 64)
    c = 1 << (bits - 1)
    codes = np.full((N, K), c, dtype=np.uint8)
    w.packed = oracle.pack(codes, bits)
    s = (w.scales.astype(np.uint32) << 16).view(np.float32)
    b = -(s * np.float32(c))                          # exact: times a power of two
    w.biases = (b.view(np.uint32) >> 16).astype(np.uint16)
    x = synth.x_bf16(10, 4, K)
    y = run_qmm(x, 4, w, N, K, True, qmm.QMM_F32)
    assert np.abs(y.cpu().numpy()).max() <= 1e-6


def test_zero_x_gives_zero():
    N, K = 32, 128
    w = synth.quant_weight(12, N, K, 5, 32)
    x = np.zeros((3, K), dtype=np.uint16)
    y = run_qmm(x, 3, w, N, K, True, qmm.QMM_F32)
    assert (y.cpu().numpy() == 0).all()


def test_constant_weight_matmul_exact():
    """Every code 0, scale 1, bias 1 or 2, x = ones(64): y = 64 or 128 (the
    construction of nuvec_core's gather_qmm doctest)."""
    N, K = 4, 64
    for bias_bits, want in ((0x3F80, 64.0), (0x4000, 128.0)):
        w = synth.QuantWeight(np.zeros((N, K // 8), np.uint32), np.full((N, 1), 0x3F80, np.uint16),
                              np.full((N, 1), bias_bits, np.uint16), N, K, 4, 64)
        x = np.full((1, K), 0x3F80, dtype=np.uint16)
        y = run_qmm(x, 1, w, N, K, True, qmm.QMM_F32)
        assert (y.cpu().numpy() == want).all()


@pytest.mark.parametrize("bits", (4, 8))
def test_chained_launches_with_programmatic_dependent_launch(bits):
    """With QMM_LAUNCH_PDL each decode launch may start before the previous
    kernel ends; it must still read the x that kernel wrote.  Chain
    y1 = x0 . W1^T, y2 = y1 . W2^T, y3 = y2 . W3^T back to back, then check
    every link against the oracle fed with the GPU's own intermediate."""
    N = K = 2048
    ws = [synth.quant_weight(900 + i + bits, N, K, bits, 64) for i in range(3)]
    dws = [weight(w) for w in ws]
    x0 = synth.x_bf16(901, 1, K)
    ys = [dev(x0)] + [empty_out((1, N), qmm.QMM_BF16) for _ in ws]
    prev = qmm.qmm_set_launch_flags(qmm.QMM_LAUNCH_PDL)
    try:
        for i, (w, (pw, ps, pb)) in enumerate(zip(ws, dws)):
            qmm.qmm_quantized_matmul(ys[i], 1, pw, ps, pb, N, K, 1, 64, bits, ys[i + 1], qmm.QMM_BF16)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_launch_flags(prev)
    for i, w in enumerate(ws):
        x_in = ys[i].cpu().numpy().view(np.uint16)
        ref, absy = oracle.qmm(x_in, 1, w.packed, w.scales, w.biases, N, K, True, 64, bits)
        assert_within_tolerance(ys[i + 1], ref, absy, "link %d" % i)


@pytest.mark.parametrize("M", (1, 4, 16))
@pytest.mark.parametrize("bits", (4, 8))
def test_x_on_a_16_byte_boundary(bits, M):
    # x 16- but not 32-byte aligned takes 16-byte loads instead of 32-byte
    # ones (M > 1); the results are the same bits as from an aligned x.
    N, K = 512, 1024
    w = synth.quant_weight(900 + bits, N, K, bits, 64)
    x = synth.x_bf16(901 + M, M, K)
    pw, ps, pb = weight(w)
    buf = torch.zeros(M * K + 16, dtype=torch.int16, device="cuda")
    xs = []
    for off in (0, 8):  # elements: 0 and 16 bytes past a 512-byte aligned base
        assert (buf.data_ptr() + 2 * off) % 32 == (16 if off else 0)
        buf[off:off + M * K] = dev(x).reshape(-1)
        y = empty_out((M, N), qmm.QMM_F32)
        qmm.qmm_quantized_matmul(buf[off:off + M * K], M, pw, ps, pb, N, K, 1, 64, bits, y,
                                 qmm.QMM_F32)
        torch.cuda.synchronize()
        xs.append(y.cpu().numpy())
    assert np.array_equal(xs[0].view(np.uint32), xs[1].view(np.uint32))
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, 64, bits)
    assert_within_tolerance(torch.from_numpy(xs[1]), ref, absy, "16-byte x bits=%d M=%d" % (bits, M))
