"""GPU parity of qmm_gather_qmm against the oracle's gather_qmm: every output
within 8e-3 * sum_k |x w| + 1e-6, the doctest values exactly, and index
errors reported through the device error word."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth
from conftest import ints, load_golden

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import assert_within_tolerance, dev, empty_out, host_f64  # noqa: E402


def experts(seed, E, rows, cols, bits, gs):
    ws = [synth.quant_weight(seed + e, rows, cols, bits, gs) for e in range(E)]
    return (np.stack([w.packed for w in ws]), np.stack([w.scales for w in ws]),
            np.stack([w.biases for w in ws]))


def run(x, XB, M, packed, s, b, E, N, K, lhs, rhs, B, transpose, gs, bits, sorted_=False,
        y_dtype=qmm.QMM_F32):
    y = empty_out((B, M, N), y_dtype)
    qmm.qmm_gather_qmm(dev(x), XB, M, dev(packed), dev(s), dev(b), E, N, K,
                       None if lhs is None else dev(lhs), None if rhs is None else dev(rhs), B,
                       transpose, gs, bits, sorted_, y, y_dtype)
    torch.cuda.synchronize()
    return y


def check(x, XB, M, packed, s, b, E, N, K, lhs, rhs, B, transpose, gs, bits, sorted_=False,
          y_dtype=qmm.QMM_F32, what=""):
    y = run(x, XB, M, packed, s, b, E, N, K, lhs, rhs, B, transpose, gs, bits, sorted_, y_dtype)
    ref, absy = oracle.gather_qmm(x, XB, M, packed, s, b, E, N, K, lhs, rhs, transpose, gs, bits)
    return assert_within_tolerance(y, ref, absy, what)


def test_doctest_values():
    g = load_golden("gather_qmm_experts.txt")
    E, N, K, bits, gs = (int(g[k][0]) for k in ("experts", "N", "K", "bits", "group_size"))
    rhs = np.array(ints(g["rhs"]), dtype=np.uint32)
    packed = np.zeros((E, N, K * bits // 32), dtype=np.uint32)
    s = np.full((E, N, K // gs), 0x3F80, dtype=np.uint16)
    b = np.stack([np.full((N, K // gs), int(np.float32(e + 1).view(np.uint32) >> 16),
                          dtype=np.uint16) for e in range(E)])
    x = np.full((len(rhs), 1, K), 0x3F80, dtype=np.uint16)
    y = host_f64(run(x, len(rhs), 1, packed, s, b, E, N, K, None, rhs, len(rhs), 1, gs, bits))
    assert list(y.reshape(-1)[:5]) == [float(v) for v in g["expect_first5"]]


@pytest.mark.parametrize("bits", (2, 4, 5, 8))
@pytest.mark.parametrize("M", (1, 3, 16, 20))
@pytest.mark.parametrize("K", (512, 320))   # TMA kernel (K % 128 == 0), plain loads
def test_transposed_random_indices(bits, M, K):
    E, XB, B, N, gs = 5, 4, 9, 200, 32
    packed, s, b = experts(100 * bits + M, E, N, K, bits, gs)
    x = synth.x_bf16(7 + M, XB * M, K)
    g = np.random.default_rng(bits + M + K)
    lhs = g.integers(0, XB, B).astype(np.uint32)
    rhs = g.integers(0, E, B).astype(np.uint32)
    check(x, XB, M, packed, s, b, E, N, K, lhs, rhs, B, 1, gs, bits,
          what="transposed bits=%d M=%d K=%d" % (bits, M, K))


@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("M", (1, 17))
def test_not_transposed_random_indices(bits, M):
    E, XB, B, N, K, gs = 3, 2, 5, 256, 96, 64
    packed, s, b = experts(200 + bits, E, K, N, bits, gs)
    x = synth.x_bf16(9 + M, XB * M, K)
    g = np.random.default_rng(bits * M)
    lhs = g.integers(0, XB, B).astype(np.uint32)
    rhs = g.integers(0, E, B).astype(np.uint32)
    check(x, XB, M, packed, s, b, E, N, K, lhs, rhs, B, 0, gs, bits, y_dtype=qmm.QMM_BF16,
          what="W stored [K, N] bits=%d M=%d" % (bits, M))


def test_default_indices():
    E = XB = B = 3
    M, N, K, bits, gs = 2, 64, 256, 4, 64
    packed, s, b = experts(300, E, N, K, bits, gs)
    x = synth.x_bf16(301, XB * M, K)
    check(x, XB, M, packed, s, b, E, N, K, None, None, B, 1, gs, bits, what="defaults")


@pytest.mark.parametrize("bits", (4, 8))
@pytest.mark.parametrize("y_dtype", (qmm.QMM_F32, qmm.QMM_BF16))
def test_sorted_runs(bits, y_dtype):
    # 40 tokens over 8 experts, two of them unused, runs of 1 to 12 tokens
    # (longer than one 8-row pass); N = 200 leaves a ragged last tile.
    E, N, K, gs = 8, 200, 1024, 64
    packed, s, b = experts(400 + bits, E, N, K, bits, gs)
    g = np.random.default_rng(bits)
    rhs = np.sort(g.choice([0, 1, 2, 4, 5, 7], 40, p=[.3, .05, .1, .05, .2, .3])).astype(np.uint32)
    B = len(rhs)
    x = synth.x_bf16(401, B, K)
    check(x, B, 1, packed, s, b, E, N, K, None, rhs, B, 1, gs, bits, sorted_=True, y_dtype=y_dtype,
          what="sorted runs bits=%d" % bits)


@pytest.mark.parametrize("bits", (3, 4, 5))
@pytest.mark.parametrize("sorted_", (False, True))
@pytest.mark.parametrize("y_dtype", (qmm.QMM_F32, qmm.QMM_BF16))
def test_many_row_tiles(bits, sorted_, y_dtype):
    # 8 experts of 1000 rows (63 row tiles, the last ragged) and 24 slots:
    # more blocks than two a multiprocessor, so the decode runs 8-warp blocks.
    E, N, K, gs = 8, 1000, 512, 64
    packed, s, b = experts(800 + bits, E, N, K, bits, gs)
    rhs = np.random.default_rng(bits).integers(0, E, 24).astype(np.uint32)
    if sorted_:
        rhs = np.sort(rhs)
    B = len(rhs)
    x = synth.x_bf16(801, B, K)
    check(x, B, 1, packed, s, b, E, N, K, None, rhs, B, 1, gs, bits, sorted_=sorted_,
          y_dtype=y_dtype, what="many row tiles bits=%d sorted=%d" % (bits, sorted_))


@pytest.mark.parametrize("sorted_", (False, True))
def test_index_past_the_weights_gives_zeros_and_is_reported(sorted_):
    E, N, K, bits, gs = 3, 64, 256, 4, 64
    packed, s, b = experts(500, E, N, K, bits, gs)
    rhs = np.array([0, 2, 2, 9, 11], dtype=np.uint32)   # sorted; the last two are past E
    B = len(rhs)
    x = synth.x_bf16(501, B, K)
    qmm.qmm_get_device_error()                            # start clean
    y = run(x, B, 1, packed, s, b, E, N, K, None, rhs, B, 1, gs, bits, sorted_)
    assert qmm.qmm_get_device_error() == qmm.QMM_ERR_INDEX
    assert qmm.qmm_get_device_error() == qmm.QMM_OK      # reading clears it
    got = host_f64(y)
    assert (got[3:] == 0).all()
    ref, absy = oracle.gather_qmm(x, B, 1, packed, s, b, E, N, K, None, rhs, True, gs, bits)
    assert_within_tolerance(y, ref, absy, "past the weights")


def test_more_batches_than_one_grid_holds():
    # 70000 output batches: the launch is split over the grid's z dimension.
    E, N, K, bits, gs = 2, 16, 128, 4, 32
    packed, s, b = experts(600, E, N, K, bits, gs)
    B = 70000
    rhs = (np.arange(B) % E).astype(np.uint32)
    x = synth.x_bf16(601, 4, K)
    lhs = (np.arange(B) % 4).astype(np.uint32)
    y = host_f64(run(x, 4, 1, packed, s, b, E, N, K, lhs, rhs, B, 1, gs, bits))
    # batch b depends only on (lhs[b], rhs[b]) = (b % 4, b % 2): period 4
    ref, absy = oracle.gather_qmm(x, 4, 1, packed, s, b, E, N, K, lhs[:4], rhs[:4], True, gs, bits)
    want = np.tile(ref, (B // 4, 1, 1))
    bound = 8e-3 * np.tile(absy, (B // 4, 1, 1)) + 1e-6
    assert (np.abs(y - want) <= bound).all()


@pytest.mark.parametrize("bits,y_dtype", ((4, qmm.QMM_BF16), (3, qmm.QMM_F32), (8, qmm.QMM_F32)))
def test_sorted_long_runs_take_the_tensor_cores(bits, y_dtype):
    """Prefill-sized mixture of experts: 1100 tokens over 8 experts (at least
    32 per expert on average), sorted, one x row each -- the grouped tcgen05
    path.  Runs of 0, 1, 255, 256, 257 and 600 tokens (row tiles of 256, a
    ragged last tile, an empty expert), N = 384 (a ragged column tile), and
    tokens whose index is past the last expert (zero rows, index bit)."""
    E, N, K, gs = 8, 384, 512, 64
    runs = [255, 0, 256, 1, 257, 600, 17, 40]
    bad = 12                                   # tokens with index E (past the experts)
    rhs = np.concatenate([np.full(r, e, dtype=np.uint32) for e, r in enumerate(runs)] +
                         [np.full(bad, E, dtype=np.uint32)])
    B = rhs.size
    assert B >= 32 * E
    packed, s, b = experts(700 + bits, E, N, K, bits, gs)
    x = synth.x_bf16(701 + bits, B, K)
    y = run(x, B, 1, packed, s, b, E, N, K, None, rhs, B, 1, gs, bits, True, y_dtype)
    assert qmm.qmm_get_device_error() == qmm.QMM_ERR_INDEX
    ref, absy = oracle.gather_qmm(x, B, 1, packed, s, b, E, N, K, None, rhs, 1, gs, bits)
    assert_within_tolerance(y, ref, absy, "grouped bits=%d" % bits)
    assert (host_f64(y)[B - bad:] == 0).all()
    # the same call again gives the same bits (no accumulation across calls)
    y2 = run(x, B, 1, packed, s, b, E, N, K, None, rhs, B, 1, gs, bits, True, y_dtype)
    assert torch.equal(y, y2)
