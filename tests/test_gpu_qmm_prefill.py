"""GPU parity of qmm_quantized_matmul on the tensor-core path (M > 16) against the
fp64 oracle: every checked output within 8e-3 * sum_k |x w| + 1e-6.  Small
shapes are checked in full; the full-size prefill shapes on sampled outputs
(whole rows and columns plus uniform samples)."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import assert_within_tolerance, dev, empty_out, host_f64, weight  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)


def run_qmm(x, M, w, N, K, transpose, y_dtype=qmm.QMM_BF16):
    pw, ps, pb = weight(w)
    y = empty_out((M, N), y_dtype)
    qmm.qmm_quantized_matmul(dev(x), M, pw, ps, pb, N, K, transpose, w.group_size, w.bits, y, y_dtype)
    torch.cuda.synchronize()
    return y


def check_full(x, M, w, N, K, transpose, y_dtype=qmm.QMM_BF16, what=""):
    y = run_qmm(x, M, w, N, K, transpose, y_dtype)
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, w.group_size, w.bits)
    return assert_within_tolerance(y, ref, absy, what)


def check_sampled(x, M, w, N, K, transpose, seed, y_dtype=qmm.QMM_BF16, what=""):
    y = run_qmm(x, M, w, N, K, transpose, y_dtype)
    g = synth.rng(seed)
    ms = [g.integers(0, M, 3000)]
    ns = [g.integers(0, N, 3000)]
    # two whole output rows and two whole columns, and the last corner
    for m in (0, M - 1):
        ms.append(np.full(N, m))
        ns.append(np.arange(N))
    for n in (0, N - 1):
        ms.append(np.arange(M))
        ns.append(np.full(M, n))
    ms, ns = np.concatenate(ms).astype(np.int64), np.concatenate(ns).astype(np.int64)
    ref, absy = oracle.qmm_sampled(x, M, w.packed, w.scales, w.biases, N, K, transpose,
                                   w.group_size, w.bits, ms, ns)
    got = host_f64(y)[ms, ns]
    err = np.abs(got - ref)
    bound = 8e-3 * absy + 1e-6
    assert (err <= bound).all(), "%s: %d of %d sampled outputs out of tolerance" % (
        what, (err > bound).sum(), err.size)


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M,N,K,gs", [(17, 256, 64, 64), (200, 300, 512, 32), (128, 512, 96, 32),
                                      (300, 64, 256, 128)])
def test_tensor_core_path_small(bits, M, N, K, gs):
    w = synth.quant_weight(1000 + bits + M + N, N, K, bits, gs)
    x = synth.x_bf16(2000 + M + bits, M, K)
    check_full(x, M, w, N, K, True, what="b%d M%d N%d K%d g%d" % (bits, M, N, K, gs))


@pytest.mark.parametrize("y_dtype", (qmm.QMM_F32, qmm.QMM_BF16))
def test_tensor_core_path_output_dtypes(y_dtype):
    M, N, K = 256, 520, 1024          # N not a multiple of 8: scalar stores on the edge
    w = synth.quant_weight(5, N, K, 4, 64)
    x = synth.x_bf16(6, M, K)
    check_full(x, M, w, N, K, True, y_dtype, "dtype %d" % y_dtype)


def test_many_tiles_per_block():
    """More output tiles than SMs: every block walks several tiles, so both TMEM
    accumulators and every pipeline stage are reused.  Every output is checked,
    so a fault on any later tile of a block shows."""
    M, N, K = 1024, 8192, 512          # 8 x 32 = 256 tiles
    w = synth.quant_weight(7, N, K, 4, 32)
    x = synth.x_bf16(8, M, K)
    check_full(x, M, w, N, K, True, what="many tiles")


def test_prefill_full_size():
    """x [2048, 4096] . W[14336, 4096]^T at 4 bits, group 64."""
    p = synth.PREFILL
    M, N, K = p["M"], p["N"], p["K"]
    w = synth.quant_weight(3, N, K, 4, 64)
    x = synth.x_bf16(4, M, K)
    check_sampled(x, M, w, N, K, True, seed=11, what="prefill")


@pytest.mark.parametrize("shape", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("M", (128, 2048))
@pytest.mark.parametrize("bits", (4, 8))
def test_sweep_shapes(shape, M, bits):
    N, K = shape
    w = synth.quant_weight(N + K + bits, N, K, bits, 64)
    x = synth.x_bf16(M + bits, M, K)
    check_sampled(x, M, w, N, K, True, seed=M + N, what="sweep %s M%d b%d" % (shape, M, bits))


# -- transpose = false: W stored [K, N], packed and grouped along N ------------

@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M,N,K,gs", [(17, 256, 64, 64), (200, 320, 136, 32), (300, 512, 96, 128)])
def test_not_transposed_tensor_core_small(bits, M, N, K, gs):
    w = synth.quant_weight(3000 + bits + M + N, K, N, bits, gs)     # stored [K, N]
    x = synth.x_bf16(3100 + M + bits, M, K)
    check_full(x, M, w, N, K, False, what="t0 b%d M%d N%d K%d g%d" % (bits, M, N, K, gs))


def test_not_transposed_odd_k_falls_back():
    """K = 77: x rows are not 16-byte aligned, so the tensor-map path cannot
    address them; the call must still be correct."""
    M, N, K = 40, 128, 77
    w = synth.quant_weight(41, K, N, 4, 32)
    x = synth.x_bf16(42, M, K)
    check_full(x, M, w, N, K, False, qmm.QMM_F32, "t0 odd K")


def test_prefill_not_transposed_full_size():
    """x [2048, 4096] . W with W stored [4096, 14336] at 4 bits, group 64."""
    p = synth.PREFILL
    M, N, K = p["M"], p["N"], p["K"]
    w = synth.quant_weight(13, K, N, 4, 64)
    x = synth.x_bf16(14, M, K)
    check_sampled(x, M, w, N, K, False, seed=15, what="prefill t0")


# Split-K: with fewer output tiles than SMs, each tile's K range is split and
# the fp32 partials are added by a second kernel.
@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("y_dtype", (qmm.QMM_F32, qmm.QMM_BF16))
def test_split_k_ragged_n(bits, y_dtype):
    # N = 202: not a multiple of 4, so the partials are added one element at a
    # time; one 256-row tile, so K = 1024 (16 k-blocks) is split 8 ways.
    M, N, K = 40, 202, 1024
    w = synth.quant_weight(500 + bits, N, K, bits, 32)
    x = synth.x_bf16(501 + bits, M, K)
    check_full(x, M, w, N, K, True, y_dtype, "split-K ragged N bits=%d" % bits)


@pytest.mark.parametrize("bits", (2, 4, 6))
def test_split_k_not_transposed(bits):
    M, N, K = 64, 256, 1024
    w = synth.quant_weight(510 + bits, K, N, bits, 64)
    x = synth.x_bf16(511 + bits, M, K)
    check_full(x, M, w, N, K, False, qmm.QMM_F32, "split-K W stored [K, N] bits=%d" % bits)


def test_split_k_repeats_bit_for_bit():
    # The partials are added in a fixed order: two runs give the same bits.
    M, N, K = 128, 1024, 4096
    w = synth.quant_weight(520, N, K, 4, 64)
    x = synth.x_bf16(521, M, K)
    a = run_qmm(x, M, w, N, K, True, qmm.QMM_F32).cpu()
    b = run_qmm(x, M, w, N, K, True, qmm.QMM_F32).cpu()
    assert torch.equal(a, b)
