"""GPU parity, against the oracle, of every workload the benchmark prints that
the other test files do not already cover in the launch configuration the
benchmark times:

* the layer sweep at M = 1 (all four shapes, 4 and 8 bits), every output --
  this includes [4096, 14336], whose K range the decode kernel splits across a
  cluster of blocks;
* the layer sweep at M = 16 and 8 bits, every output;
* the sweep's bf16 dequantize of each weight, bit for bit on sampled rows;
* the small reference case (x [1, 512] . W[256, 512]^T, fp32 out) and its
  fp32 dequantize, which the benchmark times as latency lines.

Matmul outputs must satisfy |y - y_ref| <= 8e-3 * sum_k |x w| + 1e-6 against
the fp64 oracle (nuvec_core quantized.rs, `quantized_matmul`); dequantize is
bit-exact (`dequantize`)."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import (assert_within_tolerance, dev, empty_out, host_bits,  # noqa: E402
                      oracle_bits, weight)


def qmm_full(x, M, w, N, K, y_dtype=qmm.QMM_BF16, what=""):
    pw, ps, pb = weight(w)
    y = empty_out((M, N), y_dtype)
    qmm.qmm_quantized_matmul(dev(x), M, pw, ps, pb, N, K, 1, w.group_size, w.bits, y, y_dtype)
    torch.cuda.synchronize()
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, w.group_size, w.bits)
    return assert_within_tolerance(y, ref, absy, what)


@pytest.mark.parametrize("shape", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("bits", (4, 8))
def test_sweep_m1_every_output(shape, bits):
    N, K = shape
    w = synth.quant_weight(170 + N // 1024 + K // 1024 + bits, N, K, bits, 64)
    x = synth.x_bf16(171 + bits, 1, K)
    qmm_full(x, 1, w, N, K, what="sweep %s M1 b%d" % (shape, bits))


@pytest.mark.parametrize("shape", synth.SWEEP_SHAPES)
def test_sweep_m16_8bit_every_output(shape):
    N, K = shape
    w = synth.quant_weight(180 + N // 1024 + K // 1024, N, K, 8, 64)
    x = synth.x_bf16(181, 16, K)
    qmm_full(x, 16, w, N, K, what="sweep %s M16 b8" % (shape,))


@pytest.mark.parametrize("shape", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("bits", (4, 8))
def test_sweep_dequantize_bf16_sampled_rows(shape, bits):
    """Full dequantize of the sweep weight to bf16; 256 random rows plus the
    first and last checked bit for bit."""
    N, K = shape
    w = synth.quant_weight(190 + N // 1024 + K // 1024 + bits, N, K, bits, 64)
    pw, ps, pb = weight(w)
    out = empty_out((N, K), qmm.QMM_BF16)
    qmm.qmm_dequantize(pw, ps, pb, N, K, 64, bits, out, qmm.QMM_BF16)
    torch.cuda.synchronize()
    got = host_bits(out)
    rows = np.concatenate([synth.indices(191, 256, N), np.array([0, N - 1], np.uint32)])
    want, bad = oracle.rows(w.packed, w.scales, w.biases, N, K, rows, 64, bits, "bf16")
    assert bad == 0 and (got[rows.astype(np.int64)] == oracle_bits(want)).all()


def test_small_reference_case_as_benchmarked():
    """x [1, 512] . W[256, 512]^T at 4 bits, group 64, fp32 out, then the fp32
    dequantize of W: the two launches the benchmark's reference-case line
    times, on the same seeded inputs."""
    w = synth.pr1_weight(0)
    x = synth.x_bf16(0, 1, 512)
    qmm_full(x, 1, w, 256, 512, qmm.QMM_F32, "reference case")
    pw, ps, pb = weight(w)
    out = empty_out((256, 512), qmm.QMM_F32)
    qmm.qmm_dequantize(pw, ps, pb, 256, 512, 64, 4, out, qmm.QMM_F32)
    torch.cuda.synchronize()
    want = oracle.dequantize(w.packed, w.scales, w.biases, 256, 512, 64, 4, "f32")
    assert (host_bits(out) == oracle_bits(want)).all()
