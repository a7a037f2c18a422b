"""GPU parity of qmm_dequantize and qmm_rows against the CPU oracle: bit-exact
for fp32 output and for bf16 output (round to nearest even)."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import dev, empty_out, host_bits, oracle_bits, weight  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)
DTYPES = {"f32": qmm.QMM_F32, "bf16": qmm.QMM_BF16}


def run_dequant(w, out_dtype):
    pw, ps, pb = weight(w)
    out = empty_out((w.rows, w.cols), out_dtype)
    qmm.qmm_dequantize(pw, ps, pb, w.rows, w.cols, w.group_size, w.bits, out, out_dtype)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("gs", (32, 64, 128))
@pytest.mark.parametrize("dt", sorted(DTYPES))
def test_dequantize_bit_exact(bits, gs, dt):
    # 37 rows (ragged), 2304 columns: two blocks per row, the second partial.
    w = synth.quant_weight(1000 + 17 * bits + gs, 37, 2304, bits, gs)
    got = host_bits(run_dequant(w, DTYPES[dt]))
    want = oracle_bits(oracle.dequantize(w.packed, w.scales, w.biases, w.rows, w.cols, gs, bits, dt))
    assert (got == want).all()


@pytest.mark.parametrize("shape", [(1, 32), (3, 96), (5, 4096 + 128)])
@pytest.mark.parametrize("bits", (3, 4, 8))
def test_dequantize_small_and_ragged(shape, bits):
    w = synth.quant_weight(77 + bits, shape[0], shape[1], bits, 32)
    got = host_bits(run_dequant(w, qmm.QMM_BF16))
    want = oracle_bits(oracle.dequantize(w.packed, w.scales, w.biases, w.rows, w.cols, 32, bits, "bf16"))
    assert (got == want).all()


def test_dequantize_small_reference_case_fp32():
    """W [256, 512] at 4 bits, group 64, dequantized to fp32."""
    w = synth.pr1_weight(0)
    got = host_bits(run_dequant(w, qmm.QMM_F32))
    want = oracle_bits(oracle.dequantize(w.packed, w.scales, w.biases, 256, 512, 64, 4, "f32"))
    assert (got == want).all()


def test_zero_codes_dequantize_to_bias():
    w = synth.quant_weight(5, 8, 256, 4, 64)
    w.packed[:] = 0
    got = host_bits(run_dequant(w, qmm.QMM_BF16))
    assert (got == np.repeat(w.biases, 64, axis=1)).all()


@pytest.mark.parametrize("bits", (4, 8))
def test_dequantize_full_size_sampled_rows(bits):
    """[14336, 4096] at group 64 to bf16; 300 random rows checked bit for bit."""
    w = synth.quant_weight(40 + bits, 14336, 4096, bits, 64)
    got = host_bits(run_dequant(w, qmm.QMM_BF16))
    rows = synth.indices(9, 300, w.rows)
    want, bad = oracle.rows(w.packed, w.scales, w.biases, w.rows, w.cols, rows, 64, bits, "bf16")
    assert bad == 0 and (got[rows.astype(np.int64)] == oracle_bits(want)).all()


def run_rows(w, idx, out_dtype):
    pw, ps, pb = weight(w)
    di = dev(idx)
    out = empty_out((idx.size, w.cols), out_dtype)
    qmm.qmm_rows(pw, ps, pb, w.rows, w.cols, di, idx.size, w.group_size, w.bits, out, out_dtype)
    status = qmm.qmm_get_device_error()
    return out, status


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("dt", sorted(DTYPES))
def test_rows_bit_exact_with_duplicates(bits, dt):
    w = synth.quant_weight(300 + bits, 1000, 640, bits, 64)
    idx = synth.indices(301, 257, 1000)
    idx[5] = idx[9] = idx[100]                       # duplicates
    idx[0], idx[-1] = 0, 999                         # first and last rows
    out, status = run_rows(w, idx, DTYPES[dt])
    want, bad = oracle.rows(w.packed, w.scales, w.biases, 1000, 640, idx, 64, bits, dt)
    assert status == qmm.QMM_OK and bad == 0
    assert (host_bits(out) == oracle_bits(want)).all()


def test_rows_out_of_table_index_reports_and_zeroes():
    w = synth.quant_weight(31, 50, 128, 4, 32)
    idx = np.array([3, 50, 0xFFFFFFFF, 49, 7], dtype=np.uint32)
    out, status = run_rows(w, idx, qmm.QMM_BF16)
    want, bad = oracle.rows(w.packed, w.scales, w.biases, 50, 128, idx, 32, 4, "bf16")
    assert bad == 2 and status == qmm.QMM_ERR_INDEX
    assert (host_bits(out) == oracle_bits(want)).all()
    # The error word is cleared by reading it.
    assert qmm.qmm_get_device_error() == qmm.QMM_OK


def test_rows_full_size_embedding_gather():
    """4096 uniform indices into a [128256, 4096] table at 4 bits, group 64."""
    T, C = synth.ROWS_TABLE
    w = synth.quant_weight(2, T, C, 4, 64)
    idx = synth.indices(3, synth.ROWS_GATHER, T)
    out, status = run_rows(w, idx, qmm.QMM_BF16)
    want, bad = oracle.rows(w.packed, w.scales, w.biases, T, C, idx, 64, 4, "bf16")
    assert status == qmm.QMM_OK and bad == 0
    assert (host_bits(out) == oracle_bits(want)).all()


@pytest.mark.parametrize("bits", (3, 4, 8))
@pytest.mark.parametrize("dt", sorted(DTYPES))
def test_dequantize_and_rows_into_16_byte_aligned_outputs(bits, dt):
    """Outputs 16 bytes past a 32-byte boundary (the minimum alignment the calls
    accept) take the kernels' 16-byte stores; the 32-byte-aligned ones their
    32-byte stores.  Both give the same bits."""
    w = synth.quant_weight(70 + bits, 21, 640, bits, 64)
    pw, ps, pb = weight(w)
    esz = 4 if dt == "f32" else 2
    want = oracle_bits(oracle.dequantize(w.packed, w.scales, w.biases, 21, 640, 64, bits, dt))
    big = empty_out((21 * 640 + 64,), DTYPES[dt])
    assert big.data_ptr() % 32 == 0
    off = 16 // esz
    out = big[off:off + 21 * 640]
    qmm.qmm_dequantize(pw, ps, pb, 21, 640, 64, bits, out.data_ptr(), DTYPES[dt])
    torch.cuda.synchronize()
    assert (host_bits(out).reshape(21, 640) == want).all()
    idx = synth.indices(71, 9, 21)
    outr = big[off:off + 9 * 640]
    qmm.qmm_rows(pw, ps, pb, 21, 640, dev(idx), 9, 64, bits, outr.data_ptr(), DTYPES[dt])
    torch.cuda.synchronize()
    assert (host_bits(outr).reshape(9, 640) == want[idx]).all()
