"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- values printed on the pages (tests/golden), a library
routine (numpy's bit unpacker, torch's bf16 rounding, numpy matmul), closed
forms and brute force on tiny shapes.  A plausible mistake in the oracle (MSB
first, bias subtracted, bias dropped, a wrong group index, a transposed
operand, truncation instead of round-to-nearest-even) fails at least one."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import synth
from conftest import ints, load_golden

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)


# -- independent helpers (numpy / torch library routines) -------------------

def np_codes(packed, cols, bits):
    """Codes via numpy's unpackbits on the little-endian bytes of the words."""
    packed = np.atleast_2d(np.asarray(packed, dtype="<u4"))
    stream = np.unpackbits(packed.view(np.uint8), axis=1, bitorder="little")
    stream = stream[:, : cols * bits].reshape(packed.shape[0], cols, bits).astype(np.uint32)
    return (stream << np.arange(bits, dtype=np.uint32)).sum(axis=2).astype(np.uint32)


def bf16_f64(u16):
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def np_dense_f64(w):
    """dequant(W) in fp64 with numpy's unpacker and np.repeat for the groups."""
    c = np_codes(w.packed, w.cols, w.bits).astype(np.float64)
    s = np.repeat(bf16_f64(w.scales), w.group_size, axis=1)
    b = np.repeat(bf16_f64(w.biases), w.group_size, axis=1)
    return s * c + b


def torch_bf16_bits(f32):
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


# -- values printed on the pages ---------------------------------------------

def _golden_weight(g):
    words = np.array(ints(g["words"]), dtype=np.uint32)[None, :]
    bits, cols, gs = int(g["bits"][0]), int(g["cols"][0]), int(g["group_size"][0])
    groups = cols // gs
    s = np.full((1, groups), int(g["scale_bf16"][0], 0), dtype=np.uint16)
    b = np.full((1, groups), int(g["bias_bf16"][0], 0), dtype=np.uint16)
    return words, s, b, cols, gs, bits


def test_lsb_first_plus_bias():
    g = load_golden("lsb_first_plus_bias.txt")
    words, s, b, cols, gs, bits = _golden_weight(g)
    out = oracle.dequantize(words, s, b, 1, cols, gs, bits, "f32")
    assert out.ravel().tolist() == [float(v) for v in g["expect_f32"]]
    assert oracle.unpack(words, cols, bits).ravel().tolist() == ints(g["codes"])


def test_identity_shape():
    g = load_golden("identity_shape.txt")
    words, s, b, cols, gs, bits = _golden_weight(g)
    out = oracle.dequantize(words, s, b, 1, cols, gs, bits, "f32")
    assert out.size == int(g["expect_len"][0])
    assert out.ravel().tolist() == [float(v) for v in g["expect_f32"]]


def test_int8_byte_layout():
    g = load_golden("int8_byte_layout.txt")
    words = np.array(ints(g["words"]), dtype=np.uint32)
    codes = oracle.unpack(words, int(g["cols"][0]), int(g["bits"][0]))
    assert codes.ravel().tolist() == ints(g["codes"])


def test_pack_shape():
    g = load_golden("pack_shape.txt")
    rows, cols = ints(g["weight_shape"])
    bits = int(g["bits"][0])
    codes = np.arange(rows * cols, dtype=np.uint8).reshape(rows, cols) % (1 << bits)
    packed = oracle.pack(codes, bits)
    assert list(packed.shape) == ints(g["packed_shape"])
    assert oracle.unpack(packed, cols, bits).shape == (rows, cols)


def test_three_bit_stream_by_hand():
    g = load_golden("three_bit_stream.txt")
    codes = np.array(ints(g["codes"]), dtype=np.uint8)[None, :]
    packed = oracle.pack(codes, int(g["bits"][0]))
    assert packed.ravel().tolist() == ints(g["words"])
    assert oracle.unpack(packed, codes.shape[1], 3).ravel().tolist() == ints(g["codes"])


def test_constant_weight_matmul():
    g = load_golden("constant_weight_matmul.txt")
    N, K, bits, gs = (int(g[k][0]) for k in ("N", "K", "bits", "group_size"))
    packed = np.zeros((N, K * bits // 32), dtype=np.uint32)
    x = np.full((1, K), 0x3F80, dtype=np.uint16)            # ones
    s = np.full((N, K // gs), 0x3F80, dtype=np.uint16)      # 1.0
    for bias, want in zip(g["bias_values"], g["expect_y"]):
        bias_bits = int(np.float32(float(bias)).view(np.uint32) >> 16)
        b = np.full((N, K // gs), bias_bits, dtype=np.uint16)
        y, a = oracle.qmm(x, 1, packed, s, b, N, K, True, gs, bits)
        assert (y == float(want)).all() and (a == float(want)).all()


# -- library routines and closed forms --------------------------------------

@pytest.mark.parametrize("bits", ALL_BITS)
def test_unpack_matches_numpy_unpackbits(bits):
    g = synth.rng(100 + bits)
    cols = 256
    packed = synth.random_words(g, 5, cols, bits)
    assert (oracle.unpack(packed, cols, bits) == np_codes(packed, cols, bits)).all()


@pytest.mark.parametrize("bits", ALL_BITS)
def test_pack_unpack_round_trip(bits):
    g = synth.rng(200 + bits)
    packed = synth.random_words(g, 3, 128, bits)
    codes = oracle.unpack(packed, 128, bits)
    assert codes.max() <= (1 << bits) - 1
    assert (oracle.pack(codes, bits) == packed).all()


@pytest.mark.parametrize("bits", ALL_BITS)
def test_zero_codes_give_bias(bits):
    w = synth.quant_weight(7, 6, 128, bits, 32)
    w.packed[:] = 0
    out = oracle.dequantize(w.packed, w.scales, w.biases, 6, 128, 32, bits, "f32")
    assert (out.astype(np.float64) == np.repeat(bf16_f64(w.biases), 32, axis=1)).all()


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("gs", (32, 64, 128))
def test_dequant_f32_is_exact_value_rounded_once(bits, gs):
    """fp32 dequant = the exact fp64 s*c+b rounded once to fp32 (the product is
    exact, so only the add rounds); group index from np.repeat."""
    w = synth.quant_weight(1000 + 10 * bits + gs, 7, 256, bits, gs)
    out = oracle.dequantize(w.packed, w.scales, w.biases, 7, 256, gs, bits, "f32")
    assert (out == np_dense_f64(w).astype(np.float32)).all()


def test_bf16_rounding_matches_torch():
    g = synth.rng(5)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32) * 10.0,
        # exact ties between two bf16 values, both parities
        ((np.arange(64, dtype=np.uint32) << 16) | 0x8000 | 0x3F800000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -3e-39, 3.3895314e38, np.inf, -np.inf], np.float32),
    ])
    mine = oracle.f32_to_bf16_array(vals)
    assert (mine == torch_bf16_bits(vals)).all()
    nan = oracle.f32_to_bf16(float("nan"))
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


@pytest.mark.parametrize("bits", (3, 4, 8))
def test_dequant_bf16_is_rne_of_f32(bits):
    w = synth.quant_weight(11, 9, 512, bits, 64)
    f = oracle.dequantize(w.packed, w.scales, w.biases, 9, 512, 64, bits, "f32")
    h = oracle.dequantize(w.packed, w.scales, w.biases, 9, 512, 64, bits, "bf16")
    assert (h == torch_bf16_bits(f)).all()


def test_thread_count_does_not_change_results():
    w = synth.quant_weight(12, 33, 256, 5, 32)
    a = oracle.dequantize(w.packed, w.scales, w.biases, 33, 256, 32, 5, "f32", nthreads=1)
    b = oracle.dequantize(w.packed, w.scales, w.biases, 33, 256, 32, 5, "f32", nthreads=7)
    assert (a == b).all()


# -- matmul -------------------------------------------------------------------

def _brute_force(x_u16, dense_kn):
    """A naive triple loop over (m, n, k) in Python floats (fp64)."""
    x = bf16_f64(x_u16)
    M, K = x.shape
    N = dense_kn.shape[1]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[m, k] * dense_kn[k, n]
            y[m, n] = acc
    return y


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("K", (32, 64, 128))
@pytest.mark.parametrize("transpose", (True, False))
def test_qmm_brute_force_tiny(bits, K, transpose):
    M, N = 3, 8 if transpose else 32        # transpose=False packs along N
    gs = 32
    x = synth.x_bf16(300 + bits, M, K)
    if transpose:
        w = synth.quant_weight(400 + bits + K, N, K, bits, gs)   # stored [N, K]
        dense_kn = np_dense_f64(w).T
    else:
        w = synth.quant_weight(500 + bits + K, K, N, bits, gs)   # stored [K, N]
        dense_kn = np_dense_f64(w)
    y, a = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits)
    want = _brute_force(x, dense_kn)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    want_abs = np.abs(bf16_f64(x))[:, :, None] * np.abs(dense_kn)[None, :, :]
    assert np.allclose(a, want_abs.sum(axis=1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("transpose", (True, False))
def test_qmm_matches_numpy_matmul(transpose):
    M, K, bits, gs = 5, 256, 4, 64
    N = 96 if transpose else 128            # packed along N when not transposed
    x = synth.x_bf16(21, M, K)
    if transpose:
        w = synth.quant_weight(22, N, K, bits, gs)
        dense_kn = np_dense_f64(w).T
    else:
        w = synth.quant_weight(23, K, N, bits, gs)
        dense_kn = np_dense_f64(w)
    y, _ = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits)
    assert np.allclose(y, bf16_f64(x) @ dense_kn, rtol=1e-12, atol=1e-12)


def test_transpose_flag_is_not_a_no_op():
    """With a square weight the two layouts give different products."""
    K = N = 64
    x = synth.x_bf16(31, 2, K)
    w = synth.quant_weight(32, N, K, 4, 32)
    y_t, _ = oracle.qmm(x, 2, w.packed, w.scales, w.biases, N, K, True, 32, 4)
    y_n, _ = oracle.qmm(x, 2, w.packed, w.scales, w.biases, N, K, False, 32, 4)
    dense = np_dense_f64(w)
    assert np.allclose(y_t, bf16_f64(x) @ dense.T, rtol=1e-12)
    assert np.allclose(y_n, bf16_f64(x) @ dense, rtol=1e-12)
    assert not np.allclose(y_t, y_n)


def test_qmm_sampled_matches_full():
    M, N, K = 4, 64, 128
    x = synth.x_bf16(41, M, K)
    w = synth.quant_weight(42, N, K, 6, 64)
    y, a = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, 64, 6)
    g = synth.rng(43)
    ms = g.integers(0, M, 50)
    ns = g.integers(0, N, 50)
    ys, as_ = oracle.qmm_sampled(x, M, w.packed, w.scales, w.biases, N, K, True, 64, 6, ms, ns)
    assert (ys == y[ms, ns]).all() and (as_ == a[ms, ns]).all()


# -- rows -------------------------------------------------------------------

def test_rows_is_a_gather_of_dequantize():
    w = synth.quant_weight(51, 40, 256, 3, 64)
    idx = np.array([5, 0, 39, 5, 17], dtype=np.uint32)
    out, bad = oracle.rows(w.packed, w.scales, w.biases, 40, 256, idx, 64, 3, "f32")
    dense = np_dense_f64(w).astype(np.float32)
    assert bad == 0 and (out == dense[idx]).all()


def test_rows_out_of_table_gives_zero_row():
    w = synth.quant_weight(52, 10, 64, 4, 32)
    idx = np.array([3, 10, 4000000000, 9], dtype=np.uint32)
    out, bad = oracle.rows(w.packed, w.scales, w.biases, 10, 64, idx, 32, 4, "bf16")
    assert bad == 2
    assert (out[1] == 0).all() and (out[2] == 0).all()
    full = oracle.dequantize(w.packed, w.scales, w.biases, 10, 64, 32, 4, "bf16")
    assert (out[0] == full[3]).all() and (out[3] == full[9]).all()


# -- gather_qmm -----------------------------------------------------------------

def test_gather_qmm_doctest_values():
    g = load_golden("gather_qmm_experts.txt")
    E, N, K, bits, gs = (int(g[k][0]) for k in ("experts", "N", "K", "bits", "group_size"))
    rhs = np.array(ints(g["rhs"]), dtype=np.uint32)
    packed = np.zeros((E, N, K * bits // 32), dtype=np.uint32)
    s = np.full((E, N, K // gs), 0x3F80, dtype=np.uint16)                  # scale 1.0
    b = np.stack([np.full((N, K // gs), int(np.float32(e + 1).view(np.uint32) >> 16),
                          dtype=np.uint16) for e in range(E)])             # bias e + 1
    x = np.full((len(rhs), 1, K), 0x3F80, dtype=np.uint16)                 # ones
    y, _ = oracle.gather_qmm(x, len(rhs), 1, packed, s, b, E, N, K, None, rhs, True, gs, bits)
    assert y.shape == (len(rhs), 1, N)
    assert list(y.reshape(-1)[:5]) == [float(v) for v in g["expect_first5"]]


@pytest.mark.parametrize("transpose", (True, False))
def test_gather_qmm_matches_numpy_gather_then_matmul(transpose):
    # Independent route: numpy's unpacker for dense weights, fancy indexing for
    # the gather, numpy matmul for the product.
    E, XB, M, N, K, bits, gs = 3, 4, 2, 32, 64, 5, 32
    rows, cols = (N, K) if transpose else (K, N)
    ws = [synth.quant_weight(900 + e, rows, cols, bits, gs) for e in range(E)]
    packed = np.stack([w.packed for w in ws]); s = np.stack([w.scales for w in ws])
    b = np.stack([w.biases for w in ws])
    x = synth.x_bf16(901, XB * M, K).reshape(XB, M, K)
    lhs = np.array([3, 0, 0, 2, 1], dtype=np.uint32)
    rhs = np.array([2, 2, 0, 1, 0], dtype=np.uint32)
    y, _ = oracle.gather_qmm(x, XB, M, packed, s, b, E, N, K, lhs, rhs, transpose, gs, bits)
    dense = np.stack([np_dense_f64(w) for w in ws])                        # [E, rows, cols]
    xf = bf16_f64(x)
    for i in range(len(lhs)):
        wd = dense[rhs[i]]
        want = xf[lhs[i]] @ (wd.T if transpose else wd)
        np.testing.assert_allclose(y[i], want, rtol=1e-12, atol=1e-12)


def test_gather_qmm_out_of_range_index_gives_zero_batch():
    E, N, K = 2, 4, 64
    w = synth.quant_weight(910, E * N, K, 4, 64)
    x = synth.x_bf16(911, 2, K).reshape(2, 1, K)
    y, a = oracle.gather_qmm(x, 2, 1, w.packed, w.scales, w.biases, E, N, K, None,
                             np.array([1, 7], dtype=np.uint32), True, 64, 4)
    assert (y[1] == 0).all() and (a[1] == 0).all() and (y[0] != 0).any()


# -- fused decode GEMVs ------------------------------------------------------------

def test_silu_gate_zero_gate_gives_resid_exactly():
    N, K, M = 16, 128, 2
    w = synth.quant_weight(920, N, K, 4, 64)
    gate = np.zeros((M, K), dtype=np.uint16)
    up = synth.x_bf16(921, M, K)
    resid = synth.x_bf16(922, M, N)
    y, a = oracle.silu_gate_qmm(gate, up, M, w.packed, w.scales, w.biases, N, K, 64, 4, resid)
    assert (y == bf16_f64(resid)).all() and (a == np.abs(bf16_f64(resid))).all()


@pytest.mark.parametrize("bits", (3, 4, 8))
def test_silu_gate_matches_scipy_expit_route(bits):
    # Independent route: scipy's logistic function for silu(g) = g * expit(g),
    # numpy's unpacker for the dense weight, numpy matmul.
    special = pytest.importorskip("scipy.special")
    N, K, M, gs = 24, 256, 3, 32
    w = synth.quant_weight(930 + bits, N, K, bits, gs)
    gate = synth.x_bf16(931, M, K)
    up = synth.x_bf16(932, M, K)
    resid = synth.x_bf16(933, M, N)
    y, _ = oracle.silu_gate_qmm(gate, up, M, w.packed, w.scales, w.biases, N, K, gs, bits, resid)
    g = bf16_f64(gate)
    x = g * special.expit(g) * bf16_f64(up)
    want = x @ np_dense_f64(w).T + bf16_f64(resid)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


# -- quantize -------------------------------------------------------------------

def _doctest_weight():
    # the module doctest's weight: w[r, c] = (64 r + c) / 64, [4, 64]
    rows, cols = 4, 64
    f = (np.arange(rows * cols, dtype=np.float32) / 64.0).reshape(rows, cols)
    return (f.view(np.uint32) >> 16).astype(np.uint16), rows, cols


def test_quantize_doctest_shapes():
    g = load_golden("pack_shape.txt")
    w, rows, cols = _doctest_weight()
    assert [rows, cols] == ints(g["weight_shape"])
    bits = int(g["bits"][0])
    packed, s, b = oracle.quantize(w, rows, cols, 64, bits)
    assert list(packed.shape) == ints(g["packed_shape"])
    assert s.shape == b.shape == (rows, 1)


@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("gs", (32, 128))
def test_quantize_codes_follow_the_stated_rule(bits, gs):
    # round((w - bias) / scale) clamped to [0, 2^bits - 1], with the oracle's
    # scales and biases, recomputed with numpy float32 and numpy's unpacker;
    # the bias is the group minimum, the group minimum gets code 0 and the
    # group maximum code 2^bits - 1.
    rows, cols = 6, 256
    w = synth.x_bf16(940 + bits, rows, cols)
    packed, s, b = oracle.quantize(w, rows, cols, gs, bits)
    wf = bf16_f64(w).astype(np.float32).reshape(rows, cols // gs, gs)
    sf = bf16_f64(s).astype(np.float32)[:, :, None]
    bf = bf16_f64(b).astype(np.float32)[:, :, None]
    assert (bf[:, :, 0] == wf.min(axis=2)).all()
    top = (1 << bits) - 1
    want = np.clip(np.rint((wf - bf) / sf), 0, top).astype(np.uint32).reshape(rows, cols)
    got = np_codes(packed, cols, bits)
    assert (got == want).all()
    g3 = got.reshape(rows, cols // gs, gs)
    assert (g3[wf == wf.min(axis=2, keepdims=True)] == 0).all()
    # The bf16 scale is within 2^-9 of (max - min) / top, so the maximum lands
    # within top * 2^-9 of top: exactly top below 8 bits, top or top - 1 at 8.
    slack = 1 if bits == 8 else 0
    assert (g3[wf == wf.max(axis=2, keepdims=True)] >= top - slack).all()


@pytest.mark.parametrize("bits", ALL_BITS)
def test_quantize_round_trip_within_half_a_step(bits):
    rows, cols, gs = 5, 128, 64
    w = synth.x_bf16(950 + bits, rows, cols)
    packed, s, b = oracle.quantize(w, rows, cols, gs, bits)
    back = oracle.dequantize(packed, s, b, rows, cols, gs, bits).astype(np.float64)
    step = np.repeat(bf16_f64(s), gs, axis=1)
    # half a step, plus the clamp at the top code: the bf16 scale's relative
    # error 2^-9 over the 2^bits - 1 steps of the range
    top = (1 << bits) - 1
    bound = 0.5 * step * (1 + 1e-3) + top * 2.0 ** -9 * step + 1e-6
    assert (np.abs(back - bf16_f64(w)) <= bound).all()


def test_quantize_constant_groups_are_exact():
    rows, cols, gs = 3, 64, 32
    vals = np.array([0.0, 1.0, -2.5], dtype=np.float32)
    w = np.repeat((vals.view(np.uint32) >> 16).astype(np.uint16)[:, None], cols, axis=1)
    packed, s, b = oracle.quantize(w, rows, cols, gs, 4)
    assert (s == 0).all() and (packed == 0).all()
    back = oracle.dequantize(packed, s, b, rows, cols, gs, 4)
    assert (back == vals[:, None]).all()


# -- other dtypes ----------------------------------------------------------------
# fp16 and fp32 scales, biases and x (nuvec_core quantized.rs: `quantize` keeps
# w's dtype for the scales and biases, `dequantize` returns the scales' dtype,
# `quantized_matmul` promotes x, scales and biases to one float type).

DTYPES = ("bf16", "f16", "f32")


def np_f64(a, dtype):
    """Values of a stored buffer via numpy's own conversions."""
    a = np.asarray(a)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return a.astype(np.uint16).view(np.float16).astype(np.float64)
    return bf16_f64(a)


def np_dense_typed_f64(w):
    c = np_codes(w.packed, w.cols, w.bits).astype(np.float64)
    s = np.repeat(np_f64(w.scales, w.sb_dtype), w.group_size, axis=1)
    b = np.repeat(np_f64(w.biases, w.sb_dtype), w.group_size, axis=1)
    return s * c + b


def np_f16_bits(f32):
    with np.errstate(over="ignore"):
        return np.asarray(f32, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_f16_to_f64_matches_numpy_every_pattern():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(p)) for p in pats])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), pats[~same][:8]
    # signs of zero
    assert np.signbit(oracle.f16_to_f64(0x8000)) and not np.signbit(oracle.f16_to_f64(0))


def test_f32_to_f16_matches_numpy():
    g = synth.rng(17)
    mags = 10.0 ** g.uniform(-9, 5.5, size=6000)
    vals = (mags * np.where(g.random(6000) < 0.5, -1.0, 1.0)).astype(np.float32)
    # midpoints between neighbouring fp16 values (ties), normal and subnormal,
    # both parities of the lower neighbour
    lo = np.arange(0, 0x7BFF, 37, dtype=np.uint32).astype(np.uint16)
    mid = ((lo.view(np.float16).astype(np.float64)
            + (lo + 1).view(np.float16).astype(np.float64)) / 2).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65519.0, 65519.996, 65520.0, 65536.0, 1e9,
                     2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -26,
                     6.1e-5, np.inf, -np.inf], dtype=np.float32)
    allv = np.concatenate([vals, mid, -mid, edge])
    got = np.array([oracle.f32_to_f16(float(v)) for v in allv], dtype=np.uint16)
    assert (got == np_f16_bits(allv)).all(), allv[got != np_f16_bits(allv)][:8]
    nan = oracle.f32_to_f16(float("nan"))
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0


def _golden_typed(sb):
    g = load_golden("lsb_first_plus_bias.txt")
    words = np.array(ints(g["words"]), dtype=np.uint32)[None, :]
    bits, cols, gs = int(g["bits"][0]), int(g["cols"][0]), int(g["group_size"][0])
    scale = float(bf16_f64(int(g["scale_bf16"][0], 0)))
    bias = float(bf16_f64(int(g["bias_bf16"][0], 0)))
    s = synth.as_dtype(np.full((1, cols // gs), scale), sb)
    b = synth.as_dtype(np.full((1, cols // gs), bias), sb)
    return words, s, b, cols, gs, bits, [float(v) for v in g["expect_f32"]]


def _is_correctly_rounded_f32(v32, exact):
    """v32 is the fp32 nearest to the exact rational value (ties to even)."""
    from fractions import Fraction
    v = Fraction(float(v32))
    up = Fraction(float(np.nextafter(np.float32(v32), np.float32(np.inf))))
    dn = Fraction(float(np.nextafter(np.float32(v32), np.float32(-np.inf))))
    d = abs(v - exact)
    if d > abs(up - exact) or d > abs(dn - exact):
        return False
    if d == abs(up - exact) or d == abs(dn - exact):  # a tie: the even one
        return (np.float32(v32).view(np.uint32) & 1) == 0
    return True


@pytest.mark.parametrize("sb", ("f16", "f32"))
def test_typed_dequant_pins(sb):
    from fractions import Fraction
    # the printed example: codes 0..7 with scale 2, bias -1 -> 2c - 1
    words, s, b, cols, gs, bits, expected = _golden_typed(sb)
    out = oracle.dequantize(words, s, b, 1, cols, gs, bits, "f32", sb_dtype=sb)
    assert out.ravel().astype(np.float64).tolist() == expected
    # zero codes give the bias exactly
    w = synth.quant_weight_typed(71, 6, 128, 4, 32, sb)
    w.packed[:] = 0
    out = oracle.dequantize(w.packed, w.scales, w.biases, 6, 128, 32, 4, "f32", sb_dtype=sb)
    assert (out.astype(np.float64) == np.repeat(np_f64(w.biases, sb), 32, axis=1)).all()
    # every element is s*c + b rounded once to fp32 (exact rational arithmetic)
    for bits in (3, 4, 8):
        w = synth.quant_weight_typed(72 + bits, 3, 64, bits, 32, sb)
        out = oracle.dequantize(w.packed, w.scales, w.biases, 3, 64, 32, bits, "f32",
                                sb_dtype=sb)
        codes = np_codes(w.packed, 64, bits)
        s = np_f64(w.scales, sb)
        b = np_f64(w.biases, sb)
        for r in range(3):
            for j in range(64):
                exact = Fraction(s[r, j // 32]) * int(codes[r, j]) + Fraction(b[r, j // 32])
                assert _is_correctly_rounded_f32(out[r, j], exact), (bits, r, j)


@pytest.mark.parametrize("sb", DTYPES)
def test_typed_dequant_f16_out_is_rne_of_f32(sb):
    w = synth.quant_weight_typed(81, 9, 512, 5, 64, sb)
    f = oracle.dequantize(w.packed, w.scales, w.biases, 9, 512, 64, 5, "f32", sb_dtype=sb)
    h = oracle.dequantize(w.packed, w.scales, w.biases, 9, 512, 64, 5, "f16", sb_dtype=sb)
    assert (h == np_f16_bits(f)).all()
    bb = oracle.dequantize(w.packed, w.scales, w.biases, 9, 512, 64, 5, "bf16", sb_dtype=sb)
    assert (bb == torch_bf16_bits(f)).all()
    # and the fp32 value is the exact fp64 one rounded once (16-bit scales:
    # s*c + b is exact in fp64)
    if sb != "f32":
        assert (f == np_dense_typed_f64(w).astype(np.float32)).all()


def test_typed_rows_is_a_gather_of_typed_dequantize():
    w = synth.quant_weight_typed(91, 40, 128, 6, 32, "f16")
    full = oracle.dequantize(w.packed, w.scales, w.biases, 40, 128, 32, 6, "f16", sb_dtype="f16")
    idx = synth.indices(92, 17, 40)
    got, bad = oracle.rows(w.packed, w.scales, w.biases, 40, 128, idx, 32, 6, "f16",
                           sb_dtype="f16")
    assert bad == 0 and (got == full[idx]).all()


@pytest.mark.parametrize("x_dtype,sb_dtype,transpose", [
    ("f16", "f16", True), ("f16", "f16", False), ("f32", "f32", True), ("f32", "bf16", False),
    ("bf16", "f16", True), ("f16", "f32", False)])
def test_typed_qmm_brute_force_tiny(x_dtype, sb_dtype, transpose):
    M, K, bits, gs = 3, 64, 5, 32
    N = 8 if transpose else 32
    x = synth.x_typed(310, M, K, x_dtype)
    if transpose:
        w = synth.quant_weight_typed(410, N, K, bits, gs, sb_dtype)
        dense_kn = np_dense_typed_f64(w).T
    else:
        w = synth.quant_weight_typed(510, K, N, bits, gs, sb_dtype)
        dense_kn = np_dense_typed_f64(w)
    y, a = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits,
                      x_dtype=x_dtype, sb_dtype=sb_dtype)
    xf = np_f64(x, x_dtype)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += xf[m, k] * dense_kn[k, n]
            want[m, n] = acc
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf) @ np.abs(dense_kn), rtol=1e-12, atol=1e-12)
    ms, ns = np.array([0, 2, 1], np.int64), np.array([N - 1, 0, 3], np.int64)
    ys, _ = oracle.qmm_sampled(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits,
                               ms, ns, x_dtype=x_dtype, sb_dtype=sb_dtype)
    assert (ys == y[ms, ns]).all()


def _holds(values, t):
    """Whether every (finite) value is exactly a value of type t."""
    v = np.asarray(values, dtype=np.float64)
    v = v[np.isfinite(v)]
    if t == "f32":
        return bool((v.astype(np.float32).astype(np.float64) == v).all())
    if t == "f16":
        with np.errstate(over="ignore"):
            return bool((v.astype(np.float16).astype(np.float64) == v).all())
    f = v.astype(np.float32)
    return bool(((f.astype(np.float64) == v) & ((f.view(np.uint32) & 0xFFFF) == 0)).all())


def test_promote_types_holds_both_exactly_and_is_narrowest():
    every = {"bf16": bf16_f64(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)),
             "f16": np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
             .astype(np.float64),
             # fp32 values no 16-bit type holds (fraction and exponent range)
             "f32": np.array([1.0 + 2.0 ** -23, 2.0 ** -140, 3.0e38, 1.0], np.float32)
             .astype(np.float64)}
    width = {"bf16": 16, "f16": 16, "f32": 32}
    for a in DTYPES:
        for b in DTYPES:
            t = oracle.promote_types(a, b)
            assert t == oracle.promote_types(b, a)
            both = np.concatenate([every[a], every[b]])
            assert _holds(both, t), (a, b, t)
            narrower = [u for u in DTYPES if width[u] < width[t]]
            assert not any(_holds(both, u) for u in narrower), (a, b, t)
    assert oracle.promote_types("bf16", "f16") == "f32"


@pytest.mark.parametrize("w_dtype", ("f16", "f32"))
@pytest.mark.parametrize("bits", (2, 4, 8))
def test_typed_quantize_codes_follow_the_stated_rule(w_dtype, bits):
    rows, cols, gs = 6, 256, 64
    w = synth.x_typed(960 + bits, rows, cols, w_dtype)
    packed, s, b = oracle.quantize(w, rows, cols, gs, bits, w_dtype=w_dtype)
    assert s.dtype == b.dtype == np.asarray(w).dtype
    wf = np_f64(w, w_dtype).astype(np.float32).reshape(rows, cols // gs, gs)
    sf = np_f64(s, w_dtype).astype(np.float32)[:, :, None]
    bf = np_f64(b, w_dtype).astype(np.float32)[:, :, None]
    assert (bf[:, :, 0] == wf.min(axis=2)).all()
    top = (1 << bits) - 1
    # the stored scale is (max - min) / top in fp32, then in w's dtype
    sc = (wf.max(axis=2) - wf.min(axis=2)) / np.float32(top)
    want_s = sc if w_dtype == "f32" else sc.astype(np.float16).astype(np.float32)
    assert (sf[:, :, 0] == want_s).all()
    want = np.clip(np.rint((wf - bf) / sf), 0, top).astype(np.uint32).reshape(rows, cols)
    assert (np_codes(packed, cols, bits) == want).all()
    back = oracle.dequantize(packed, s, b, rows, cols, gs, bits, sb_dtype=w_dtype)
    step = np.repeat(sf[:, :, 0].astype(np.float64), gs, axis=1)
    rel = 2.0 ** -11 if w_dtype == "f16" else 2.0 ** -23
    bound = 0.5 * step * (1 + 1e-3) + top * rel * step + 1e-6
    assert (np.abs(back.astype(np.float64) - np_f64(w, w_dtype)) <= bound).all()
