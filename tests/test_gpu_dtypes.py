"""Other dtypes on the GPU against the oracle: fp16 and fp32 scales and biases,
fp16 and fp32 x and outputs, and MLX's promotion of x, scales and biases to one
type (nuvec_core quantized.rs: `quantize` keeps w's dtype for the scales and
biases, `dequantize` returns the scales' dtype, `quantized_matmul` promotes).

dequantize, rows and quantize are compared bit for bit.  Matmuls must meet
the stated tolerance, 8e-3 * sum_k |x w| + 1e-6, and tighter bounds that
follow from the type they compute in:
  fp32: fp32 weights (2^-24 relative) and fp32 sums over K terms plus at most
        64 split partials: (K + 66) * 2^-24 * sum_k |x w| (the recursive
        summation bound);
  fp16: weights rounded once to fp16 (2^-11 relative), exact fp16 products,
        fp32 sums: 2e-3 * sum_k |x w|, and 3e-3 when y itself is fp16.
One-hot rows of x pin every weight inside the matmul exactly: y[m, n] is the
kernel's own dequantized weight."""
import numpy as np
import pytest

import oracle
from mlx_grouped_affine_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from gpu_util import TOL_ABS, TOL_REL, dev  # noqa: E402

ALL_BITS = (1, 2, 3, 4, 5, 6, 8)
Q = {"f32": qmm.QMM_F32, "bf16": qmm.QMM_BF16, "f16": qmm.QMM_F16}


def out_tensor(shape, dtype):
    return torch.empty(shape, dtype=torch.float32 if dtype == "f32" else torch.int16,
                       device="cuda")


def host(t, dtype):
    """Stored bits (uint32 for fp32, uint16 otherwise)."""
    a = t.cpu().numpy()
    return a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)


def host_f64(t, dtype):
    a = t.cpu().numpy()
    if dtype == "f32":
        return a.astype(np.float64)
    u = a.view(np.uint16)
    if dtype == "f16":
        return u.view(np.float16).astype(np.float64)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bits_of(a, dtype):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)


def first_diff(got, want):
    bad = got != want
    return "%d of %d differ, first at %s" % (bad.sum(), bad.size, tuple(np.argwhere(bad)[0]))


# -- dequantize and rows ---------------------------------------------------------

@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("sb", ("f16", "f32"))
@pytest.mark.parametrize("out", ("f32", "same"))
def test_dequantize_typed_bit_exact(bits, sb, out):
    out = sb if out == "same" else out
    rows, cols, gs = 45, 384, 64 if bits % 2 else 32
    w = synth.quant_weight_typed(600 + bits, rows, cols, bits, gs, sb)
    o = out_tensor((rows, cols), out)
    qmm.qmm_dequantize_typed(dev(w.packed), dev(w.scales), dev(w.biases), Q[sb], rows, cols, gs,
                             bits, o, Q[out])
    torch.cuda.synchronize()
    want = oracle.dequantize(w.packed, w.scales, w.biases, rows, cols, gs, bits, out,
                             sb_dtype=sb)
    got, ref = host(o, out), bits_of(want, out)
    assert (got == ref).all(), first_diff(got, ref)


@pytest.mark.parametrize("sb", ("f16", "f32"))
def test_rows_typed_bit_exact_with_a_bad_index(sb):
    T, cols, gs, bits = 300, 256, 64, 4
    w = synth.quant_weight_typed(610, T, cols, bits, gs, sb)
    idx = synth.indices(611, 77, T)
    idx[5] = T + 3                       # outside the table: a zero row and the index bit
    o = out_tensor((idx.size, cols), sb)
    qmm.qmm_rows_typed(dev(w.packed), dev(w.scales), dev(w.biases), Q[sb], T, cols,
                       dev(idx.view(np.int32)), idx.size, gs, bits, o, Q[sb])
    assert qmm.qmm_get_device_error() == qmm.QMM_ERR_INDEX
    want, bad = oracle.rows(w.packed, w.scales, w.biases, T, cols, idx, gs, bits, sb, sb_dtype=sb)
    assert bad == 1
    got, ref = host(o, sb), bits_of(want, sb)
    assert (got == ref).all(), first_diff(got, ref)


def test_dequantize_typed_rejects_cross_type_output():
    w = synth.quant_weight_typed(612, 4, 64, 4, 32, "f16")
    o = out_tensor((4, 64), "bf16")
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_dequantize_typed(dev(w.packed), dev(w.scales), dev(w.biases), qmm.QMM_F16, 4, 64,
                                 32, 4, o, qmm.QMM_BF16)
    assert e.value.status == qmm.QMM_ERR_UNSUPPORTED


# -- quantize --------------------------------------------------------------------

@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("wt", ("f16", "f32", "bf16"))
def test_quantize_typed_bit_exact(bits, wt):
    rows, cols, gs = 29, 384, (32, 64, 128)[bits % 3]
    w = synth.x_typed(620 + bits, rows, cols, wt)
    w[3, :gs] = w[3, 0]                  # a constant group: scale 0, codes 0
    packed = torch.empty((rows, cols * bits // 32), dtype=torch.int32, device="cuda")
    s = out_tensor((rows, cols // gs), wt)
    b = out_tensor((rows, cols // gs), wt)
    qmm.qmm_quantize_typed(dev(w), Q[wt], rows, cols, gs, bits, packed, s, b)
    torch.cuda.synchronize()
    wp, ws, wb = oracle.quantize(w, rows, cols, gs, bits, w_dtype=wt)
    assert (packed.cpu().numpy().view(np.uint32) == wp).all(), first_diff(
        packed.cpu().numpy().view(np.uint32), wp)
    assert (host(s, wt) == bits_of(ws, wt)).all(), first_diff(host(s, wt), bits_of(ws, wt))
    assert (host(b, wt) == bits_of(wb, wt)).all(), first_diff(host(b, wt), bits_of(wb, wt))


# -- quantized_matmul ------------------------------------------------------------

def promoted(x_dt, sb_dt):
    return oracle.promote_types(x_dt, sb_dt)


def run_mm(x, x_dt, M, w, N, K, transpose, y_dt):
    y = out_tensor((M, N), y_dt)
    qmm.qmm_quantized_matmul_typed(dev(x), Q[x_dt], M, dev(w.packed), dev(w.scales),
                                   dev(w.biases), Q[w.sb_dtype], N, K, transpose, w.group_size,
                                   w.bits, y, Q[y_dt])
    torch.cuda.synchronize()
    return host_f64(y, y_dt)


def check_mm(got, ref, absy, d, y_dt, K, what):
    err = np.abs(got - ref)
    stated = TOL_REL * absy + TOL_ABS
    if d == "f32":
        tight = (K + 66) * 2.0 ** -24 * absy + TOL_ABS
    elif d == "f16":
        tight = (3e-3 if y_dt == "f16" else 2e-3) * absy + TOL_ABS
    else:
        tight = stated
    for name, bound in (("stated", stated), ("dtype", tight)):
        bad = err > bound
        if bad.any():
            i = tuple(np.argwhere(bad)[0])
            raise AssertionError("%s: %d outputs beyond the %s bound; first %s: y=%r ref=%r "
                                 "bound=%r" % (what, bad.sum(), name, i, got[i], ref[i], bound[i]))


COMBOS = (("f16", "f16"), ("f32", "f32"), ("bf16", "f16"), ("f16", "f32"), ("bf16", "f32"),
          ("f32", "bf16"), ("f32", "f16"))


@pytest.mark.parametrize("x_dt,sb_dt", COMBOS)
@pytest.mark.parametrize("M", (1, 5, 16, 40, 300))
@pytest.mark.parametrize("transpose", (True, False))
def test_matmul_typed_against_oracle(x_dt, sb_dt, M, transpose):
    bits = (3, 4, 8)[M % 3]
    gs = 64
    N, K = (200, 512) if transpose else (256, 333)   # ragged N tile / odd K
    w = synth.quant_weight_typed(700 + M + bits, N if transpose else K, K if transpose else N,
                                 bits, gs, sb_dt)
    x = synth.x_typed(710 + M, M, K, x_dt)
    d = promoted(x_dt, sb_dt)
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits,
                           x_dtype=x_dt, sb_dtype=sb_dt)
    for y_dt in sorted({"f32", d}):
        got = run_mm(x, x_dt, M, w, N, K, transpose, y_dt)
        check_mm(got, ref, absy, d, y_dt, K, "%s x %s M=%d T=%s y=%s" % (x_dt, sb_dt, M, transpose, y_dt))


@pytest.mark.parametrize("sb_dt,x_dt", (("f16", "f16"), ("f32", "f32"), ("f16", "bf16")))
@pytest.mark.parametrize("bits", ALL_BITS)
@pytest.mark.parametrize("M,transpose", ((1, True), (16, True), (40, True), (16, False),
                                         (40, False)))
def test_matmul_typed_weights_are_exact(sb_dt, x_dt, bits, M, transpose):
    """One-hot x rows: y[m, n] = the weight w[k_m, n] the kernel used, which
    must be the dequantized weight rounded to the compute type: fp16
    RN(s*c + b) (once, or via fp32) for fp16, fp32 fma(s, c, b) for fp32."""
    rows, cols, gs = (200, 1024, 32) if transpose else (1024, 256, 32)
    w = synth.quant_weight_typed(800 + bits + M, rows, cols, bits, gs, sb_dt)
    N, K = (rows, cols) if transpose else (cols, rows)
    ks = np.random.default_rng(M + bits).choice(K, size=M, replace=False)
    x = np.zeros((M, K), dtype=np.float32)
    x[np.arange(M), ks] = 1.0
    x = synth.as_dtype(x, x_dt)
    got = run_mm(x, x_dt, M, w, N, K, transpose, "f32")
    d = promoted(x_dt, sb_dt)
    f32 = oracle.dequantize(w.packed, w.scales, w.biases, rows, cols, gs, bits, "f32",
                            sb_dtype=sb_dt).astype(np.float64)
    if d == "f16":
        via = oracle.dequantize(w.packed, w.scales, w.biases, rows, cols, gs, bits, "f16",
                                sb_dtype=sb_dt).view(np.float16).astype(np.float64)
        codes = oracle.unpack(w.packed, cols, bits).astype(np.float64)
        rep = np.repeat(np.arange(cols // gs), gs)
        s = synth_vals(w.scales, sb_dt)[:, rep]
        b = synth_vals(w.biases, sb_dt)[:, rep]
        once = (s * codes + b).astype(np.float16).astype(np.float64)
        accept = (via, once)
    else:
        accept = (f32,)
    ok = np.zeros(got.shape, dtype=bool)
    for a in accept:
        want = a[:, ks].T if transpose else a[ks, :]
        ok |= got == want
    if not ok.all():
        m, n = np.argwhere(~ok)[0]
        raise AssertionError("%d of %d weights differ; first (m=%d, n=%d): got %r" % (
            (~ok).sum(), ok.size, m, n, got[m, n]))


def synth_vals(a, dtype):
    a = np.asarray(a)
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("x_dt,sb_dt,M", (("f16", "f16", 1), ("f16", "f16", 16),
                                          ("f16", "f16", 2048), ("f32", "f32", 1),
                                          ("f32", "f32", 300)))
def test_matmul_typed_full_size_sampled(x_dt, sb_dt, M):
    """The benchmark's layers: W [14336, 4096] at 4 bits, group 64 (decode
    rows at [4096, 4096]); sampled outputs against the oracle."""
    N, K = (4096, 4096) if M <= 16 else (14336, 4096)
    w = synth.quant_weight_typed(900 + M, N, K, 4, 64, sb_dt)
    x = synth.x_typed(901 + M, M, K, x_dt)
    d = promoted(x_dt, sb_dt)
    got = run_mm(x, x_dt, M, w, N, K, True, d)
    g = np.random.default_rng(902)
    ms = g.integers(0, M, size=300).astype(np.int64)
    ns = g.integers(0, N, size=300).astype(np.int64)
    ms[:2], ns[:2] = (0, M - 1), (0, N - 1)
    ref, absy = oracle.qmm_sampled(x, M, w.packed, w.scales, w.biases, N, K, True, 64, 4, ms, ns,
                                   x_dtype=x_dt, sb_dtype=sb_dt)
    check_mm(got[ms, ns], ref, absy, d, d, K, "full %s x %s M=%d" % (x_dt, sb_dt, M))


@pytest.mark.parametrize("M,transpose", ((1, True), (16, True), (3, False), (200, True)))
def test_matmul_f32_split_k_repeats_bit_for_bit_and_long_k(M, transpose):
    """K = 14336 splits the fp32 path's K range over many blocks (28 slices of
    512 at M <= 16); the slices are added in a fixed order, so two calls give
    the same bits, and the result meets the fp32 bound for that K."""
    N, K, gs, bits = 256, 14336, 128, 4
    w = synth.quant_weight_typed(950 + M, N if transpose else K, K if transpose else N, bits, gs,
                                 "f32")
    x = synth.x_typed(951 + M, M, K, "f32")
    a = run_mm(x, "f32", M, w, N, K, transpose, "f32")
    b = run_mm(x, "f32", M, w, N, K, transpose, "f32")
    assert (a.view(np.uint64) == b.view(np.uint64)).all()
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, transpose, gs, bits,
                           x_dtype="f32", sb_dtype="f32")
    check_mm(a, ref, absy, "f32", "f32", K, "f32 long K M=%d T=%s" % (M, transpose))


@pytest.mark.parametrize("x_dt,sb_dt", (("f16", "f16"), ("f32", "f32"), ("bf16", "f16")))
@pytest.mark.parametrize("M", (1, 5, 16, 24))
def test_matmul_typed_k_not_a_multiple_of_128(x_dt, sb_dt, M):
    """W stored [N, K] with K = 320 (a multiple of the group, not of 128): the
    decode kernels' plain-load form (no TMA boxes) in fp16, the fp32 GEMV form,
    and the tensor-core GEMM at M = 24."""
    N, K, gs, bits = 136, 320, 32, 5
    w = synth.quant_weight_typed(990 + M, N, K, bits, gs, sb_dt)
    x = synth.x_typed(991 + M, M, K, x_dt)
    d = promoted(x_dt, sb_dt)
    ref, absy = oracle.qmm(x, M, w.packed, w.scales, w.biases, N, K, True, gs, bits,
                           x_dtype=x_dt, sb_dtype=sb_dt)
    for y_dt in sorted({"f32", d}):
        got = run_mm(x, x_dt, M, w, N, K, True, y_dt)
        check_mm(got, ref, absy, d, y_dt, K, "K=320 %s x %s M=%d y=%s" % (x_dt, sb_dt, M, y_dt))
