"""Host-side tests of the C ABI (no GPU): the library loads, exports every entry
point include/qmm.h declares, and rejects every invalid argument before it
launches anything (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

from mlx_grouped_affine_gb300 import qmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 1 << 20          # a 16-byte aligned fake device address
S = 0                # NULL stream


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = qmm.lib()
    names = declared_functions()
    assert set(names) == set(qmm.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


def test_last_error_starts_empty_per_thread():
    import threading
    seen = []
    t = threading.Thread(target=lambda: seen.append(qmm.qmm_last_error()))
    t.start()
    t.join()
    assert seen == [""]


def deq(**kw):
    args = dict(w=A, s=A, b=A, rows=4, cols=64, G=32, bits=4, out=A, dt=qmm.QMM_F32)
    args.update(kw)
    return qmm.lib().qmm_dequantize(args["w"], args["s"], args["b"], args["rows"], args["cols"],
                                    args["G"], args["bits"], args["out"], args["dt"], S)


def mm(**kw):
    args = dict(x=A, M=1, w=A, s=A, b=A, N=64, K=64, tr=1, G=32, bits=4, y=A, dt=qmm.QMM_BF16)
    args.update(kw)
    return qmm.lib().qmm_quantized_matmul(args["x"], args["M"], args["w"], args["s"], args["b"],
                                          args["N"], args["K"], args["tr"], args["G"],
                                          args["bits"], args["y"], args["dt"], S)


def rows(**kw):
    args = dict(w=A, s=A, b=A, T=10, cols=64, idx=A, n=3, G=64, bits=4, out=A, dt=qmm.QMM_BF16)
    args.update(kw)
    return qmm.lib().qmm_rows(args["w"], args["s"], args["b"], args["T"], args["cols"],
                              args["idx"], args["n"], args["G"], args["bits"], args["out"],
                              args["dt"], S)


BAD = qmm.QMM_ERR_INVALID_ARG


@pytest.mark.parametrize("G", [0, 16, 48, 96, 256, -64])
def test_group_size_rule(G):
    assert deq(G=G) == BAD and mm(G=G) == BAD and rows(G=G) == BAD
    assert "group size" in qmm.qmm_last_error()


@pytest.mark.parametrize("bits", [0, 7, 9, 16, -4])
def test_bits_rule(bits):
    assert deq(bits=bits) == BAD and mm(bits=bits) == BAD and rows(bits=bits) == BAD
    assert "bits" in qmm.qmm_last_error()


def test_grouped_axis_must_divide():
    assert deq(cols=96, G=64) == BAD
    assert deq(cols=0) == BAD
    assert mm(K=96, G=64) == BAD               # transposed: K is grouped
    assert mm(tr=0, N=96, G=64) == BAD          # not transposed: N is grouped
    assert rows(cols=100) == BAD


def test_shape_signs():
    assert deq(rows=-1) == BAD
    assert mm(M=-1) == BAD and mm(N=-1) == BAD and mm(K=0) == BAD
    assert rows(n=-2) == BAD and rows(T=-1) == BAD


def test_transpose_flag():
    assert mm(tr=2) == BAD and mm(tr=-1) == BAD


def test_null_and_misaligned_pointers():
    assert deq(w=0) == BAD and deq(s=0) == BAD and deq(b=0) == BAD and deq(out=0) == BAD
    assert deq(w=A + 4) == BAD and deq(out=A + 8) == BAD and deq(s=A + 2) == BAD
    assert mm(x=0) == BAD and mm(y=0) == BAD and mm(x=A + 2) == BAD and mm(w=A + 4) == BAD
    assert rows(idx=0) == BAD and rows(idx=A + 4) == BAD and rows(out=0) == BAD
    assert "aligned" in qmm.qmm_last_error() or "null" in qmm.qmm_last_error()


def test_unsupported_output_dtype():
    assert deq(dt=2) == qmm.QMM_ERR_UNSUPPORTED
    assert mm(dt=7) == qmm.QMM_ERR_UNSUPPORTED
    assert rows(dt=-1) == qmm.QMM_ERR_UNSUPPORTED
    assert "dtype" in qmm.qmm_last_error()


def test_empty_outputs_are_no_ops():
    # No launch happens, so these succeed even without a GPU.
    assert deq(rows=0, out=0) == qmm.QMM_OK
    assert mm(M=0, x=0, y=0) == qmm.QMM_OK
    assert mm(N=0, x=0, y=0) == qmm.QMM_OK
    assert rows(n=0, idx=0, out=0) == qmm.QMM_OK


def test_python_binding_raises():
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_dequantize(A, A, A, 4, 64, 33, 4, A, qmm.QMM_F32, stream=0)
    assert e.value.status == qmm.QMM_ERR_INVALID_ARG


def test_launch_flags_are_per_thread_and_checked():
    import threading
    assert qmm.qmm_set_launch_flags(qmm.QMM_LAUNCH_PDL) == 0
    seen = []
    t = threading.Thread(target=lambda: seen.append(qmm.qmm_set_launch_flags(0)))
    t.start()
    t.join()
    assert seen == [0]                                   # other thread starts at 0
    assert qmm.qmm_set_launch_flags(0x10 | qmm.QMM_LAUNCH_PDL) == qmm.QMM_LAUNCH_PDL
    assert "unknown flag" in qmm.qmm_last_error()
    assert qmm.qmm_set_launch_flags(0) == qmm.QMM_LAUNCH_PDL   # the unknown bit was dropped


def test_wait_limit_is_per_thread_and_restorable():
    import threading
    assert qmm.qmm_set_wait_limit(5) == 0                # 0: the default until set
    seen = []
    t = threading.Thread(target=lambda: seen.append(qmm.qmm_set_wait_limit(7)))
    t.start()
    t.join()
    assert seen == [0]                                   # other thread has its own
    assert qmm.qmm_set_wait_limit(0) == 5
    assert qmm.qmm_set_wait_limit(0) == 0


# -- typed calls (dtypes) ----------------------------------------------------------

def test_promote_types_matches_the_oracle():
    import oracle
    names = {"f32": qmm.QMM_F32, "bf16": qmm.QMM_BF16, "f16": qmm.QMM_F16}
    for a, qa in names.items():
        for b, qb in names.items():
            assert qmm.qmm_promote_types(qa, qb) == names[oracle.promote_types(a, b)], (a, b)
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_promote_types(qmm.QMM_F16, 9)
    assert e.value.status == qmm.QMM_ERR_UNSUPPORTED


def mm_typed(**kw):
    args = dict(x=A, xt=qmm.QMM_F16, M=1, w=A, s=A, b=A, st=qmm.QMM_F16, N=64, K=64, tr=1, G=32,
                bits=4, y=A, dt=qmm.QMM_F16)
    args.update(kw)
    return qmm.lib().qmm_quantized_matmul_typed(
        args["x"], args["xt"], args["M"], args["w"], args["s"], args["b"], args["st"], args["N"],
        args["K"], args["tr"], args["G"], args["bits"], args["y"], args["dt"], S)


def test_typed_calls_check_dtypes_before_launching():
    U = qmm.QMM_ERR_UNSUPPORTED
    L = qmm.lib()
    # output: fp32 or the computed (promoted) type only
    assert mm_typed(dt=qmm.QMM_BF16) == U
    assert mm_typed(xt=qmm.QMM_BF16, dt=qmm.QMM_F16) == U          # bf16 x f16 -> f32
    assert mm_typed(xt=qmm.QMM_BF16, dt=qmm.QMM_BF16) == U
    assert mm_typed(xt=5) == U and mm_typed(st=-1) == U
    assert "dtype" in qmm.qmm_last_error()
    assert mm_typed(M=0, x=0, y=0) == qmm.QMM_OK
    assert mm_typed(xt=qmm.QMM_BF16, dt=qmm.QMM_F32, M=0, x=0, y=0) == qmm.QMM_OK
    assert mm_typed(x=A + 2) == BAD and mm_typed(G=48) == BAD
    assert L.qmm_dequantize_typed(A, A, A, qmm.QMM_F16, 4, 64, 32, 4, A, qmm.QMM_BF16, S) == U
    assert L.qmm_dequantize_typed(A, A, A, 3, 4, 64, 32, 4, A, qmm.QMM_F32, S) == U
    assert L.qmm_dequantize_typed(A, A, A, qmm.QMM_F32, 0, 64, 32, 4, 0, qmm.QMM_F32, S) == qmm.QMM_OK
    assert L.qmm_rows_typed(A, A, A, qmm.QMM_F16, 10, 64, A, 3, 64, 4, A, qmm.QMM_BF16, S) == U
    assert L.qmm_rows_typed(A, A, A, qmm.QMM_F16, 10, 64, A, 0, 64, 4, A, qmm.QMM_F16, S) == qmm.QMM_OK
    assert L.qmm_quantize_typed(A, 7, 4, 64, 32, 4, A, A, A, S) == U
    assert L.qmm_quantize_typed(A, qmm.QMM_F32, 0, 64, 32, 4, A, A, A, S) == qmm.QMM_OK
    assert L.qmm_quantize_typed(A, qmm.QMM_F32, 4, 48, 32, 4, A, A, A, S) == BAD


def test_rows_checks_its_index_count_before_its_pointer():
    assert rows(n=-3, idx=0) == BAD and "negative index count" in qmm.qmm_last_error()
    assert rows(n=-3) == BAD
    L = qmm.lib()
    assert L.qmm_rows_typed(A, A, A, qmm.QMM_F16, 10, 64, 0, -1, 64, 4, A, qmm.QMM_F16, S) == BAD
    assert "negative index count" in qmm.qmm_last_error()


def test_each_entry_point_names_itself_in_its_errors():
    L = qmm.lib()
    assert deq(G=48) == BAD and qmm.qmm_last_error().startswith("qmm_dequantize:")
    assert mm(G=48) == BAD and qmm.qmm_last_error().startswith("qmm_quantized_matmul:")
    assert rows(G=48) == BAD and qmm.qmm_last_error().startswith("qmm_rows:")
    assert L.qmm_quantized_matmul_noalloc(A, 1, A, A, A, 64, 64, 1, 48, 4, A, qmm.QMM_BF16, S) == BAD
    assert qmm.qmm_last_error().startswith("qmm_quantized_matmul_noalloc:")
    assert mm_typed(G=48) == BAD and qmm.qmm_last_error().startswith("qmm_quantized_matmul_typed:")
    assert L.qmm_quantize(A, 4, 64, 48, 4, A, A, A, S) == BAD
    assert qmm.qmm_last_error().startswith("qmm_quantize:")
