"""Marshalling helpers for the GPU tests: host numpy arrays to device tensors and
back, and the matmul tolerance check.  No arithmetic of the method here."""
import numpy as np
import torch

from mlx_grouped_affine_gb300 import qmm

TOL_REL = 8e-3
TOL_ABS = 1e-6


def dev(a):
    """A device tensor holding the same bytes as the numpy array."""
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint32): np.int32, np.dtype(np.uint16): np.int16}.get(a.dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a).cuda()


def weight(w):
    return dev(w.packed), dev(w.scales), dev(w.biases)


def empty_out(shape, out_dtype):
    dt = torch.float32 if out_dtype == qmm.QMM_F32 else torch.int16
    return torch.empty(shape, dtype=dt, device="cuda")


def host_bits(t):
    """Raw bits of a device output: uint32 for fp32, uint16 for bf16."""
    a = t.cpu().numpy()
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def host_f64(t):
    a = t.cpu().numpy()
    if a.dtype == np.float32:
        return a.astype(np.float64)
    return (a.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def oracle_bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_within_tolerance(y_dev, y_ref, absy, what=""):
    """|y - y_ref| <= 8e-3 * sum_k |x w| + 1e-6 for every output, after the
    output's own rounding."""
    y = host_f64(y_dev).reshape(y_ref.shape)
    err = np.abs(y - y_ref)
    bound = TOL_REL * absy + TOL_ABS
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d outputs out of tolerance; first at %s: y=%r ref=%r "
                             "bound=%r" % (what, bad.sum(), bad.size, tuple(i), y[tuple(i)],
                                           y_ref[tuple(i)], bound[tuple(i)]))
    return float((err / bound).max()) if err.size else 0.0
