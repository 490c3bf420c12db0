"""Boundary queries that need the device: conv_fwd_workspace_size (through
the C ABI) equals conv_fwd_plan's workspace_bytes on every workload shape,
and a buffer of that size runs the plan the query describes."""
import ctypes

import pytest
import torch

import conv_workloads as cw

pytestmark = pytest.mark.gpu

I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _ndhwc(wl):
    if wl.x_layout == "ncdhw":
        n, c, d, h, w = wl.x_shape
        return (n, d, h, w, c)
    return tuple(wl.x_shape)


def _ktrsc(wl):
    if wl.w_layout == "kctrs":
        k, c, t, r, s = wl.w_shape
        return (k, t, r, s, c)
    return tuple(wl.w_shape)


@pytest.mark.parametrize("name", [w.name for w in cw.WORKLOADS + cw.PATCH_WORKLOADS])
def test_workspace_size_equals_plan(pkg, name):
    wl = cw.BY_NAME[name]
    xs, ws = _ndhwc(wl), _ktrsc(wl)
    dtype = 1 if wl.dtype == "fp8" else 0
    lib = ctypes.CDLL(pkg.LIB_PATH)
    lib.conv_fwd_workspace_size.restype = ctypes.c_size_t
    n = lib.conv_fwd_workspace_size(I5(*xs), I5(*ws), I3(*wl.stride), I3(*wl.pad),
                                    I3(*wl.dil), dtype)
    assert n == pkg.conv_fwd_plan(xs, ws, wl.stride, wl.pad, wl.dil, dtype)["workspace_bytes"]
    assert n == pkg.conv_fwd_workspace_size(xs, ws, wl.stride, wl.pad, wl.dil, dtype)


def test_workspace_size_of_an_unsupported_problem_is_zero(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    lib.conv_fwd_workspace_size.restype = ctypes.c_size_t
    lib.conv_last_error.restype = ctypes.c_char_p
    # C * 2 bytes = 6: neither the implicit classes nor a GEMM class read it
    n = lib.conv_fwd_workspace_size(I5(1, 4, 8, 8, 3), I5(8, 3, 3, 3, 3), I3(1, 1, 1),
                                    I3(1, 1, 1), I3(1, 1, 1), 0)
    assert n == 0 and lib.conv_last_error() != b""
