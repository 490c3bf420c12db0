"""conv_fwd_noalloc: the entry point for callers that cannot allocate device
memory (for example engines that reserve all device memory up front, or
latency-bound code that cannot afford cudaMalloc's implicit synchronisation).
It keeps split-K partials in the library's static device scratch instead of a
caller workspace.  Called here through the C ABI (ctypes), on a problem whose
plan uses split-K, and compared with conv_fwd on the same inputs, two calls in
a row (the scratch keeps the previous call's contents, which must not leak
into the next result).  This file is collected last so that a run stopping
at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import conv_workloads as cw
from _gpu_util import as_f64, assert_close

pytestmark = pytest.mark.gpu

I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _call_noalloc(lib, x, w, st, pa, di, out):
    return lib.conv_fwd_noalloc(
        ctypes.c_void_p(x.data_ptr()), I5(*x.shape), ctypes.c_void_p(w.data_ptr()), I5(*w.shape),
        I3(*st), I3(*pa), I3(*di), 0, None, None, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_conv_fwd_on_two_calls_in_a_row(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    st, pa, di = (1, 1, 1), (1, 1, 1), (1, 1, 1)
    cases = [((1, 4, 8, 8, 16), (32, 3, 3, 3, 16)), ((2, 5, 9, 11, 64), (48, 3, 3, 3, 64))]
    for i, (xs, ws) in enumerate(cases):
        plan = pkg.conv_fwd_plan(xs, ws, st, pa, di)
        assert plan["splits"] > 1 and 0 < plan["workspace_bytes"] <= (8 << 20)
        x = cw.randn_bf16(xs, 700 + i, 1.0, "cuda")
        w = cw.randn_bf16(ws, 710 + i, 1.0 / np.sqrt(np.prod(ws[1:])), "cuda")
        ref = pkg.conv_fwd(x, w, st, pa, di)
        for call in range(2):
            out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call_noalloc(lib, x, w, st, pa, di, out) == pkg.CONV_OK
            torch.cuda.synchronize()
            assert pkg.conv_get_device_status() == 0
            assert_close(as_f64(out), as_f64(ref), f"noalloc {xs} call {call}")


def test_noalloc_rejects_scratch_beyond_its_maximum(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    lib.conv_last_error.restype = ctypes.c_char_p
    xs, ws = (1, 4, 8, 8, 64), (4096, 3, 3, 3, 64)
    plan = pkg.conv_fwd_plan(xs, ws, 1, 1, 1)
    assert plan["workspace_bytes"] > (8 << 20)
    x = torch.zeros(xs, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(ws, dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 4, 8, 8, 4096), dtype=torch.bfloat16, device="cuda")
    rc = _call_noalloc(lib, x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1), out)
    assert rc == pkg.CONV_ERR_INVALID
    assert b"static scratch" in lib.conv_last_error()
