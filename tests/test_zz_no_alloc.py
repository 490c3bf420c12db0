"""conv_fwd_noalloc: the entry point for callers that cannot allocate device
memory (for example engines that reserve all device memory up front, or
latency-bound code that cannot afford cudaMalloc's implicit synchronisation).
It keeps split-K partials and operand copies in the library's static device
scratch instead of a caller workspace.

Called here through the C ABI (ctypes) and checked against the fp64 oracle,
element by element, and against conv_fwd bit for bit (both run the same plan
and the split-K reduction sums in a fixed order).  The scratch keeps the
previous call's contents, so the calls alternate between problems of
different partial sizes (the larger first) and repeat each one: stale
partials of an earlier call must not reach a later result.  Point-output
problems put their aligned operand copies in the scratch (the two-phase
weight copies, or both operands), and a patch-class problem its gathered
rows.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import conv_workloads as cw
from _gpu_util import as_f64, assert_close, oracle_conv

pytestmark = pytest.mark.gpu

I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3
SCRATCH = 8 << 20   # CONV_NOALLOC_SCRATCH_BYTES


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


# (x NDHWC, w KTRSC, stride, pad, dil, plan class, what lands in the scratch)
CASES = [
    ((2, 5, 9, 11, 64), (224, 3, 3, 3, 64), (1, 1, 1), (1, 1, 1), (1, 1, 1), "generic",
     "split-K partials (the largest)"),
    ((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), (1, 1, 1), (1, 1, 1), (1, 1, 1), "generic",
     "split-K partials (small, another K)"),
    ((1100, 1, 14, 14, 3), (256, 1, 14, 14, 3), (1, 14, 14), (0, 0, 0), (1, 1, 1), "point_gemm",
     "two shifted weight copies (1176-byte rows)"),
    ((4000, 1, 3, 3, 2), (96, 1, 3, 3, 2), (1, 3, 3), (0, 0, 0), (1, 1, 1), "point_gemm",
     "aligned copies of both operands (36-byte rows)"),
    ((4, 1, 64, 64, 3), (128, 1, 16, 16, 3), (1, 16, 16), (0, 0, 0), (1, 1, 1), "patch_gemm",
     "gathered patch rows and weights"),
]


def _operands(case, i):
    xs, ws = case[0], case[1]
    x = cw.randn_bf16(xs, 700 + i, 1.0, "cuda")
    w = cw.randn_bf16(ws, 710 + i, 1.0 / np.sqrt(np.prod(ws[1:])), "cuda")
    return x, w


def test_noalloc_matches_oracle_and_conv_fwd_over_alternating_calls(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    prepared = []
    for i, case in enumerate(CASES):
        xs, ws, st, pa, di, cls, _ = case
        plan = pkg.conv_fwd_plan(xs, ws, st, pa, di)
        assert plan["class"] == cls and 0 < plan["workspace_bytes"] <= SCRATCH, (case, plan)
        x, w = _operands(case, i)
        ref = oracle_conv(x, w, st, pa, di)
        y = pkg.conv_fwd(x, w, st, pa, di)   # conv_fwd with its preferred workspace
        prepared.append((case, x, w, ref, y))
    assert prepared[0][0][5] == "generic"
    # the largest partials first, then every other problem, then all again
    for rnd in range(2):
        for case, x, w, ref, y in prepared:
            xs, ws, st, pa, di, cls, what = case
            out = torch.full(y.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call_noalloc(lib, x, w, st, pa, di, out) == pkg.CONV_OK
            torch.cuda.synchronize()
            assert pkg.conv_get_device_status() == 0
            label = f"noalloc {cls} ({what}) call {rnd}"
            assert_close(as_f64(out), ref, label)
            assert torch.equal(out.view(torch.int16), y.view(torch.int16)), label


def test_noalloc_rejects_scratch_beyond_its_maximum(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    lib.conv_last_error.restype = ctypes.c_char_p
    xs, ws = (1, 4, 8, 8, 64), (4096, 3, 3, 3, 64)
    plan = pkg.conv_fwd_plan(xs, ws, 1, 1, 1)
    assert plan["workspace_bytes"] > SCRATCH
    x = torch.zeros(xs, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(ws, dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 4, 8, 8, 4096), dtype=torch.bfloat16, device="cuda")
    rc = _call_noalloc(lib, x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1), out)
    assert rc == pkg.CONV_ERR_INVALID
    assert b"static scratch" in lib.conv_last_error()
    # a patch-class problem whose gathered rows exceed the scratch
    xs, ws = (64, 1, 224, 224, 3), (768, 1, 16, 16, 3)
    assert pkg.conv_fwd_plan(xs, ws, (1, 16, 16), 0, 1)["workspace_bytes"] > SCRATCH
    x = torch.zeros(xs, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(ws, dtype=torch.bfloat16, device="cuda")
    out = torch.empty((64, 1, 14, 14, 768), dtype=torch.bfloat16, device="cuda")
    rc = _call_noalloc(lib, x, w, (1, 16, 16), (0, 0, 0), (1, 1, 1), out)
    assert rc == pkg.CONV_ERR_INVALID
