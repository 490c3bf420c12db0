"""GPU checks of conv_fwd_from_host: the convolution of host operands with the
copies overlapped with the kernel, slice by slice.

Every slice runs the same kernel and plan as conv_fwd over a range of its
work units, so the host result must equal conv_fwd's device result bit for
bit; the small cases are also compared with the fp64 oracle.  The device
buffers must end up holding copies of x, w and out."""
import numpy as np
import pytest
import torch

import conv_workloads as cw
from _gpu_util import as_f64, assert_close, oracle_conv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _operands(xs, ws, seed, fp8=False):
    crs = ws[1] * ws[2] * ws[3] * ws[4]
    x = cw.randn_bf16(xs, 600 + seed, 1.0, "cuda")
    w = cw.randn_bf16(ws, 700 + seed, 1.0 / np.sqrt(crs), "cuda")
    if fp8:
        x, w = x.float().to(torch.float8_e4m3fn), w.float().to(torch.float8_e4m3fn)
    return x, w


def _run(pkg, x, w, st, pa, di, chunks, pinned=True, sx=None, sw=None, stream=None,
         split_k=False):
    """conv_fwd_from_host on host copies of x and w.  split_k=False passes a
    16-byte workspace, so the plan has no split-K and the sliced path runs."""
    hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=pinned)
    hw = torch.empty(w.shape, dtype=w.dtype, pin_memory=pinned)
    hx.copy_(x.cpu())
    hw.copy_(w.cpu())
    od = pkg.conv_out_dims(tuple(x.shape), tuple(w.shape), st, pa, di)
    hout = torch.full(od, float("nan"), dtype=torch.bfloat16, pin_memory=pinned)
    # device buffers of NaN bytes (0xFF is NaN in bf16 and e4m3): a slice that
    # read input rows or weights before their copy landed computes NaNs
    xd, wd = torch.empty_like(x), torch.empty_like(w)
    xd.view(torch.uint8).fill_(0xFF)
    wd.view(torch.uint8).fill_(0xFF)
    outd = torch.full(od, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = None if split_k else torch.empty(16, dtype=torch.uint8, device="cuda")
    pkg.conv_fwd_from_host(hx, hw, st, pa, di, scale_x=sx, scale_w=sw, out_host=hout, x_dev=xd,
                           w_dev=wd, out_dev=outd, workspace=ws, chunks=chunks, stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    assert pkg.conv_get_device_status() == 0
    assert torch.equal(xd.view(torch.uint8), x.view(torch.uint8))
    assert torch.equal(wd.view(torch.uint8), w.view(torch.uint8))
    assert torch.equal(outd.cpu().view(torch.int16), hout.view(torch.int16))
    return hout


CASES = [
    # (x NDHWC, w KTRSC, stride, pad, dil): several output planes, N > 1,
    # strides and dilation along D, so the copied prefix of planes varies
    ((2, 6, 12, 10, 64), (96, 3, 3, 3, 64), 1, 1, 1),
    ((1, 9, 8, 11, 32), (64, 3, 3, 3, 32), (2, 1, 1), (1, 1, 1), (2, 1, 1)),
    ((3, 5, 7, 9, 16), (40, 2, 3, 3, 16), 1, (0, 1, 1), 1),
    ((1, 8, 10, 20, 64), (72, 3, 1, 1, 64), 1, (1, 0, 0), 1),        # temporal
    ((2, 7, 6, 30, 32), (48, 5, 1, 1, 32), (2, 1, 1), (2, 0, 0), 1),  # temporal, stride 2
    ((1, 4, 9, 9, 32), (32, 3, 3, 3, 32), 1, (3, 1, 1), 1),           # planes read only padding
    ((1, 5, 23, 6, 32), (48, 3, 3, 3, 32), (1, 2, 1), (1, 2, 1), 1),  # H stride: rows skipped
    ((2, 4, 19, 5, 16), (40, 2, 3, 2, 16), 1, (0, 3, 1), (1, 3, 2)),  # H dilation, big pad
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("chunks", [0, 1, 2, 3, 7])
def test_host_pipeline_matches_device_path_and_oracle(pkg, case, chunks):
    xs, ws, st, pa, di = case
    x, w = _operands(xs, ws, CASES.index(case))
    hout = _run(pkg, x, w, st, pa, di, chunks)
    ref_dev = pkg.conv_fwd(x, w, st, pa, di, split_k=False)
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref_dev.cpu().view(torch.int16))
    if chunks in (0, 3):
        st3, pa3, di3 = pkg._triple(st), pkg._triple(pa), pkg._triple(di)
        assert_close(as_f64(hout), oracle_conv(x, w, st3, pa3, di3), f"host {case} chunks={chunks}")


def test_host_pipeline_auto_slices_whole_waves(pkg):
    """A problem with several waves of work units: the automatic slicing is
    on; the result equals conv_fwd's bit for bit."""
    xs, ws = (2, 8, 64, 64, 32), (64, 3, 3, 3, 32)
    x, w = _operands(xs, ws, 20)
    for chunks in (0, 5):
        hout = _run(pkg, x, w, 1, 1, 1, chunks)
        ref = pkg.conv_fwd(x, w, 1, 1, 1, split_k=False)
        torch.cuda.synchronize()
        assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))


def test_host_pipeline_fp8_and_side_stream(pkg):
    x, w = _operands((2, 6, 12, 10, 64), (96, 3, 3, 3, 64), 21, fp8=True)
    sx = torch.tensor([0.5], device="cuda")
    sw = torch.tensor([1.25], device="cuda")
    s = torch.cuda.Stream()
    hout = _run(pkg, x, w, 1, 1, 1, 4, sx=sx, sw=sw, stream=s)
    ref = pkg.conv_fwd(x, w, 1, 1, 1, scale_x=sx, scale_w=sw, split_k=False)
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))


def test_host_pipeline_pageable_memory(pkg):
    x, w = _operands((1, 6, 10, 12, 32), (48, 3, 3, 3, 32), 22)
    hout = _run(pkg, x, w, 1, 1, 1, 3, pinned=False)
    assert_close(as_f64(hout), oracle_conv(x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1)), "pageable")


@pytest.mark.parametrize("case", [
    ((300, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0, 1),   # point-output GEMM
    ((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 1, 1, 1),                  # split-K plan
])
def test_host_pipeline_unsliced_plans(pkg, case):
    xs, ws, st, pa, di = case
    x, w = _operands(xs, ws, 23)
    hout = _run(pkg, x, w, st, pa, di, 0, split_k=True)
    ref = pkg.conv_fwd(x, w, st, pa, di)   # the same plan, split-K included
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))
    st3, pa3, di3 = pkg._triple(st), pkg._triple(pa), pkg._triple(di)
    assert_close(as_f64(hout), oracle_conv(x, w, st3, pa3, di3), f"unsliced {case}")


@pytest.mark.parametrize("bn", [128, 64])
def test_host_pipeline_first_slice_split_over_weight_groups(pkg, capfd, bn):
    """Eight (or sixteen) column tiles: the first slice runs as one wave per
    group of column tiles, each after its weight rows have landed.  The result
    equals conv_fwd's bit for bit, and the weights arrive whole on the
    device; with the split turned off (weight_groups=0) the bits are the
    same."""
    xs, ws = (1, 8, 48, 48, 64), (1024, 3, 3, 3, 64)
    x, w = _operands(xs, ws, 40 + bn)
    with pkg.overrides(tile=f"{bn},0,0,0,0", log=1):
        hout = _run(pkg, x, w, 1, 1, 1, 0)
        log = capfd.readouterr().err
        ref = pkg.conv_fwd(x, w, 1, 1, 1, split_k=False)
        torch.cuda.synchronize()
        plan_ctas = pkg.conv_fwd_plan(xs, ws, 1, 1, 1)["ctas"]
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))
    chunk0 = [ln for ln in log.splitlines() if ln.startswith("conv_fwd_from_host: chunk 0 ")]
    n_tiles = 1024 // bn
    if plan_ctas % 2 == 0:
        assert len(chunk0) >= 2, log   # split over weight groups
        assert chunk0[0].split("n-tiles ")[1].startswith("[0, ")
        assert not chunk0[0].split("n-tiles ")[1].startswith(f"[0, {n_tiles})")
    with pkg.overrides(tile=f"{bn},0,0,0,0", weight_groups=0):
        hout2 = _run(pkg, x, w, 1, 1, 1, 0)
    assert torch.equal(hout2.view(torch.int16), hout.view(torch.int16))



def test_slice_query_matches_the_launches(pkg, capfd):
    """conv_fwd_from_host_slices (the current device) names the output rows
    and weight groups conv_fwd_from_host then launches."""
    xs, ws = (1, 8, 48, 48, 64), (1024, 3, 3, 3, 64)
    x, w = _operands(xs, ws, 60)
    with pkg.overrides(tile="128,0,0,0,0"):
        plan = pkg.conv_fwd_from_host_slices(xs, ws, 1, 1, 1, workspace_bytes=16)
        with pkg.overrides(tile="128,0,0,0,0", log=1):
            _run(pkg, x, w, 1, 1, 1, 0)
            log = capfd.readouterr().err
    lines = [ln for ln in log.splitlines() if ln.startswith("conv_fwd_from_host: chunk ")]
    seen = []
    for ln in lines:
        lo, hi = (int(v) for v in ln.split("rows [")[1].split(")")[0].split(", "))
        if not seen or seen[-1] != (lo, hi):
            seen.append((lo, hi))
    assert seen == [tuple(r) for r in plan["rows"]], (seen, plan)
    first = [ln for ln in lines if ln.split()[2] == "0"]
    assert len(first) == plan["weight_groups"]
