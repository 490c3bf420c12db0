"""GPU parity of conv_fwd_ncdhw: T x 1 x 1 (and pointwise) convolutions of a
channel-major NCDHW activation read in place through position-contiguous
(MN-major) A tiles, against the fp64 oracle evaluated on the same NCDHW
bytes, element by element; forced plans (CTA pairs, row sub-tiles, k-step
width, split-K, launch slices); bit-equality with conv_fwd of the NDHWC copy
when both run the same plan; the argument checks."""
import contextlib
import os

import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, bits16

pytestmark = pytest.mark.gpu

MAX_FULL_MACS = 3e8   # full oracle evaluation below this, sampled above


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


# (x NCDHW, K, T, temporal stride, pad, dilation)
CASES = [
    ((1, 64, 6, 8, 16), 32, 3, 1, 1, 1),       # H*W = 128: one tile row per plane
    ((2, 136, 5, 10, 20), 100, 3, 1, 1, 1),    # ragged H*W tail, C past a chunk, K % 8 = 4
    ((1, 24, 9, 6, 12), 7, 5, 2, 2, 1),        # odd K, temporal stride
    ((3, 16, 4, 2, 4), 40, 2, 1, 1, 2),        # H*W = 8, dilation
    ((1, 640, 3, 4, 90), 640, 3, 1, 1, 1),     # the temporal workload's channels
    ((2, 64, 3, 16, 24), 48, 1, 1, 0, 1),      # pointwise
    ((1, 512, 2, 8, 45), 48, 1, 1, 0, 1),      # pointwise, 512 -> 48 filters
    ((1, 8, 7, 3, 8), 256, 3, 1, 0, 1),        # C = 8 (one row of a 64-channel box), no pad
]


def _operands(xs, K, T, seed):
    N, C, D, H, W = xs
    x = cw.randn_bf16(xs, 4100 + seed, 1.0, "cuda")
    w = cw.randn_bf16((K, T, 1, 1, C), 4200 + seed, 1.0 / np.sqrt(C * T), "cuda")
    return x, w


def _geometry(case):
    xs, K, T, sd, pd, dd = case
    return xs, K, T, (sd, 1, 1), (pd, 0, 0), (dd, 1, 1)


def _reference(x, w, st, pa, di, od, seed, scale=1.0, bias=None):
    """Oracle values at every output (or, for the larger cases, 200k sampled
    ones plus the first and last rows); returns (flat indices, values)."""
    total = int(np.prod(od))
    xs = tuple(x.shape)
    macs = total * xs[1] * w.shape[1]
    if macs <= MAX_FULL_MACS:
        idx = np.arange(total, dtype=np.int64)
    else:
        K = od[-1]
        rng = np.random.default_rng(seed)
        idx = np.concatenate([rng.integers(0, total, size=200000),
                              np.arange(min(total, 256 * K)),
                              np.arange(max(0, total - 256 * K), total)]).astype(np.int64)
    ref = oracle.conv3d_points(bits16(x), bits16(w), idx, st, pa, di, scale, 1.0,
                               bias=bias, x_layout="ncdhw")
    return idx, ref


def _got(y, idx):
    return as_f64(y).ravel()[idx]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_ncdhw_matches_oracle(pkg, i):
    xs, K, T, st, pa, di = _geometry(CASES[i])
    x, w = _operands(xs, K, T, i)
    y = pkg.conv_fwd_ncdhw(x, w, st, pa, di)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    idx, ref = _reference(x, w, st, pa, di, tuple(y.shape), i)
    assert_close(_got(y, idx), ref, f"ncdhw case {i} x{xs} K{K} T{T}")


def test_ncdhw_bias_and_scales(pkg):
    xs, K, T, st, pa, di = _geometry(CASES[1])
    x, w = _operands(xs, K, T, 40)
    g = torch.Generator(device="cpu").manual_seed(41)
    bias = torch.randn(K, generator=g).float().cuda()
    sx = torch.tensor([0.5], device="cuda")
    sw = torch.tensor([3.0], device="cuda")
    y = pkg.conv_fwd_ncdhw(x, w, st, pa, di, scale_x=sx, scale_w=sw, bias=bias)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    idx, ref = _reference(x, w, st, pa, di, tuple(y.shape), 40, scale=1.5,
                          bias=bias.cpu().double().numpy())
    assert_close(_got(y, idx), ref, "ncdhw bias + scales")


def _random_case(rng):
    N = int(rng.integers(1, 4))
    C = 8 * int(rng.integers(1, 40))
    K = int(rng.integers(1, 300))
    T = int(rng.integers(1, 5))
    sd, dd = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    pd = int(rng.integers(0, T))
    D = int(rng.integers(max(1, dd * (T - 1) + 1 - 2 * pd), 8))
    hw = 8 * int(rng.integers(1, 60))
    H = int(rng.choice([d for d in range(1, 9) if hw % d == 0]))
    return (N, C, D, H, hw // H), K, T, (sd, 1, 1), (pd, 0, 0), (dd, 1, 1)


def _random_plan(rng):
    bn = 32 * int(rng.integers(1, 9))
    bk = int(rng.choice([128, 256]))
    stages = int(rng.choice([0, 2, 3, 4]))
    splits = int(rng.choice([1, 1, 2, 3]))
    return {"tile": f"{bn},{bk},{stages},{int(rng.choice([1, 4]))},{splits}",
            "pair": int(rng.integers(0, 2)), "msub": int(rng.integers(1, 3)),
            "slices": int(rng.choice([1, 2, 3])),
            "hw_major": int(rng.integers(0, 2))}


@pytest.mark.parametrize("i", range(24))
def test_ncdhw_random_plans(pkg, i):
    rng = np.random.default_rng(5200 + i)
    while True:
        xs, K, T, st, pa, di = _random_case(rng)
        do = (xs[2] + 2 * pa[0] - di[0] * (T - 1) - 1) // st[0] + 1
        if do >= 1 and xs[0] * do * xs[3] * xs[4] * K * xs[1] * T <= 6e7:
            break
    env = _random_plan(rng)
    x, w = _operands(xs, K, T, 100 + i)
    plan = None
    with pkg.overrides(**env):
        try:
            plan = pkg.conv_fwd_ncdhw_plan(xs, tuple(w.shape), st, pa, di)
        except pkg.ConvError:   # a forced tile this shape cannot take: default plan
            pass
    if plan is None:
        env, plan = {}, pkg.conv_fwd_ncdhw_plan(xs, tuple(w.shape), st, pa, di)
    with pkg.overrides(**env):
        y = pkg.conv_fwd_ncdhw(x, w, st, pa, di)
        torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert plan["class"] == "temporal" and plan["k_bytes"] in (128, 256)
    idx, ref = _reference(x, w, st, pa, di, tuple(y.shape), 100 + i)
    assert_close(_got(y, idx), ref, f"ncdhw random {i}: x{xs} K{K} T{T} {env} {plan}")


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[4]], ids=["128", "ragged", "c640"])
def test_ncdhw_bit_equal_to_channel_last_path(pkg, case):
    """Same plan, same reduction order: conv_fwd_ncdhw over x and conv_fwd
    over its NDHWC copy give the same bits (the operand's major-ness changes
    only where the tile is read from)."""
    xs, K, T, st, pa, di = _geometry(case)
    x, w = _operands(xs, K, T, 77)
    xn = x.permute(0, 2, 3, 4, 1).contiguous()
    p_mn = pkg.conv_fwd_ncdhw_plan(xs, tuple(w.shape), st, pa, di)
    p_k = pkg.conv_fwd_plan(tuple(xn.shape), tuple(w.shape), st, pa, di)
    if p_mn != p_k:
        pytest.skip(f"plans differ: {p_mn} vs {p_k}")
    a = pkg.conv_fwd_ncdhw(x, w, st, pa, di)
    b = pkg.conv_fwd(xn, w, st, pa, di)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ncdhw_rejects_uncovered_shapes(pkg):
    x = torch.zeros((1, 64, 4, 8, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.ConvError) as e:   # a spatial filter
        pkg.conv_fwd_ncdhw(x, torch.zeros((32, 1, 3, 3, 64), dtype=torch.bfloat16,
                                          device="cuda"), 1, (0, 1, 1), 1)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    x5 = torch.zeros((1, 64, 4, 5, 5), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.ConvError) as e:   # H*W = 25
        pkg.conv_fwd_ncdhw(x5, torch.zeros((32, 3, 1, 1, 64), dtype=torch.bfloat16,
                                           device="cuda"), 1, (1, 0, 0), 1)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        pkg.conv_fwd_ncdhw(x.to(torch.float8_e4m3fn),
                           torch.zeros((32, 3, 1, 1, 64), dtype=torch.float8_e4m3fn,
                                       device="cuda"), 1, (1, 0, 0), 1)


# Channel planes past 1 MB with several taps: x is packed to an NDHWC copy in
# the workspace, then convolved.
PIPE_CASES = [
    ((1, 16, 40, 128, 128), 32, 3, 1, 1, 1),    # 1.3 MB channel planes
    ((2, 16, 32, 128, 160), 48, 2, 1, 1, 1),    # two images
    ((1, 32, 36, 128, 128), 40, 3, 2, 2, 2),    # temporal stride and dilation
]


@pytest.mark.parametrize("i", range(len(PIPE_CASES)))
def test_ncdhw_packed_copy_matches_oracle(pkg, i):
    xs, K, T, st, pa, di = _geometry(PIPE_CASES[i])
    x, w = _operands(xs, K, T, 300 + i)
    plan = pkg.conv_fwd_ncdhw_plan(xs, tuple(w.shape), st, pa, di)
    assert plan["workspace_bytes"] >= x.numel() * 2   # the NDHWC copy
    y = pkg.conv_fwd_ncdhw(x, w, st, pa, di)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    idx, ref = _reference(x, w, st, pa, di, tuple(y.shape), 300 + i)
    assert_close(_got(y, idx), ref, f"packed-copy case {i} x{xs} K{K} T{T}")
    # the same bits as conv_fwd over an NDHWC copy (same plan, same reduction order)
    xn = x.permute(0, 2, 3, 4, 1).contiguous()
    b = pkg.conv_fwd(xn, w, st, pa, di)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), b.view(torch.int16))


def test_ncdhw_small_workspace_reads_in_place(pkg):
    """Without room for the NDHWC copy (or with the ncdhw_in_place override) the
    same problem reads x in place; both against the oracle."""
    xs, K, T, st, pa, di = _geometry(PIPE_CASES[0])
    x, w = _operands(xs, K, T, 310)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    a = pkg.conv_fwd_ncdhw(x, w, st, pa, di, workspace=ws)
    with pkg.overrides(ncdhw_in_place=1):
        b = pkg.conv_fwd_ncdhw(x, w, st, pa, di)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    idx, ref = _reference(x, w, st, pa, di, tuple(a.shape), 310)
    assert_close(_got(a, idx), ref, "in place (small workspace)")
    assert_close(_got(b, idx), ref, "in place (forced)")


def test_ncdhw_packed_copy_on_side_stream(pkg):
    """The call on a non-default stream: the result is ordered on that stream."""
    xs, K, T, st, pa, di = _geometry(PIPE_CASES[1])
    x, w = _operands(xs, K, T, 320)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = pkg.conv_fwd_ncdhw(x, w, st, pa, di, stream=s)
        z = y.float().sum()
    s.synchronize()
    xn = x.permute(0, 2, 3, 4, 1).contiguous()
    b = pkg.conv_fwd(xn, w, st, pa, di)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), b.view(torch.int16))
    assert torch.isfinite(z)
