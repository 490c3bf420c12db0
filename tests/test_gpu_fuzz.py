"""Seeded random parity sweep of the forward convolution.

Each case draws a random problem of one dispatch class (im2col implicit GEMM,
temporal T x 1 x 1, point-output GEMM, pointwise GEMM, non-overlapping
patches) in bf16 or fp8-e4m3, an optional bias and activation, and a random
plan (tile width, k-step bytes, pipeline depth, raster group, split-K, CTA
pair, row sub-tiles, launch slices) forced through the plan overrides.  A plan
the library rejects for the shape falls back to the default plan, so every
drawn problem runs.  Every output element is compared with the fp64 oracle
on the exact bytes the GPU consumed."""
import contextlib
import os

import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, oracle_conv

pytestmark = pytest.mark.gpu

N_CASES = 96
MAX_MACS = 4e7   # keeps each oracle call well under a second


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _out_len(n, f, s, p, d):
    return (n + 2 * p - d * (f - 1) - 1) // s + 1


def _draw_problem(rng):
    fp8 = bool(rng.random() < 0.3)
    kind = rng.choice(["generic", "temporal", "point", "pointwise", "patch"],
                      p=[0.40, 0.20, 0.13, 0.12, 0.15])
    K = int(rng.integers(1, 321))
    if kind == "point":
        T, R, S = (int(v) for v in rng.integers(1, 9, size=3))
        C = int(rng.integers(1, 9)) * (4 if fp8 else 2)
        N = int(rng.integers(1, 400))
        return fp8, kind, (N, T, R, S, C), (K, T, R, S, C), (T, R, S), (0, 0, 0), (1, 1, 1)
    if kind == "patch":
        # stride == filter, zero padding, many patches, leftovers past the
        # last whole patch; channels an RGB-like count or a 16-byte multiple
        T = int(rng.choice([1, 1, 2]))
        R, S = (int(v) for v in rng.integers(2, 17, size=2))
        C = int(rng.choice([1, 3, 4, 8, 16])) * (4 if fp8 and rng.random() < 0.5 else 1)
        D = T * int(rng.integers(1, 3)) + int(rng.integers(0, T))
        H = R * int(rng.integers(1, 5)) + int(rng.integers(0, R))
        W = S * int(rng.integers(1, 5)) + int(rng.integers(0, S))
        N = int(rng.integers(1, 5))
        return fp8, kind, (N, D, H, W, C), (K, T, R, S, C), (T, R, S), (0, 0, 0), (1, 1, 1)
    C = int(rng.integers(1, 25)) * (16 if fp8 else 8)
    N = int(rng.integers(1, 4))
    if kind == "pointwise":
        D, H, W = (int(v) for v in rng.integers(1, 12, size=3))
        return fp8, kind, (N, D, H, W, C), (K, 1, 1, 1, C), (1, 1, 1), (0, 0, 0), (1, 1, 1)
    if kind == "temporal":
        T = int(rng.integers(1, 6))
        sd, dd = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        pd = int(rng.integers(0, T))
        D = int(rng.integers(max(1, dd * (T - 1) + 1 - 2 * pd), 9))
        H, W = int(rng.integers(1, 20)), int(rng.integers(1, 40))
        return fp8, kind, (N, D, H, W, C), (K, T, 1, 1, C), (sd, 1, 1), (pd, 0, 0), (dd, 1, 1)
    f = [int(v) for v in rng.integers(1, 4, size=3)]
    if f[1] == 1 and f[2] == 1:
        f[2] = 3
    st = [int(v) for v in rng.integers(1, 4, size=3)]
    dl = [int(v) for v in rng.integers(1, 3, size=3)]
    pd = [int(rng.integers(0, fi)) if fi > 1 else 0 for fi in f]
    ext = [max(1, d * (fi - 1) + 1 - 2 * p) for fi, d, p in zip(f, dl, pd)]
    D, H, W = (int(rng.integers(e, e + 9)) for e in ext)
    return fp8, kind, (N, D, H, W, C), (K, *f, C), tuple(st), tuple(pd), tuple(dl)


def _draw_plan(rng):
    bn = 32 * int(rng.integers(1, 9))
    bk = int(rng.choice([32, 64, 128, 256]))
    stages = int(rng.choice([0, 0, 2, 3, 4, 6]))
    group = int(rng.choice([1, 2, 4, 8]))
    splits = int(rng.choice([1, 1, 2, 3, 5]))
    return {"tile": f"{bn},{bk},{stages},{group},{splits}",
            "pair": int(rng.integers(0, 2)), "msub": int(rng.integers(1, 3)),
            "slices": int(rng.choice([1, 1, 2, 3]))}


def _case(i):
    rng = np.random.default_rng(7000 + i)
    while True:
        prob = _draw_problem(rng)
        fp8, kind, xs, ws, st, pa, di = prob
        od = [_out_len(n, f, s, p, d) for n, f, s, p, d in zip(xs[1:4], ws[1:4], st, pa, di)]
        macs = xs[0] * od[0] * od[1] * od[2] * ws[0] * ws[1] * ws[2] * ws[3] * ws[4]
        if min(od) >= 1 and macs <= MAX_MACS:
            return prob, _draw_plan(rng)


def _epilogue(i, K):
    """Cases 0-95 draw nothing here (their draws stay as they were); an
    independent generator picks a bias (fp32 [K]) and an activation."""
    rng = np.random.default_rng(17000 + i)
    bias = rng.standard_normal(K).astype(np.float32) * 0.5 if rng.random() < 0.35 else None
    act = str(rng.choice(["none", "none", "none", "relu", "silu", "gelu"]))
    return bias, act


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem_random_plan(pkg, i):
    (fp8, kind, xs, ws, st, pa, di), plan = _case(i)
    crs = ws[1] * ws[2] * ws[3] * ws[4]
    x = cw.randn_bf16(xs, 8000 + i, 1.0, "cuda")
    w = cw.randn_bf16(ws, 9000 + i, 1.0 / np.sqrt(crs), "cuda")
    sx = sw = None
    sxv = swv = 1.0
    if fp8:
        # e4m3 operands by torch's cast (input generation only), with scales
        x = x.float().to(torch.float8_e4m3fn)
        w = w.float().to(torch.float8_e4m3fn)
        sxv, swv = 0.75, 1.5
        sx = torch.tensor([sxv], device="cuda")
        sw = torch.tensor([swv], device="cuda")
    dtype = 1 if fp8 else 0
    try:
        pkg.conv_fwd_plan(xs, ws, st, pa, di, dtype)
    except pkg.ConvError as e:
        assert e.status == pkg.CONV_ERR_UNSUPPORTED
        pytest.skip(f"shape outside coverage: {e}")
    env = plan
    with pkg.overrides(**env):
        try:
            p = pkg.conv_fwd_plan(xs, ws, st, pa, di, dtype)
        except pkg.ConvError:
            env, p = {}, None
    bias, act = _epilogue(i, ws[0])
    bias_t = torch.from_numpy(bias).cuda() if bias is not None else None
    with pkg.overrides(**env):
        if p is None:
            p = pkg.conv_fwd_plan(xs, ws, st, pa, di, dtype)
        y = pkg.conv_fwd(x, w, st, pa, di, scale_x=sx, scale_w=sw, bias=bias_t, act=act)
        torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle_conv(x, w, st, pa, di, sxv, swv)
    if bias is not None:
        ref = ref + bias.astype(np.float64)
    ref = oracle.activate(ref, act)
    assert_close(as_f64(y), ref, f"case {i}: {kind} fp8={fp8} x{xs} w{ws} s{st} p{pa} d{di} "
                                 f"env={env} plan={p} bias={bias is not None} act={act}")
