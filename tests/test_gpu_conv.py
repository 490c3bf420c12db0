"""GPU parity of the bf16 forward convolution against the fp64 oracle, element
by element, through the C ABI.  Shapes span several tiles with ragged M and N
tails and cover every dispatch class (im2col implicit GEMM, temporal T x 1 x 1,
point-output / pointwise GEMM by TMA and by row gather), with and without
split-K, plus forced tile shapes, exact delta filters, the 2-D / 1-D wrappers
and NaN-prefilled canary guards."""

import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, bits16, oracle_conv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def forced_tile(spec):
    """Plan override: tile "BN,BK,stages,group_m,splits" (0 keeps the plan's)."""
    import implicit_gemm_convolution_conv3d_gb300 as p
    return p.overrides(tile=spec)


def _inputs(xs, ws, seed):
    C = ws[4]
    crs = ws[1] * ws[2] * ws[3] * C
    x = cw.randn_bf16(xs, 100 + seed, 1.0, "cuda")
    w = cw.randn_bf16(ws, 200 + seed, 1.0 / np.sqrt(crs), "cuda")
    return x, w


def _run_and_check(pkg, xs, ws, stride, pad, dil, seed, split_k=True, what=""):
    x, w = _inputs(xs, ws, seed)
    y = pkg.conv_fwd(x, w, stride, pad, dil, split_k=split_k)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    st, pa, di = pkg._triple(stride), pkg._triple(pad), pkg._triple(dil)
    ref = oracle_conv(x, w, st, pa, di)
    assert_close(as_f64(y), ref, what or f"{xs} {ws} s{stride} p{pad} d{dil} split={split_k}")
    return x, w, y


GENERIC = [
    ((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 1, 1, 1),
    ((2, 5, 9, 11, 64), (48, 3, 3, 3, 64), 1, 1, 1),
    ((1, 6, 10, 12, 24), (16, 3, 3, 3, 24), 1, 1, 1),
    ((1, 3, 17, 13, 8), (32, 1, 3, 3, 8), 1, (0, 1, 1), 1),
    ((2, 7, 9, 8, 136), (272, 3, 3, 3, 136), 1, 1, 1),
    ((1, 9, 12, 10, 32), (40, 3, 3, 3, 32), 2, 1, 1),
    ((1, 8, 11, 9, 16), (24, 3, 3, 3, 16), (1, 2, 3), (1, 0, 2), (2, 1, 1)),
    ((3, 4, 6, 5, 16), (32, 2, 2, 2, 16), 2, 0, 1),
    ((2, 5, 5, 5, 16), (32, 4, 4, 4, 16), 4, 0, 1),
    ((1, 1, 16, 16, 64), (64, 1, 3, 3, 64), 1, (0, 1, 1), (1, 2, 2)),
    ((1, 5, 20, 30, 256), (256, 3, 3, 3, 256), 1, 1, 1),
]

TEMPORAL = [
    ((1, 5, 10, 20, 64), (32, 3, 1, 1, 64), 1, (1, 0, 0), 1),
    ((2, 6, 8, 16, 16), (48, 3, 1, 1, 16), (2, 1, 1), (1, 0, 0), 1),
    ((1, 7, 9, 9, 32), (64, 5, 1, 1, 32), 1, (2, 0, 0), 1),
    ((1, 9, 4, 4, 128), (96, 3, 1, 1, 128), 1, (2, 0, 0), (2, 1, 1)),
    ((1, 4, 3, 50, 16), (16, 1, 1, 1, 16), (2, 1, 1), 0, 1),
    ((1, 6, 16, 90, 640), (640, 3, 1, 1, 640), 1, (1, 0, 0), 1),
]

POINT = [
    ((300, 1, 14, 14, 3), (1280, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((129, 2, 4, 4, 8), (96, 2, 4, 4, 8), (2, 4, 4), 0, 1),
    ((2, 3, 5, 7, 64), (80, 1, 1, 1, 64), 1, 0, 1),
    ((50, 1, 16, 16, 3), (64, 1, 16, 16, 3), (1, 16, 16), 0, 1),
    ((37, 1, 3, 3, 6), (40, 1, 3, 3, 6), (1, 3, 3), 0, 1),
]


def _ids(cases):
    return [f"x{c[0]}-w{c[1]}-s{c[2]}-p{c[3]}-d{c[4]}".replace(" ", "") for c in cases]


@pytest.mark.parametrize("case", GENERIC, ids=_ids(GENERIC))
@pytest.mark.parametrize("split_k", [True, False])
def test_generic_im2col(pkg, case, split_k):
    xs, ws, st, pa, di = case
    assert pkg.conv_fwd_plan(xs, ws, st, pa, di)["class"] == "generic"
    _run_and_check(pkg, xs, ws, st, pa, di, seed=GENERIC.index(case), split_k=split_k)


@pytest.mark.parametrize("case", TEMPORAL, ids=_ids(TEMPORAL))
@pytest.mark.parametrize("split_k", [True, False])
def test_temporal(pkg, case, split_k):
    xs, ws, st, pa, di = case
    assert pkg.conv_fwd_plan(xs, ws, st, pa, di)["class"] == "temporal"
    _run_and_check(pkg, xs, ws, st, pa, di, seed=50 + TEMPORAL.index(case), split_k=split_k)


@pytest.mark.parametrize("case", POINT, ids=_ids(POINT))
@pytest.mark.parametrize("split_k", [True, False])
def test_point_gemm(pkg, case, split_k):
    xs, ws, st, pa, di = case
    assert pkg.conv_fwd_plan(xs, ws, st, pa, di)["class"] == "point_gemm"
    _run_and_check(pkg, xs, ws, st, pa, di, seed=80 + POINT.index(case), split_k=split_k)


@pytest.mark.parametrize("spec", ["32,32,2,1,1", "64,64,3,2,1", "128,128,4,1,1", "256,128,2,3,1",
                                  "96,64,5,8,3", "160,128,3,2,2", "224,32,8,1,5"])
def test_forced_tiles_generic(pkg, spec):
    with forced_tile(spec):
        _run_and_check(pkg, (2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1, seed=7,
                       what=f"tile {spec}")


@pytest.mark.parametrize("spec", ["64,128,3,1,1", "256,128,4,4,1", "128,64,6,2,4"])
def test_forced_tiles_temporal_and_gemm(pkg, spec):
    bk = int(spec.split(",")[1])
    with forced_tile(spec):
        _run_and_check(pkg, (1, 5, 10, 20, 64), (200, 3, 1, 1, 64), 1, (1, 0, 0), 1, seed=9,
                       what=f"temporal tile {spec}")
        _run_and_check(pkg, (150, 1, 4, 4, 16), (100, 1, 4, 4, 16), (1, 4, 4), 0, 1, seed=10,
                       what=f"gemm tile {spec}")
        if bk == 128:
            _run_and_check(pkg, (300, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0, 1,
                           seed=11, what=f"gather tile {spec}")


def test_tiny_workload(pkg):
    wl = cw.BY_NAME["tiny_conv3d_bf16"]
    x, w = cw.make_inputs(wl, "cuda")
    for split_k in (True, False):
        y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil, split_k=split_k)
        torch.cuda.synchronize()
        assert_close(as_f64(y), oracle_conv(x, w, wl.stride, wl.pad, wl.dil), wl.name)


def test_split_k_is_deterministic(pkg):
    x, w = _inputs((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 3)
    a = pkg.conv_fwd(x, w, 1, 1, 1)
    b = pkg.conv_fwd(x, w, 1, 1, 1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_delta_filter_is_exact_shift(pkg):
    """One unit tap per output channel: every output is a single bf16 input
    value, so the GPU result must equal the shifted copy bit for bit."""
    C = 32
    x = cw.randn_bf16((2, 5, 7, 9, C), 5, 1.0, "cuda")
    for (T, R, S), tap, st, pa, di in [((3, 3, 3), (2, 0, 1), 1, 1, 1),
                                       ((1, 3, 3), (0, 2, 2), (1, 2, 1), (0, 1, 1), (1, 1, 2)),
                                       ((3, 1, 1), (0, 0, 0), (2, 1, 1), (1, 0, 0), (2, 1, 1))]:
        w = torch.zeros((C, T, R, S, C), dtype=torch.bfloat16, device="cuda")
        for k in range(C):
            w[k, tap[0], tap[1], tap[2], k] = 1.0
        y = pkg.conv_fwd(x, w, st, pa, di)
        torch.cuda.synchronize()
        ref = oracle_conv(x, w, pkg._triple(st), pkg._triple(pa), pkg._triple(di))
        assert np.array_equal(as_f64(y), ref)


def test_conv2d_and_conv1d_wrappers(pkg):
    x2 = cw.randn_bf16((2, 13, 11, 32), 21, 1.0, "cuda")
    w2 = cw.randn_bf16((48, 3, 3, 32), 22, 1.0 / np.sqrt(288), "cuda")
    y2 = pkg.conv2d(x2, w2, stride=(2, 1), padding=1)
    torch.cuda.synchronize()
    ref = oracle_conv(x2.unsqueeze(1), w2.unsqueeze(1), (1, 2, 1), (0, 1, 1), (1, 1, 1))
    assert_close(as_f64(y2), ref[:, 0], "conv2d")
    x1 = cw.randn_bf16((3, 41, 16), 23, 1.0, "cuda")
    w1 = cw.randn_bf16((24, 5, 16), 24, 1.0 / np.sqrt(80), "cuda")
    y1 = pkg.conv1d(x1, w1, stride=1, padding=2, dilation=2)
    torch.cuda.synchronize()
    ref = oracle_conv(x1[:, None, None], w1[:, None, None], (1, 1, 1), (0, 0, 2), (1, 1, 2))
    assert_close(as_f64(y1), ref[:, 0, 0], "conv1d")


def test_output_fully_written_and_canaries_untouched(pkg):
    """NaN-prefilled output inside a larger buffer: every output element is
    overwritten, and 4 KB guard regions on both sides stay NaN."""
    for xs, ws, st, pa in [((2, 5, 9, 11, 64), (48, 3, 3, 3, 64), 1, 1),
                           ((1, 5, 10, 20, 64), (40, 3, 1, 1, 64), 1, (1, 0, 0)),
                           ((37, 1, 3, 3, 6), (40, 1, 3, 3, 6), (1, 3, 3), 0)]:
        x, w = _inputs(xs, ws, 31)
        od = pkg.conv_out_dims(xs, ws, st, pa, 1)
        n = int(np.prod(od))
        guard = 2048   # bf16 elements = 4 KB
        buf = torch.full((guard + n + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
        out = buf[guard:guard + n].view(od)
        for split_k in (True, False):
            buf[guard:guard + n] = float("nan")
            pkg.conv_fwd(x, w, st, pa, 1, out=out, split_k=split_k)
            torch.cuda.synchronize()
            assert not torch.isnan(out).any()
            assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + n:]).all()
        ref = oracle_conv(x, w, pkg._triple(st), pkg._triple(pa), (1, 1, 1))
        assert_close(as_f64(out), ref, f"canary {xs}")


def test_scales_apply_to_bf16(pkg):
    x, w = _inputs((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 40)
    sx = torch.tensor([0.5], device="cuda")
    sw = torch.tensor([3.0], device="cuda")
    y = pkg.conv_fwd(x, w, 1, 1, 1, scale_x=sx, scale_w=sw)
    torch.cuda.synchronize()
    assert_close(as_f64(y), oracle_conv(x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1), 0.5, 3.0), "scaled")


def test_unsupported_shape_raises(pkg):
    x = torch.zeros((1, 4, 8, 8, 12), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 3, 3, 3, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd(x, w, 1, 1, 1)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED


# CTA-pair kernel (two SMs per 256-row unit), forced on small shapes with
# several units per pair and ragged M / N tails, for every TMA operand mode.
PAIR_CASES = [
    ((2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1, "128,128,0,0,1"),
    ((2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1, "256,128,0,0,1"),
    ((1, 6, 10, 12, 32), (96, 3, 3, 3, 32), (1, 2, 1), (1, 1, 0), (2, 1, 1), "96,64,0,0,1"),
    ((1, 5, 10, 50, 64), (200, 3, 1, 1, 64), 1, (1, 0, 0), 1, "224,128,0,0,1"),
    ((1, 7, 9, 30, 32), (64, 3, 1, 1, 32), 1, (1, 0, 0), 1, "64,64,0,0,1"),
    ((600, 1, 4, 4, 16), (160, 1, 4, 4, 16), (1, 4, 4), 0, 1, "160,128,0,0,1"),
    ((3, 4, 7, 9, 64), (256, 1, 1, 1, 64), 1, 0, 1, "256,128,0,0,1"),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[str(i) for i in range(len(PAIR_CASES))])
def test_cta_pair_kernel(pkg, case):
    xs, ws, st, pa, di, spec = case
    with pkg.overrides(pair=1), forced_tile(spec):
        _run_and_check(pkg, xs, ws, st, pa, di, seed=90 + PAIR_CASES.index(case),
                       split_k=False, what=f"pair {case}")


# Two row sub-tiles per unit sharing each B stage, with and without CTA pairs.
MSUB_CASES = [
    ((2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1, "128,128,0,0,1"),
    ((2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1, "256,128,0,0,1"),
    ((1, 6, 10, 12, 32), (96, 3, 3, 3, 32), (1, 2, 1), (1, 1, 0), (2, 1, 1), "96,64,0,0,1"),
    ((1, 5, 10, 70, 64), (200, 3, 1, 1, 64), 1, (1, 0, 0), 1, "224,128,0,0,1"),
    ((900, 1, 4, 4, 16), (160, 1, 4, 4, 16), (1, 4, 4), 0, 1, "160,128,0,0,1"),
]


@pytest.mark.parametrize("case", MSUB_CASES, ids=[str(i) for i in range(len(MSUB_CASES))])
@pytest.mark.parametrize("pair", [0, 1])
def test_two_row_subtiles(pkg, case, pair):
    xs, ws, st, pa, di, spec = case
    with pkg.overrides(msub=2, pair=pair), forced_tile(spec):
        _run_and_check(pkg, xs, ws, st, pa, di, seed=120 + MSUB_CASES.index(case),
                       split_k=False, what=f"msub2 pair={pair} {case}")


# 256-byte k-steps (two 128-byte swizzle boxes per operand and stage) with
# reduction rows that end inside the first box, inside the second, or on a
# k-step boundary, for every TMA operand mode, alone, paired and with two
# row sub-tiles; the last case adds split-K.
WIDE_K_CASES = [
    ((2, 5, 9, 11, 136), (272, 3, 3, 3, 136), 1, 1, 1),                  # 272 B rows
    ((1, 6, 10, 12, 256), (96, 3, 3, 3, 256), (1, 2, 1), (1, 1, 0), (2, 1, 1)),  # 512 B
    ((1, 4, 7, 9, 40), (64, 3, 3, 3, 40), 1, 1, 1),                      # 80 B: one box part-filled
    ((1, 5, 10, 50, 200), (200, 3, 1, 1, 200), 1, (1, 0, 0), 1),         # temporal, 400 B
    ((1, 7, 9, 30, 64), (64, 3, 1, 1, 64), 1, (1, 0, 0), 1),             # temporal, 128 B
    ((600, 1, 4, 4, 16), (160, 1, 4, 4, 16), (1, 4, 4), 0, 1),           # point GEMM, 512 B
    ((3, 4, 7, 9, 200), (256, 1, 1, 1, 200), 1, 0, 1),                   # pointwise, 400 B
    ((300, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0, 1),       # repacked rows, 1184 B
]
WIDE_K_PLANS = [(0, 1, "128,256,0,0,1"), (1, 1, "224,256,0,0,1"), (0, 2, "96,256,0,0,1"),
                (1, 2, "256,256,0,0,1"), (0, 1, "64,256,3,2,3")]


@pytest.mark.parametrize("case", WIDE_K_CASES, ids=[str(i) for i in range(len(WIDE_K_CASES))])
@pytest.mark.parametrize("plan", WIDE_K_PLANS, ids=[p[2] + f"-pair{p[0]}-msub{p[1]}"
                                                    for p in WIDE_K_PLANS])
def test_wide_k_steps(pkg, case, plan):
    xs, ws, st, pa, di = case
    pair, msub, spec = plan
    with pkg.overrides(msub=msub, pair=pair), forced_tile(spec):
        assert pkg.conv_fwd_plan(xs, ws, st, pa, di)["k_bytes"] == 256
        _run_and_check(pkg, xs, ws, st, pa, di, seed=140 + WIDE_K_CASES.index(case),
                       split_k=True, what=f"bk256 pair={pair} msub={msub} {spec} {case}")


# Point-output GEMM whose rows are 8 bytes past a 16-byte multiple (the 14x14x3
# patch embedding): two row phases over the caller's x, only the weights
# copied.  Odd and even image counts, two and three images, K below / not a
# multiple of 8 (direct-store epilogue), split-K, forced CTA pairs.
TWO_PHASE = [
    ((301, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((600, 1, 14, 14, 3), (96, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((2, 1, 14, 14, 3), (40, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((3, 1, 14, 14, 3), (36, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((517, 1, 2, 2, 1), (100, 1, 2, 2, 1), (1, 2, 2), 0, 1),     # 8-byte rows, K % 8 = 4
    ((260, 1, 2, 2, 5), (72, 1, 2, 2, 5), (1, 2, 2), 0, 1),      # 20 elements = 40-byte rows
]


@pytest.mark.parametrize("case", TWO_PHASE, ids=[str(i) for i in range(len(TWO_PHASE))])
@pytest.mark.parametrize("split_k", [True, False])
def test_point_gemm_two_phases(pkg, case, split_k):
    xs, ws, st, pa, di = case
    x, w = _inputs(xs, ws, 160 + TWO_PHASE.index(case))
    rb = ws[1] * ws[2] * ws[3] * ws[4] * 2
    assert rb % 16 == 8
    plan = pkg.conv_fwd_plan(xs, ws, st, pa, di)
    assert plan["class"] == "point_gemm"
    ws_t = None
    if not split_k:   # room for the weight copies only: no split-K
        ws_t = torch.empty(2 * ((ws[0] * (rb + 8) + 255) // 256 * 256), dtype=torch.uint8,
                           device="cuda")
    y = pkg.conv_fwd(x, w, st, pa, di, workspace=ws_t)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle_conv(x, w, pkg._triple(st), pkg._triple(pa), pkg._triple(di))
    assert_close(as_f64(y), ref, f"two-phase {case} split={split_k}")
    if split_k:
        # the same problem through the full operand repack (two_phase=0)
        with pkg.overrides(two_phase=0):
            y1 = pkg.conv_fwd(x, w, st, pa, di)
            torch.cuda.synchronize()
        assert_close(as_f64(y1), ref, f"repack {case}")


@pytest.mark.parametrize("pair", [0, 1])
def test_point_gemm_two_phases_forced_pair(pkg, pair):
    xs, ws = (1100, 1, 14, 14, 3), (256, 1, 14, 14, 3)
    with pkg.overrides(pair=pair), forced_tile("128,128,0,1,1"):
        _run_and_check(pkg, xs, ws, (1, 14, 14), 0, 1, seed=170, split_k=True,
                       what=f"two-phase pair={pair}")


# Per-filter fp32 bias through conv_fwd_bias: every dispatch class, ragged K
# (direct-store tail), with and without split-K (the bias then enters once,
# in the reduction).
BIAS_CASES = [
    ((2, 5, 9, 11, 64), (272, 3, 3, 3, 64), 1, 1, 1),
    ((1, 5, 10, 20, 64), (200, 3, 1, 1, 64), 1, (1, 0, 0), 1),
    ((300, 1, 14, 14, 3), (200, 1, 14, 14, 3), (1, 14, 14), 0, 1),
    ((37, 1, 3, 3, 6), (40, 1, 3, 3, 6), (1, 3, 3), 0, 1),
    ((1, 4, 8, 8, 16), (36, 3, 3, 3, 16), 1, 1, 1),
]


@pytest.mark.parametrize("case", BIAS_CASES, ids=[str(i) for i in range(len(BIAS_CASES))])
@pytest.mark.parametrize("split_k", [True, False])
def test_bias(pkg, case, split_k):
    xs, ws, st, pa, di = case
    x, w = _inputs(xs, ws, 180 + BIAS_CASES.index(case))
    g = torch.Generator(device="cpu").manual_seed(190 + BIAS_CASES.index(case))
    b = (torch.randn(ws[0], generator=g) * 0.5).float()
    y = pkg.conv_fwd(x, w, st, pa, di, split_k=split_k, bias=b.cuda())
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    st3, pa3, di3 = pkg._triple(st), pkg._triple(pa), pkg._triple(di)
    ref = oracle.conv3d(bits16(x), bits16(w), st3, pa3, di3, bias=b.double().numpy())
    assert_close(as_f64(y), ref, f"bias {case} split={split_k}")


@pytest.mark.parametrize("act", ["relu", "silu", "gelu"])
@pytest.mark.parametrize("case", BIAS_CASES, ids=[str(i) for i in range(len(BIAS_CASES))])
@pytest.mark.parametrize("split_k", [True, False])
def test_bias_activation(pkg, case, split_k, act):
    """bias + activation epilogue (conv_fwd_bias_act) in every store path:
    TMA tensor stores, staged 8-/4-byte stores, direct stores, the split-K
    reduction; against the fp64 oracle's textbook activation."""
    xs, ws, st, pa, di = case
    x, w = _inputs(xs, ws, 180 + BIAS_CASES.index(case))
    g = torch.Generator(device="cpu").manual_seed(190 + BIAS_CASES.index(case))
    b = (torch.randn(ws[0], generator=g) * 0.5).float()
    y = pkg.conv_fwd(x, w, st, pa, di, split_k=split_k, bias=b.cuda(), act=act)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    st3, pa3, di3 = pkg._triple(st), pkg._triple(pa), pkg._triple(di)
    ref = oracle.conv3d(bits16(x), bits16(w), st3, pa3, di3, bias=b.double().numpy(), act=act)
    assert_close(as_f64(y), ref, f"bias+{act} {case} split={split_k}")


def test_activation_without_bias_and_bad_code(pkg):
    xs, ws = (2, 5, 9, 11, 64), (272, 3, 3, 3, 64)
    x, w = _inputs(xs, ws, 185)
    y = pkg.conv_fwd(x, w, 1, 1, 1, act="gelu")
    torch.cuda.synchronize()
    ref = oracle.conv3d(bits16(x), bits16(w), (1, 1, 1), (1, 1, 1), (1, 1, 1), act="gelu")
    assert_close(as_f64(y), ref, "gelu without bias")
    # relu of an all-negative output is exactly zero
    yn = pkg.conv_fwd(x, w, 1, 1, 1, act="relu",
                      bias=torch.full((272,), -1e4, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(yn.float()) == 0
    lib = pkg.load_library()
    out = torch.empty_like(y)
    rc = lib.conv_fwd_bias_act(x.data_ptr(), pkg._I64_5(*xs), w.data_ptr(), pkg._I64_5(*ws),
                               pkg._I32_3(1, 1, 1), pkg._I32_3(1, 1, 1), pkg._I32_3(1, 1, 1), 0,
                               None, None, None, 7, out.data_ptr(), None, 0, None)
    assert rc == pkg.CONV_ERR_INVALID


def test_bias_zero_weights_is_exact(pkg):
    """Zero weights: every output is bf16_rn(bias[k]) exactly."""
    x = cw.randn_bf16((1, 4, 6, 6, 32), 195, 1.0, "cuda")
    w = torch.zeros((48, 3, 3, 3, 32), dtype=torch.bfloat16, device="cuda")
    b = torch.linspace(-3.0, 3.0, 48, dtype=torch.float32, device="cuda")
    for split_k in (True, False):
        y = pkg.conv_fwd(x, w, 1, 1, 1, split_k=split_k, bias=b)
        torch.cuda.synchronize()
        assert torch.equal(y.float(), b.to(torch.bfloat16).float().expand_as(y))


# Non-overlapping patches (stride == filter, zero padding) that the implicit
# classes cannot read: RGB channels (6-byte rows), strides above the im2col
# limit; leftover rows / columns / frames past the last whole patch; a
# 3-D filter; odd patch lengths (2-byte gather).
PATCH_CASES = [
    ((2, 1, 32, 48, 3), (64, 1, 16, 16, 3), (1, 16, 16)),
    ((3, 1, 44, 30, 3), (40, 1, 14, 14, 3), (1, 14, 14)),
    ((2, 5, 32, 37, 3), (48, 2, 16, 16, 3), (2, 16, 16)),
    ((2, 1, 40, 40, 16), (72, 1, 10, 10, 16), (1, 10, 10)),
    ((1, 1, 20, 20, 16), (32, 1, 14, 14, 16), (1, 14, 14)),
    ((4, 1, 56, 56, 3), (96, 1, 7, 7, 3), (1, 7, 7)),
    ((2, 1, 224, 224, 3), (256, 1, 16, 16, 3), (1, 16, 16)),
]


@pytest.mark.parametrize("case", PATCH_CASES, ids=[str(i) for i in range(len(PATCH_CASES))])
def test_patch_gemm(pkg, case):
    xs, ws, st = case
    assert pkg.conv_fwd_plan(xs, ws, st, 0, 1)["class"] == "patch_gemm"
    _run_and_check(pkg, xs, ws, st, 0, 1, seed=200 + PATCH_CASES.index(case),
                   what=f"patch {case}")
    # also with a bias and without split-K (workspace holding the gather only)
    x, w = _inputs(xs, ws, 210 + PATCH_CASES.index(case))
    b = torch.linspace(-1.0, 1.0, ws[0], dtype=torch.float32, device="cuda")
    plan = pkg.conv_fwd_plan(xs, ws, st, 0, 1)
    y = pkg.conv_fwd(x, w, st, 0, 1, bias=b)
    torch.cuda.synchronize()
    ref = oracle.conv3d(bits16(x), bits16(w), st, (0, 0, 0), (1, 1, 1),
                        bias=b.double().cpu().numpy())
    assert_close(as_f64(y), ref, f"patch+bias {case} {plan}")


def test_patch_gemm_needs_workspace(pkg):
    x, w = _inputs((2, 1, 32, 48, 3), (64, 1, 16, 16, 3), 220)
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd(x, w, (1, 16, 16), 0, 1, split_k=False)
    assert e.value.status == pkg.CONV_ERR_INVALID
    assert "workspace" in str(e.value)


@pytest.mark.parametrize("case", [GENERIC[4], TEMPORAL[5], GENERIC[10]],
                         ids=["generic", "temporal", "generic256"])
@pytest.mark.parametrize("slices", [2, 3, 7])
def test_sliced_launches_are_bit_identical(pkg, case, slices):
    """The convolution cut into several launches of whole waves (the rule for
    long reductions, forced here on small shapes) computes every tile as one
    launch does: identical bits, and the oracle's values."""
    xs, ws, st, pa, di = case
    x, w = _inputs(xs, ws, 230)
    one = pkg.conv_fwd(x, w, st, pa, di, split_k=False)
    with pkg.overrides(slices=slices):
        sl = pkg.conv_fwd(x, w, st, pa, di, split_k=False)
        n = pkg.conv_fwd_kernel_launches(xs, ws, st, pa, di, 0, 0)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert 1 <= n <= slices
    assert torch.equal(one.view(torch.int16), sl.view(torch.int16))
    assert_close(as_f64(sl), oracle_conv(x, w, pkg._triple(st), pkg._triple(pa), pkg._triple(di)),
                 f"sliced {case}")


def test_kernel_launch_counts(pkg):
    tiny = cw.BY_NAME["tiny_conv3d_bf16"]
    p = pkg.conv_fwd_plan(tiny.x_shape, tiny.w_shape, tiny.stride, tiny.pad, tiny.dil)
    assert p["splits"] > 1
    assert pkg.conv_fwd_kernel_launches(tiny.x_shape, tiny.w_shape, tiny.stride, tiny.pad,
                                        tiny.dil, 0, p["workspace_bytes"]) == 2
    assert pkg.conv_fwd_kernel_launches(tiny.x_shape, tiny.w_shape, tiny.stride, tiny.pad,
                                        tiny.dil, 0, 0) == 1
    pe = cw.BY_NAME["patch_embed_bf16"]
    p = pkg.conv_fwd_plan(pe.x_shape, pe.w_shape, pe.stride, pe.pad, pe.dil)
    assert pkg.conv_fwd_kernel_launches(pe.x_shape, pe.w_shape, pe.stride, pe.pad, pe.dil, 0,
                                        p["workspace_bytes"]) == 2   # weight copies + GEMM
    # patch class: the patch gather (which also copies the weight rows to the
    # TMA pitch when they are not already a multiple of 16 bytes), the GEMM
    for name, n_expected in (("vit_patch16_bf16", 2), ("vit_patch14_bf16", 2)):
        v = cw.BY_NAME[name]
        p = pkg.conv_fwd_plan(v.x_shape, v.w_shape, v.stride, v.pad, v.dil)
        assert p["class"] == "patch_gemm"
        assert pkg.conv_fwd_kernel_launches(v.x_shape, v.w_shape, v.stride, v.pad, v.dil, 0,
                                            p["workspace_bytes"]) == n_expected, name
    video = cw.BY_NAME["video_conv3d_bf16"]
    n = pkg.conv_fwd_kernel_launches(video.x_shape, video.w_shape, video.stride, video.pad,
                                     video.dil, 0, 0)
    assert n > 4   # the long reduction runs in slices of whole waves


def test_launches_on_the_current_stream(pkg):
    """With no stream argument the kernels go to the caller's current stream:
    queued behind a ~50 ms spin on a side stream made current, the output is
    still untouched once the default stream has drained, and correct once
    the side stream has."""
    xs, ws = (2, 5, 9, 11, 64), (96, 3, 3, 3, 64)
    x = cw.randn_bf16(xs, 1200, 1.0, "cuda")
    w = cw.randn_bf16(ws, 1201, 1.0 / np.sqrt(27 * 64), "cuda")
    ref = pkg.conv_fwd(x, w, 1, 1, 1)
    out = torch.full(ref.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_t = torch.empty(max(16, pkg.conv_fwd_workspace_size(xs, ws, 1, 1, 1)), dtype=torch.uint8,
                       device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(100_000_000)            # ~50 ms of SM cycles on the side stream
        pkg.conv_fwd(x, w, 1, 1, 1, out=out, workspace=ws_t)
    torch.cuda.default_stream().synchronize()
    assert torch.isnan(out.float()).all(), "the conv did not wait for the side stream"
    side.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
