"""The C ABI library loads, exports every declared symbol, and its host-only
logic (output dims, dispatch class, plan, argument checks) is right.  No GPU:
no call here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from implicit_gemm_convolution_conv3d_gb300 import build as pkg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "conv3d.h")


@pytest.fixture(scope="module")
def pkg():
    pkg_build.build()
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\**\s+\**\s*([A-Za-z_]\w*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for must in ("conv_fwd", "pack_ncdhw_bf16_to_ndhwc", "pack_ncdhw_bf16_to_ndhwc_fp8",
                 "conv_out_dims", "conv_fwd_plan", "conv_get_device_status",
                 "conv_fwd_from_host"):
        assert must in names


def test_workspace_size_without_a_gpu_is_zero_with_a_reason(pkg):
    """conv_fwd_workspace_size plans for the current device: with no GPU it
    answers 0 and leaves the reason in conv_last_error (no launch, no fault)."""
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests compare the size with conv_fwd_plan")
    lib = pkg.load_library()
    i64, i32 = ctypes.c_int64 * 5, ctypes.c_int * 3
    n = lib.conv_fwd_workspace_size(i64(1, 4, 8, 8, 16), i64(32, 3, 3, 3, 16), i32(1, 1, 1),
                                    i32(1, 1, 1), i32(1, 1, 1), 0)
    assert n == 0
    assert lib.conv_last_error().decode() != ""


def test_library_exports_every_declared_symbol(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_out_dims_match_oracle(pkg):
    rng = np.random.default_rng(0)
    for _ in range(200):
        xs = [int(v) for v in rng.integers(1, 20, size=5)]
        ws = [int(v) for v in rng.integers(1, 5, size=5)]
        ws[4] = xs[4]
        st = [int(v) for v in rng.integers(1, 4, size=3)]
        pa = [int(v) for v in rng.integers(0, 3, size=3)]
        di = [int(v) for v in rng.integers(1, 3, size=3)]
        ref = oracle.out_dims(xs, ws, st, pa, di)
        if min(ref) <= 0:
            with pytest.raises(pkg.ConvError):
                pkg.conv_out_dims(xs, ws, st, pa, di)
        else:
            assert pkg.conv_out_dims(xs, ws, st, pa, di) == tuple(ref)


def test_plan_classifies_the_workloads(pkg):
    import conv_workloads as cw
    sms = 148
    p = pkg.conv_fwd_plan((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 1, 1, 1, 0, sms)
    assert p["class"] == "generic" and p["splits"] > 1 and p["workspace_bytes"] > 0
    p = pkg.conv_fwd_plan((9500, 1, 14, 14, 3), (1280, 1, 14, 14, 3), (1, 14, 14), 0, 1, 0, sms)
    assert p["class"] == "point_gemm" and p["splits"] == 1
    p = pkg.conv_fwd_plan((1, 15, 120, 120, 2048), (2048, 3, 3, 3, 2048), 1, 1, 1, 0, sms)
    assert p["class"] == "generic" and p["splits"] == 1 and p["ctas"] == sms
    p = pkg.conv_fwd_plan((1, 120, 160, 90, 1024), (1024, 1, 3, 3, 1024), 1, (0, 1, 1), 1, 1, sms)
    assert p["class"] == "generic" and p["k_bytes"] == 256   # tile-table row: 256-byte k-steps
    p = pkg.conv_fwd_plan((1, 240, 160, 90, 640), (640, 3, 1, 1, 640), 1, (1, 0, 0), 1, 0, sms)
    assert p["class"] == "temporal" and p["k_bytes"] == 256
    # pointwise 1x1x1 conv is a plain GEMM too
    p = pkg.conv_fwd_plan((2, 3, 4, 5, 64), (32, 1, 1, 1, 64), 1, 0, 1, 0, sms)
    assert p["class"] == "point_gemm"
    # input spatial in (filter, 2*filter-1] with stride == filter: rows are not contiguous
    p = pkg.conv_fwd_plan((8, 5, 5, 5, 16), (32, 4, 4, 4, 16), 4, 0, 1, 0, sms)
    assert p["class"] == "generic"
    # the im2col traversal stride is at most 8; non-overlapping patches beyond
    # it (stride == filter) are gathered into GEMM rows instead
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_plan((4, 1, 20, 20, 16), (32, 1, 3, 3, 16), (1, 14, 14), 0, 1, 0, sms)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    p = pkg.conv_fwd_plan((4, 1, 20, 20, 16), (32, 1, 14, 14, 16), (1, 14, 14), 0, 1, 0, sms)
    assert p["class"] == "patch_gemm" and p["workspace_bytes"] > 0
    # ViT-style patch embeddings: 16x16 and 14x14 patches of RGB images
    for k in (16, 14):
        p = pkg.conv_fwd_plan((8, 1, 224, 224, 3), (768, 1, k, k, 3), (1, k, k), 0, 1, 0, sms)
        assert p["class"] == "patch_gemm"
        # gathered rows at a 16-byte pitch; weight rows that already are a
        # multiple of 16 bytes (16*16*3 bf16 = 1536) are read in place, the
        # 14*14*3 ones (1176 bytes) are copied to the 1184-byte pitch after them
        m, row = 8 * (224 // k) ** 2, k * k * 3 * 2
        pitch = (row + 15) // 16 * 16
        up = lambda b: (b + 255) // 256 * 256
        need = up(m * pitch) + (0 if row == pitch else up(768 * pitch))
        if p["splits"] > 1:   # fp32 partials [splits, M, K] after the copies
            need += p["splits"] * m * 768 * 4
        assert p["workspace_bytes"] == need, (k, p["workspace_bytes"], need)
    assert {w.name for w in cw.WORKLOADS} >= {"tiny_conv3d_bf16", "video_conv3d_bf16"}


def test_plan_tiles_are_legal(pkg):
    rng = np.random.default_rng(1)
    for _ in range(300):
        C = int(rng.choice([8, 16, 24, 32, 64, 96, 136, 256, 1024]))
        K = int(rng.integers(1, 600))
        xs = (int(rng.integers(1, 3)), int(rng.integers(1, 9)), int(rng.integers(1, 17)),
              int(rng.integers(1, 17)), C)
        ws = (K, int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(1, 4)), C)
        pa = [int(rng.integers(0, 2)) for _ in range(3)]
        try:
            pkg.conv_out_dims(xs, ws, 1, pa, 1)
        except pkg.ConvError:
            continue
        for dt in (0, 1):
            try:
                p = pkg.conv_fwd_plan(xs, ws, 1, pa, 1, dt, 148)
            except pkg.ConvError as e:
                # only the fp8 implicit GEMM with C % 16 != 0 is outside coverage
                assert dt == 1 and C % 16 != 0 and e.status == pkg.CONV_ERR_UNSUPPORTED
                continue
            assert p["tile_n"] % 32 == 0 and 32 <= p["tile_n"] <= 256
            assert p["k_bytes"] in (32, 64, 128, 256)
            assert 2 <= p["stages"] <= 8
            assert (p["tile_n"] * p["k_bytes"] + 128 * p["k_bytes"]) * p["stages"] + 1280 <= 232448
            assert 1 <= p["ctas"] <= 148


def test_forced_wide_k_step_plans(pkg):
    """256-byte k-steps: accepted for every TMA operand mode, the reduction is
    cut into ceil(row bytes / 256) chunks, and the pipeline fits in shared
    memory; other k-step widths are rejected as invalid overrides."""
    sms = 148
    with pkg.overrides(tile="128,256,0,1,1"):
        plans = [(pkg.conv_fwd_plan(xs, ws, st, pa, 1, 0, sms), cls) for xs, ws, st, pa, cls in [((1, 6, 10, 12, 200), (96, 3, 3, 3, 200), 1, 1, "generic"),
                                ((1, 5, 10, 50, 200), (200, 3, 1, 1, 200), 1, (1, 0, 0), "temporal"),
                                ((600, 1, 4, 4, 16), (160, 1, 4, 4, 16), (1, 4, 4), 0, "point_gemm")]]
    for p, cls in plans:
        assert p["class"] == cls and p["k_bytes"] == 256 and p["stages"] >= 2
        assert (128 * 256 + 128 * 256) * p["stages"] + 1280 <= 232448
    with pytest.raises(pkg.ConvError) as e:
        with pkg.overrides(tile="128,512,0,1,1"):
            pass
    assert e.value.status == pkg.CONV_ERR_INVALID
    # a rejected set leaves the previous overrides (none) in place
    assert pkg.conv_fwd_plan((1, 6, 10, 12, 200), (96, 3, 3, 3, 200), 1, 1, 1, 0, sms)["k_bytes"] != 256


def test_invalid_and_unsupported_arguments(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3
    args = (I5(1, 4, 8, 8, 16), None, I5(32, 3, 3, 3, 16), I3(1, 1, 1), I3(1, 1, 1), I3(1, 1, 1))
    rc = lib.conv_fwd(None, args[0], None, args[2], args[3], args[4], args[5], 0, None, None,
                      None, None, ctypes.c_size_t(0), None)
    assert rc == pkg.CONV_ERR_INVALID
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_out_dims((1, 4, 8, 8, 16), (32, 3, 3, 3, 8), 1, 1, 1)
    assert e.value.status == pkg.CONV_ERR_INVALID
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_plan((1, 4, 8, 8, 12), (32, 3, 3, 3, 12), 1, 1, 1, 0, 148)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_plan((1, 4, 8, 8, 16), (32, 3, 3, 3, 16), 1, 1, 1, 7, 148)
    assert e.value.status == pkg.CONV_ERR_INVALID
    rc = lib.pack_ncdhw_bf16_to_ndhwc(None, I5(1, 2, 3, 4, 5), None, None)
    assert rc == pkg.CONV_ERR_INVALID
    # an unknown activation code, and null tensors with a valid one: both
    # rejected before any device work
    for act in (-1, 4, 99, 1):
        rc = lib.conv_fwd_bias_act(None, args[0], None, args[2], args[3], args[4], args[5], 0,
                                   None, None, None, act, None, None, ctypes.c_size_t(0), None)
        assert rc == pkg.CONV_ERR_INVALID, act
    with pytest.raises(ValueError):
        pkg.conv_fwd(torch.zeros(1), torch.zeros(1), act="tanh")
    rc = lib.conv_fwd_ncdhw(None, I5(1, 16, 4, 8, 8), None, I5(32, 3, 1, 1, 16), args[3],
                            I3(1, 0, 0), args[5], 0, None, None, None, None, None,
                            ctypes.c_size_t(0), None)
    assert rc == pkg.CONV_ERR_INVALID
    lib.conv_status_string.restype = ctypes.c_char_p
    for s in range(5):
        assert lib.conv_status_string(s).startswith(b"CONV_")


def test_from_host_argument_checks(pkg):
    """conv_fwd_from_host rejects null operands, a negative slice count and
    misaligned device buffers before touching the device."""
    lib = ctypes.CDLL(pkg.LIB_PATH)
    lib.conv_fwd_from_host.restype = ctypes.c_int
    I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3
    xd, wd, st = I5(1, 4, 8, 8, 16), I5(32, 3, 3, 3, 16), I3(1, 1, 1)
    host = (ctypes.c_uint8 * 64)()
    hp = ctypes.cast(host, ctypes.c_void_p)
    good, odd = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 8)

    def call(x_host, x_dev, chunks):
        return lib.conv_fwd_from_host(x_host, xd, hp, wd, st, st, st, 0, None, None, hp, x_dev,
                                      good, good, None, ctypes.c_size_t(0), chunks, None)

    assert call(None, good, 0) == pkg.CONV_ERR_INVALID
    assert call(hp, None, 0) == pkg.CONV_ERR_INVALID
    assert call(hp, good, -1) == pkg.CONV_ERR_INVALID
    assert call(hp, odd, 0) == pkg.CONV_ERR_INVALID


def test_backward_argument_checks(pkg):
    """The point-output backward entry points reject null operands, misaligned
    buffers and non-point-output shapes before touching the device."""
    lib = ctypes.CDLL(pkg.LIB_PATH)
    I5, I3 = ctypes.c_int64 * 5, ctypes.c_int * 3
    pt_x, pt_w, st = I5(4, 1, 4, 4, 8), I5(8, 1, 4, 4, 8), I3(1, 4, 4)
    zero, one = I3(0, 0, 0), I3(1, 1, 1)
    a, b = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20)
    for fn in (lib.conv_bwd_data_point, lib.conv_bwd_weight_point):
        fn.restype = ctypes.c_int
        assert fn(None, b, pt_x, pt_w, st, zero, one, a, a, ctypes.c_size_t(0), None) == \
            pkg.CONV_ERR_INVALID
        assert fn(a, b, pt_x, pt_w, st, zero, one, ctypes.c_void_p((1 << 20) + 4), a,
                  ctypes.c_size_t(0), None) == pkg.CONV_ERR_INVALID
        # a 3x3 filter over an 8x8 input has many output positions
        assert fn(a, b, I5(2, 1, 8, 8, 16), I5(32, 1, 3, 3, 16), one, zero, one, a, a,
                  ctypes.c_size_t(1 << 20), None) == pkg.CONV_ERR_UNSUPPORTED


def test_ncdhw_plan_coverage(pkg):
    """conv_fwd_ncdhw plans: always the temporal class with 128- or 256-byte
    k-steps (MN-major boxes of 64 channel rows); T x 1 x 1 filters only,
    bf16 only, H*W and C multiples of 8."""
    sms = 148
    p = pkg.conv_fwd_ncdhw_plan((1, 640, 240, 160, 90), (640, 3, 1, 1, 640), 1, (1, 0, 0), 1, 0, sms)
    assert p["class"] == "temporal" and p["k_bytes"] == 256 and p["splits"] == 1
    # 6.9 MB channel planes read by three taps: packed to an NDHWC copy in the workspace
    assert p["workspace_bytes"] >= 640 * 240 * 160 * 90 * 2
    # 0.46 MB channel planes: read in place, no workspace
    p = pkg.conv_fwd_ncdhw_plan((1, 640, 16, 160, 90), (640, 3, 1, 1, 640), 1, (1, 0, 0), 1, 0, sms)
    assert p["workspace_bytes"] == 0
    # the pointwise conv stays in the temporal class (its NDHWC form is a GEMM)
    p = pkg.conv_fwd_ncdhw_plan((2, 64, 3, 4, 6), (32, 1, 1, 1, 64), 1, 0, 1, 0, sms)
    assert p["class"] == "temporal" and p["k_bytes"] >= 128
    assert pkg.conv_fwd_plan((2, 3, 4, 6, 64), (32, 1, 1, 1, 64), 1, 0, 1, 0, sms)["class"] == \
        "point_gemm"
    # narrow channel rows still take 128-byte k-steps (channels past C read zero)
    p = pkg.conv_fwd_ncdhw_plan((1, 8, 5, 4, 4), (16, 2, 1, 1, 8), (2, 1, 1), (1, 0, 0), (2, 1, 1),
                                0, sms)
    assert p["class"] == "temporal" and p["k_bytes"] == 128
    bad = [
        ((1, 64, 4, 8, 8), (32, 1, 3, 3, 64), 1, (0, 1, 1), 0),    # spatial taps
        ((1, 64, 4, 8, 8), (32, 3, 1, 1, 64), (1, 2, 2), (1, 0, 0), 0),   # H/W stride
        ((1, 64, 4, 5, 5), (32, 3, 1, 1, 64), 1, (1, 0, 0), 0),    # H*W = 25
        ((1, 60, 4, 8, 8), (32, 3, 1, 1, 60), 1, (1, 0, 0), 0),    # C % 8 != 0
        ((1, 64, 4, 8, 8), (32, 3, 1, 1, 64), 1, (1, 0, 0), 1),    # fp8
    ]
    for xs, ws, st, pa, dt in bad:
        with pytest.raises(pkg.ConvError) as e:
            pkg.conv_fwd_ncdhw_plan(xs, ws, st, pa, 1, dt, sms)
        assert e.value.status == pkg.CONV_ERR_UNSUPPORTED, (xs, ws)
    with pytest.raises(pkg.ConvError) as e:   # C of x (dim 1) against w
        pkg.conv_fwd_ncdhw_plan((1, 64, 4, 8, 8), (32, 3, 1, 1, 32), 1, 0, 1, 0, sms)
    assert e.value.status == pkg.CONV_ERR_INVALID


def test_forward_shape_cache(pkg):
    """The binding computes a problem's output dims and marshalled shape
    arguments once: the same shapes and conv parameters return the same
    entry, any difference a new one, and installing overrides (which can
    change plans and so workspace sizes) empties the cache."""
    x = torch.empty((2, 5, 9, 11, 64), dtype=torch.bfloat16)
    w = torch.empty((96, 3, 3, 3, 64), dtype=torch.bfloat16)
    e1 = pkg._fwd_shape(x, w, 1, 1, 1, 0)
    assert e1 is pkg._fwd_shape(x, w, (1, 1, 1), [1, 1, 1], 1, 0)
    assert e1.od == pkg.conv_out_dims(tuple(x.shape), tuple(w.shape), 1, 1, 1) == (2, 5, 9, 11, 96)
    assert tuple(e1.xd) == tuple(x.shape) and tuple(e1.wd) == tuple(w.shape)
    e2 = pkg._fwd_shape(x, w, 2, 1, 1, 0)
    assert e2 is not e1 and e2.od == (2, 3, 5, 6, 96)
    assert pkg._fwd_shape(x, w, 1, 1, 1, 1) is not e1          # dtype is part of the key
    assert pkg._fwd_shape(x, w, 1, 1, 1, 0) is e1
    try:
        pkg.set_overrides(stages=3)
        assert pkg._fwd_shape(x, w, 1, 1, 1, 0) is not e1
    finally:
        pkg.set_overrides()
    assert pkg._fwd_shape(x, w, 1, 1, 1, 0) is not e1   # cleared again by the reset
