"""Parity at the full sizes of the measured workloads, in the launch
configuration the benchmark times.

The fp64 oracle cannot evaluate 10^13-flop convolutions whole, so outputs are
checked on >= 1M uniformly sampled output elements plus forced samples: every
spatial corner and face centre, the first and last M tile, the last N tile,
and for the >2^31-element temporal workload at least 10k samples past flat
index 2^31 (byte offset 2^32).  The small workloads (tiny conv, patch
embedding) are checked in full.  The fp8 workload's pack is checked byte for
byte over the whole tensor."""
import os

import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, bits16, bytes8

pytestmark = pytest.mark.gpu

N_SAMPLES = int(os.environ.get("CONV3D_PARITY_SAMPLES", "1000000"))


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def _forced_indices(od, tile_n, rng):
    N, Do, Ho, Wo, K = od
    M = N * Do * Ho * Wo
    pts = []
    for n in {0, N - 1}:
        for d in {0, Do // 2, Do - 1}:
            for h in {0, Ho // 2, Ho - 1}:
                for w in {0, Wo // 2, Wo - 1}:
                    m = ((n * Do + d) * Ho + h) * Wo + w
                    pts.extend(m * K + rng.integers(0, K, size=8))
    for m in list(range(min(128, M))) + list(range(max(0, M - 128), M)):
        pts.extend(m * K + rng.integers(0, K, size=2))
    last_n0 = ((K - 1) // tile_n) * tile_n
    rows = rng.integers(0, M, size=2000)
    pts.extend(rows * K + rng.integers(last_n0, K, size=rows.size))
    return np.asarray(pts, dtype=np.int64)


def _sample(od, wl, tile_n):
    total = int(np.prod(od))
    idx = cw.sample_indices(total, N_SAMPLES, wl.sample_seed).numpy()
    rng = np.random.default_rng(wl.sample_seed)
    idx = np.concatenate([idx, _forced_indices(od, tile_n, rng)])
    if total > 2 ** 31:
        hi = rng.integers(2 ** 31, total, size=10000)
        idx = np.concatenate([idx, hi])
        assert (idx > 2 ** 31).sum() >= 10000
    return idx


def _check_sampled(y, x_host, w_host, idx, wl, scale_x=1.0, scale_w=1.0):
    got = y.view(-1)[torch.from_numpy(idx).cuda()].float().cpu().double().numpy()
    ref = oracle.conv3d_points(x_host, w_host, idx, wl.stride, wl.pad, wl.dil, scale_x, scale_w)
    assert_close(got, ref, wl.name)


def test_patch_embed_full(pkg):
    wl = cw.BY_NAME["patch_embed_bf16"]
    x, w = cw.make_inputs(wl, "cuda")
    y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d(bits16(x), bits16(w), wl.stride, wl.pad, wl.dil)
    assert_close(as_f64(y), ref, wl.name)


def test_video_conv3d_sampled(pkg):
    wl = cw.BY_NAME["video_conv3d_bf16"]
    x, w = cw.make_inputs(wl, "cuda")
    y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    plan = pkg.conv_fwd_plan(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil)
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    _check_sampled(y, bits16(x), bits16(w), idx, wl)


def test_video_conv3d_from_host_full_size(pkg):
    """The measured end-to-end path at the headline size: conv_fwd_from_host
    with its default slicing (whole-wave slices, the first split over weight
    groups) from pinned host operands equals conv_fwd bit for bit over the
    whole output, and the oracle on >= 1M sampled outputs."""
    wl = cw.BY_NAME["video_conv3d_bf16"]
    x, w = cw.make_inputs(wl, "cuda")
    y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil)
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    wh = torch.empty(w.shape, dtype=w.dtype, pin_memory=True)
    xh.copy_(x)
    wh.copy_(w)
    hout = torch.empty(y.shape, dtype=torch.bfloat16, pin_memory=True)
    hout.fill_(float("nan"))
    # NaN bytes in the device buffers: input rows or weights read before
    # their copy landed would show as NaN outputs
    xd, wd = torch.empty_like(x), torch.empty_like(w)
    xd.view(torch.uint8).fill_(0xFF)
    wd.view(torch.uint8).fill_(0xFF)
    outd = torch.full(y.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    pkg.conv_fwd_from_host(xh, wh, wl.stride, wl.pad, wl.dil, out_host=hout, x_dev=xd,
                           w_dev=wd, out_dev=outd)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert torch.equal(xd.view(torch.int16), x.view(torch.int16))
    assert torch.equal(wd.view(torch.int16), w.view(torch.int16))
    assert torch.equal(hout.view(torch.int16), y.cpu().view(torch.int16))
    plan = pkg.conv_fwd_plan(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil)
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    got = hout.view(-1)[torch.from_numpy(idx)].float().double().numpy()
    ref = oracle.conv3d_points(bits16(x), bits16(w), idx, wl.stride, wl.pad, wl.dil)
    assert_close(got, ref, "video_conv3d_bf16 from host")


def test_fp8_workload_pack_exact_and_conv_sampled(pkg):
    wl = cw.BY_NAME["fp8_conv3d_1x3x3"]
    x, w = cw.make_inputs(wl, "cuda")          # bf16 NCDHW, bf16 KCTRS
    qx, sx = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
    qw, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(w)
    torch.cuda.synchronize()
    xh = bits16(x)
    ref_qx, ref_sx = oracle.pack_ncdhw_to_ndhwc_fp8(xh)
    del xh
    qx_h = bytes8(qx)
    assert np.float32(sx.item()).tobytes() == np.float32(ref_sx).tobytes()
    assert np.array_equal(qx_h, ref_qx)
    del ref_qx
    ref_qw, ref_sw = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(w))
    qw_h = bytes8(qw)
    assert sw.item() == ref_sw and np.array_equal(qw_h, ref_qw)
    y = pkg.conv_fwd(qx, qw, wl.stride, wl.pad, wl.dil, scale_x=sx, scale_w=sw)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    plan = pkg.conv_fwd_plan(tuple(qx.shape), tuple(qw.shape), wl.stride, wl.pad, wl.dil, 1)
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    _check_sampled(y, qx_h, qw_h, idx, wl, sx.item(), sw.item())
    # the same conv with the activation quantised while it is loaded (no
    # pack pass): the scale's bits and the sampled outputs against the
    # oracle's pack and conv
    del y, qx
    torch.cuda.empty_cache()
    yf, sxf = pkg.conv_fwd_ncdhw_fp8(x, qw, wl.stride, wl.pad, wl.dil, scale_w=sw)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert np.float32(sxf.item()).tobytes() == np.float32(ref_sx).tobytes()
    _check_sampled(yf, qx_h, qw_h, idx, wl, sxf.item(), sw.item())


def test_temporal_big_sampled(pkg):
    wl = cw.BY_NAME["temporal_3x1x1_bf16_big"]
    x, w = cw.make_inputs(wl, "cuda")
    assert x.numel() > 2 ** 31
    y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert y.numel() > 2 ** 31
    plan = pkg.conv_fwd_plan(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil)
    assert plan["class"] == "temporal"
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    _check_sampled(y, bits16(x), bits16(w), idx, wl)


@pytest.mark.parametrize("name", ["temporal_3x1x1_bf16_ncdhw", "pointwise_1x1x1_bf16_ncdhw"])
def test_channel_major_sampled(pkg, name):
    """conv_fwd_ncdhw at full size on channel-major activations: the temporal
    workload (2.2e9 elements, 64-bit offsets) and the 14 GB pointwise conv,
    against the oracle reading the same NCDHW bytes."""
    wl = cw.BY_NAME[name]
    x, w = cw.make_inputs(wl, "cuda")
    y = pkg.conv_fwd_ncdhw(x, w, wl.stride, wl.pad, wl.dil)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    plan = pkg.conv_fwd_ncdhw_plan(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil)
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    got = y.view(-1)[torch.from_numpy(idx).cuda()].float().cpu().double().numpy()
    del y
    xb, wb = bits16(x), bits16(w)
    del x
    torch.cuda.empty_cache()
    ref = oracle.conv3d_points(xb, wb, idx, wl.stride, wl.pad, wl.dil, x_layout="ncdhw")
    assert_close(got, ref, wl.name)


@pytest.mark.parametrize("name", ["vit_patch16_bf16", "vit_patch14_bf16"])
def test_vit_patch_embed_sampled(pkg, name):
    """Patch embeddings with 196 / 256 patches per image, at full size: the
    gathered-patch GEMM, sampled like the other large workloads."""
    wl = cw.BY_NAME[name]
    x, w = cw.make_inputs(wl, "cuda")
    plan = pkg.conv_fwd_plan(wl.x_shape, wl.w_shape, wl.stride, wl.pad, wl.dil)
    assert plan["class"] == "patch_gemm"
    y = pkg.conv_fwd(x, w, wl.stride, wl.pad, wl.dil)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    idx = _sample(tuple(y.shape), wl, plan["tile_n"])
    _check_sampled(y, bits16(x), bits16(w), idx, wl)
