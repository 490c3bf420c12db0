"""GPU parity of the NCDHW -> NDHWC pack (bf16 copy and fp8-e4m3 quantisation)
and of the fp8 forward convolution.

The pack must equal the oracle bit for bit: every output byte and the scale's
bits.  The codec is exercised exhaustively: every finite bf16 pattern below a
chosen amax, at several amax values.  The fp8 conv is compared with the
oracle's conv of the very bytes the GPU pack produced (the fp8-cast conv
reference), times both scales."""
import os

import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, bits16, bytes8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


# C % 16 == 0 and D*H*W % 8 == 0 take the register-blocked tile kernel (with
# partial 64-channel / 64-position tiles here); the others the generic one.
PACK_SHAPES = [(1, 16, 2, 3, 8), (2, 64, 3, 5, 7), (1, 100, 1, 9, 13), (3, 24, 2, 8, 8),
               (1, 1024, 2, 16, 9), (1, 8, 1, 1, 1), (2, 130, 3, 3, 11), (2, 80, 3, 5, 8),
               (1, 48, 1, 1, 24), (3, 176, 2, 7, 4)]


@pytest.mark.parametrize("shape", PACK_SHAPES)
def test_pack_bf16_bit_exact(pkg, shape):
    x = cw.randn_bf16(shape, 300, 1.0, "cuda")
    y = pkg.pack_ncdhw_bf16_to_ndhwc(x)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(y), oracle.pack_ncdhw_to_ndhwc_bf16(bits16(x)))


@pytest.mark.parametrize("shape", PACK_SHAPES)
def test_pack_fp8_bit_exact(pkg, shape):
    x = cw.randn_bf16(shape, 301, 3.0, "cuda")
    q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(x))
    assert np.float32(s.item()).tobytes() == np.float32(ref_s).tobytes()
    assert np.array_equal(bytes8(q), ref_q)


@pytest.mark.parametrize("amax", [448.0, 1.0, 3.0, 1e-3, 2.0 ** -7, 6.5e4, 1.7e38])
def test_pack_fp8_codec_exhaustive(pkg, amax):
    """All finite bf16 patterns with |v| <= amax (amax itself included) packed
    as one tensor: the device cvt.rn.satfinite path against the oracle's
    nearest-code search, byte for byte."""
    pats = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    keep = np.isfinite(pats) & (np.abs(pats) <= np.float32(amax))
    vals = pats[keep]
    amax_bf16 = np.float32(torch.tensor(amax).to(torch.bfloat16).float().item())
    vals = np.concatenate([vals, np.array([amax_bf16, -amax_bf16], dtype=np.float32)])
    n = vals.size
    C = 16
    S = (n + C - 1) // C
    flat = np.zeros(S * C, dtype=np.float32)
    flat[:n] = vals
    xb = torch.from_numpy(flat).to(torch.bfloat16).view(1, C, 1, 1, S).cuda()
    q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(xb)
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(xb))
    assert np.float32(s.item()).tobytes() == np.float32(ref_s).tobytes()
    assert np.array_equal(bytes8(q), ref_q)


@pytest.mark.parametrize("amax", [448.0, 3.0, 1e-3, 2.0 ** -7, 1.7e38])
def test_pack_fp8_codec_exhaustive_both_kernels(pkg, amax):
    """The same exhaustive patterns in a 128-channel tensor whose position
    count is a multiple of 8: the TMA-fed pack and the register-blocked pack
    (the pack_lanes override) each equal the oracle byte for byte."""
    pats = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = pats[np.isfinite(pats) & (np.abs(pats) <= np.float32(amax))]
    amax_bf16 = np.float32(torch.tensor(amax).to(torch.bfloat16).float().item())
    vals = np.concatenate([vals, np.array([amax_bf16, -amax_bf16], dtype=np.float32)])
    C = 128
    S = (vals.size + C - 1) // C
    S = (S + 7) // 8 * 8
    flat = np.zeros(S * C, dtype=np.float32)
    flat[:vals.size] = np.random.default_rng(5).permutation(vals)
    xb = torch.from_numpy(flat).to(torch.bfloat16).view(1, C, 1, 1, S).cuda()
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(xb))
    for lanes in (None, 2):
        with pkg.overrides(pack_lanes=lanes):
            q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(xb)
            torch.cuda.synchronize()
        assert np.float32(s.item()).tobytes() == np.float32(ref_s).tobytes()
        assert np.array_equal(bytes8(q), ref_q), f"pack_lanes={lanes}"


_AMAX_SWEEP = [float(v) for v in np.exp(np.random.default_rng(41).uniform(np.log(1e-30),
                                                                          np.log(1e30), 40))]


@pytest.mark.parametrize("amax", _AMAX_SWEEP, ids=[f"{a:.3g}" for a in _AMAX_SWEEP])
def test_pack_fp8_codec_many_scales(pkg, amax):
    """Every finite bf16 pattern up to amax, for 40 seeded amax values over 60
    decades: the default (TMA-fed) pack's codes, whatever quotient it uses,
    equal the oracle's division byte for byte."""
    pats = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    amax_bf16 = np.float32(torch.tensor(amax).to(torch.bfloat16).float().item())
    vals = pats[np.isfinite(pats) & (np.abs(pats) <= amax_bf16)]
    vals = np.concatenate([vals, np.array([amax_bf16, -amax_bf16], dtype=np.float32)])
    C = 64
    S = ((vals.size + C - 1) // C + 7) // 8 * 8
    flat = np.zeros(S * C, dtype=np.float32)
    flat[:vals.size] = vals
    xb = torch.from_numpy(flat).to(torch.bfloat16).view(1, C, 1, 1, S).cuda()
    q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(xb)
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(xb))
    assert np.float32(s.item()).tobytes() == np.float32(ref_s).tobytes()
    assert np.array_equal(bytes8(q), ref_q)


@pytest.mark.parametrize("shape", [(2, 200, 3, 17, 24), (1, 1024, 3, 40, 90), (3, 8, 1, 1, 8),
                                   (1, 136, 2, 1, 260)])
def test_pack_tma_partial_tiles(pkg, shape):
    """Tensors whose channels and positions leave partial TMA tiles (200 of 128
    / 64 channels, 1224 of 256 positions, one 8-channel tile, 520 positions):
    both packs equal the oracle."""
    x = cw.randn_bf16(shape, 302, 2.0, "cuda")
    ref_b = oracle.pack_ncdhw_to_ndhwc_bf16(bits16(x))
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(x))
    y = pkg.pack_ncdhw_bf16_to_ndhwc(x)
    q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(y), ref_b)
    assert np.float32(s.item()).tobytes() == np.float32(ref_s).tobytes()
    assert np.array_equal(bytes8(q), ref_q)


def test_pack_fp8_all_zero_tensor(pkg):
    x = torch.zeros((1, 32, 2, 2, 2), dtype=torch.bfloat16, device="cuda")
    q, s = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
    torch.cuda.synchronize()
    assert s.item() == 1.0 and not bytes8(q).any()


def _fp8_operands(pkg, x_ncdhw, w_kctrs):
    qx, sx = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x_ncdhw)
    qw, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(w_kctrs)
    torch.cuda.synchronize()
    # the pack is itself checked against the oracle before the conv is
    ref_qx, ref_sx = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(x_ncdhw))
    ref_qw, ref_sw = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(w_kctrs))
    assert np.array_equal(bytes8(qx), ref_qx) and np.array_equal(bytes8(qw), ref_qw)
    assert sx.item() == ref_sx and sw.item() == ref_sw
    return qx, sx, qw, sw


FP8_CASES = [
    # (x NCDHW, w KCTRS, stride, pad, dil, class)
    ((1, 64, 4, 9, 11), (96, 64, 1, 3, 3), 1, (0, 1, 1), 1, "generic"),
    ((2, 32, 5, 7, 6), (48, 32, 3, 3, 3), 1, 1, 1, "generic"),
    ((1, 144, 3, 10, 12), (272, 144, 1, 3, 3), (1, 2, 1), (0, 1, 1), 1, "generic"),
    ((1, 16, 6, 8, 16), (32, 16, 3, 1, 1), 1, (1, 0, 0), 1, "temporal"),
    ((1, 128, 5, 12, 20), (160, 128, 3, 1, 1), 1, (1, 0, 0), 1, "temporal"),
    ((40, 3, 1, 16, 16), (64, 3, 1, 16, 16), (1, 16, 16), 0, 1, "point_gemm"),
    ((70, 3, 1, 14, 14), (96, 3, 1, 14, 14), (1, 14, 14), 0, 1, "point_gemm"),
    ((2, 64, 2, 3, 5), (40, 64, 1, 1, 1), 1, 0, 1, "point_gemm"),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[str(i) for i in range(len(FP8_CASES))])
@pytest.mark.parametrize("split_k", [True, False])
def test_fp8_conv(pkg, case, split_k):
    xs, ws, st, pa, di, cls = case
    crs = ws[1] * ws[2] * ws[3] * ws[4]
    x = cw.randn_bf16(xs, 400 + FP8_CASES.index(case), 1.0, "cuda")
    w = cw.randn_bf16(ws, 500 + FP8_CASES.index(case), 1.0 / np.sqrt(crs), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    assert pkg.conv_fwd_plan(tuple(qx.shape), tuple(qw.shape), st, pa, di, 1)["class"] == cls
    y = pkg.conv_fwd(qx, qw, st, pa, di, scale_x=sx, scale_w=sw, split_k=split_k)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d(bytes8(qx), bytes8(qw), pkg._triple(st), pkg._triple(pa), pkg._triple(di),
                        sx.item(), sw.item())
    assert_close(as_f64(y), ref, f"fp8 {case} split={split_k}")


@pytest.mark.parametrize("case", FP8_CASES, ids=[str(i) for i in range(len(FP8_CASES))])
@pytest.mark.parametrize("plan", [(0, "128,256,0,0,1"), (1, "256,256,0,0,1")],
                         ids=["single", "pair"])
def test_fp8_conv_wide_k_steps(pkg, case, plan):
    """256-byte k-steps (two 128-byte boxes per operand) on the fp8 shapes,
    whose channel rows end inside the first or second box."""
    pair, spec = plan
    xs, ws, st, pa, di, cls = case
    crs = ws[1] * ws[2] * ws[3] * ws[4]
    x = cw.randn_bf16(xs, 400 + FP8_CASES.index(case), 1.0, "cuda")
    w = cw.randn_bf16(ws, 500 + FP8_CASES.index(case), 1.0 / np.sqrt(crs), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    with pkg.overrides(tile=spec, pair=pair):
        assert pkg.conv_fwd_plan(tuple(qx.shape), tuple(qw.shape), st, pa, di, 1)["k_bytes"] == 256
        y = pkg.conv_fwd(qx, qw, st, pa, di, scale_x=sx, scale_w=sw)
        torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d(bytes8(qx), bytes8(qw), pkg._triple(st), pkg._triple(pa), pkg._triple(di),
                        sx.item(), sw.item())
    assert_close(as_f64(y), ref, f"fp8 bk256 pair={pair} {case}")


def test_fp8_point_gemm_two_phases(pkg):
    """fp8 point-output GEMM with 24-byte rows (8 past a 16-byte multiple):
    the two-phase path over the packed activation."""
    xs, ws = (333, 6, 1, 2, 2), (48, 6, 1, 2, 2)   # NCDHW / KCTRS: 24 elements per row
    x = cw.randn_bf16(xs, 420, 1.0, "cuda")
    w = cw.randn_bf16(ws, 520, 1.0 / np.sqrt(24), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    plan = pkg.conv_fwd_plan(tuple(qx.shape), tuple(qw.shape), (1, 2, 2), 0, 1, 1)
    assert plan["class"] == "point_gemm"
    y = pkg.conv_fwd(qx, qw, (1, 2, 2), 0, 1, scale_x=sx, scale_w=sw)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d(bytes8(qx), bytes8(qw), (1, 2, 2), (0, 0, 0), (1, 1, 1), sx.item(), sw.item())
    assert_close(as_f64(y), ref, "fp8 two-phase")


def test_fp8_conv_with_bias(pkg):
    """The fp8 conv with both scales and a bias (FlyDSL PR #860's bias test
    case): bias added after the dequantisation scales."""
    xs, ws = (1, 64, 4, 9, 11), (96, 64, 1, 3, 3)
    x = cw.randn_bf16(xs, 430, 1.0, "cuda")
    w = cw.randn_bf16(ws, 530, 1.0 / np.sqrt(576), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    b = torch.linspace(-1.0, 2.0, 96, dtype=torch.float32, device="cuda")
    for split_k in (True, False):
        y = pkg.conv_fwd(qx, qw, 1, (0, 1, 1), 1, scale_x=sx, scale_w=sw, split_k=split_k, bias=b)
        torch.cuda.synchronize()
        assert pkg.conv_get_device_status() == 0
        ref = oracle.conv3d(bytes8(qx), bytes8(qw), (1, 1, 1), (0, 1, 1), (1, 1, 1), sx.item(),
                            sw.item(), bias=b.double().cpu().numpy())
        assert_close(as_f64(y), ref, f"fp8 bias split={split_k}")


@pytest.mark.parametrize("act", ["relu", "silu", "gelu"])
def test_fp8_conv_with_bias_and_activation(pkg, act):
    """The fp8 conv with both scales, a bias and an activation."""
    xs, ws = (1, 64, 4, 9, 11), (96, 64, 1, 3, 3)
    x = cw.randn_bf16(xs, 431, 1.0, "cuda")
    w = cw.randn_bf16(ws, 531, 1.0 / np.sqrt(576), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    b = torch.linspace(-1.0, 2.0, 96, dtype=torch.float32, device="cuda")
    for split_k in (True, False):
        y = pkg.conv_fwd(qx, qw, 1, (0, 1, 1), 1, scale_x=sx, scale_w=sw, split_k=split_k, bias=b,
                         act=act)
        torch.cuda.synchronize()
        assert pkg.conv_get_device_status() == 0
        ref = oracle.conv3d(bytes8(qx), bytes8(qw), (1, 1, 1), (0, 1, 1), (1, 1, 1), sx.item(),
                            sw.item(), bias=b.double().cpu().numpy(), act=act)
        assert_close(as_f64(y), ref, f"fp8 bias+{act} split={split_k}")


@pytest.mark.parametrize("shapes", [((2, 3, 1, 32, 48), (64, 3, 1, 16, 16), (1, 16, 16)),
                                    ((3, 3, 1, 28, 35), (40, 3, 1, 7, 7), (1, 7, 7))])
def test_fp8_patch_gemm(pkg, shapes):
    """fp8 non-overlapping patches (the gathered-patch GEMM), packed from
    NCDHW / KCTRS bf16; the 7x7x3 patch is 147 bytes (byte-wise gather)."""
    xs, ws, st = shapes
    x = cw.randn_bf16(xs, 440, 1.0, "cuda")
    w = cw.randn_bf16(ws, 540, 1.0 / np.sqrt(ws[1] * ws[3] * ws[4]), "cuda")
    qx, sx, qw, sw = _fp8_operands(pkg, x, w)
    assert pkg.conv_fwd_plan(tuple(qx.shape), tuple(qw.shape), st, 0, 1, 1)["class"] == "patch_gemm"
    y = pkg.conv_fwd(qx, qw, st, 0, 1, scale_x=sx, scale_w=sw)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d(bytes8(qx), bytes8(qw), st, (0, 0, 0), (1, 1, 1), sx.item(), sw.item())
    assert_close(as_f64(y), ref, f"fp8 patch {shapes}")
