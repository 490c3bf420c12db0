"""GPU parity of conv_fwd_ncdhw_fp8: the e4m3 convolution of a bf16
channel-major (NCDHW) activation quantised while it is loaded, against the
fp64 oracle's conv of the oracle's own pack of the same activation (the
fp8-cast conv reference): the scale's bits must equal the oracle's, and every
output element must be within the tolerance.  Shapes cover several strips
and row tiles, frames narrower and wider than a tile, partial 128-channel
chunks and column tiles, N and D > 1, 1x1 / 1x3 / 3x1 / 3x3 / 5x5 filters,
single CTAs and CTA pairs, bias, and the argument checks."""
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


# (x NCDHW, w KCTRS with T = 1)
CASES = [
    ((1, 32, 2, 10, 12), (40, 32, 1, 3, 3)),
    ((2, 144, 1, 9, 20), (96, 144, 1, 3, 3)),
    ((1, 16, 3, 5, 7), (32, 16, 1, 5, 5)),
    ((1, 48, 1, 4, 40), (64, 48, 1, 1, 3)),
    ((1, 16, 2, 6, 6), (32, 16, 1, 1, 1)),
    ((1, 16, 1, 30, 3), (32, 16, 1, 3, 1)),
    ((1, 256, 2, 24, 90), (272, 256, 1, 3, 3)),
    ((1, 64, 1, 40, 33), (512, 64, 1, 3, 3)),
]


def _run(pkg, xs, ws, seed, bias=False, small_ws=False):
    x = cw.randn_bf16(xs, 950 + seed, 1.0, "cuda")
    crs = ws[1] * ws[2] * ws[3] * ws[4]
    wb = cw.randn_bf16(ws, 960 + seed, 1.0 / np.sqrt(crs), "cuda")
    qw, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(wb)          # e4m3 KTRSC + scale
    pad = (0, (ws[3] - 1) // 2, (ws[4] - 1) // 2)
    b = None
    if bias:
        g = torch.Generator(device="cpu").manual_seed(970 + seed)
        b = torch.randn(ws[0], generator=g).float().cuda()
    wsp = torch.empty(16, dtype=torch.uint8, device="cuda") if small_ws else None
    y, sx = pkg.conv_fwd_ncdhw_fp8(x, qw, 1, pad, 1, scale_w=sw, bias=b, workspace=wsp)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref_q, ref_s = oracle.pack_ncdhw_to_ndhwc_fp8(bits16(x))
    assert np.float32(sx.item()).tobytes() == np.float32(ref_s).tobytes()
    ref = oracle.conv3d(ref_q, bytes8(qw), (1, 1, 1), pad, (1, 1, 1), ref_s, sw.item())
    if bias:
        ref = ref + b.cpu().double().numpy()
    return x, qw, sw, sx, y, ref, pad


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("small_ws", [False, True], ids=["ahead", "in-place"])
@pytest.mark.parametrize("k_bytes", [128, 256], ids=["tap", "two-taps"])
def test_fused_quantising_loader_matches_oracle(pkg, case, pair, small_ws, k_bytes):
    """With the preferred workspace the converters work one m-tile ahead into
    a scratch and the strips are copied back for every column tile; with only
    the amax word they convert each chunk in place: the same values either
    way.  Weight stages hold one filter tap or two (the last group of an odd
    tap count half empty)."""
    xs, ws = case
    with pkg.overrides(pair=pair, k_bytes=k_bytes):
        _, _, _, _, y, ref, _ = _run(pkg, xs, ws, CASES.index(case), small_ws=small_ws)
    assert_close(as_f64(y), ref,
                 f"fused e4m3 NCDHW {case} pair={pair} small_ws={small_ws} k_bytes={k_bytes}")


def test_fused_with_bias_and_against_pack_then_conv(pkg):
    """With a bias against the oracle; and without one, the pack + conv_fwd
    route on the same operands gives the same scale bits and the same values
    within the tolerance (the codes are the same; only the fp32 summation
    order may differ)."""
    xs, ws = (2, 128, 2, 12, 30), (160, 128, 1, 3, 3)
    _, _, _, _, y, ref, _ = _run(pkg, xs, ws, 20, bias=True)
    assert_close(as_f64(y), ref, "fused with bias")
    x, qw, sw, sx, y0, ref0, pad = _run(pkg, xs, ws, 21)
    qx, sx2 = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(x)
    y2 = pkg.conv_fwd(qx, qw, 1, pad, 1, scale_x=sx2, scale_w=sw)
    torch.cuda.synchronize()
    assert np.float32(sx.item()).tobytes() == np.float32(sx2.item()).tobytes()
    assert_close(as_f64(y2), ref0, "pack + conv_fwd")
    assert_close(as_f64(y0), as_f64(y2), "fused vs pack + conv_fwd")


def test_fused_all_zero_activation(pkg):
    x = torch.zeros((1, 32, 1, 6, 8), dtype=torch.bfloat16, device="cuda")
    wb = cw.randn_bf16((32, 32, 1, 3, 3), 990, 0.1, "cuda")
    qw, sw = pkg.pack_ncdhw_bf16_to_ndhwc_fp8(wb)
    y, sx = pkg.conv_fwd_ncdhw_fp8(x, qw, 1, (0, 1, 1), 1, scale_w=sw)
    torch.cuda.synchronize()
    assert sx.item() == 1.0 and not y.float().abs().sum().item()


@pytest.mark.parametrize("ws,stride,pad", [
    ((32, 32, 3, 3, 3), 1, (1, 1, 1)),        # T > 1
    ((32, 32, 1, 3, 3), (1, 2, 2), (0, 1, 1)),  # stride
    ((32, 32, 1, 2, 2), 1, (0, 0, 0)),        # even filter
    ((32, 32, 1, 3, 3), 1, (0, 0, 0)),        # not "same" padding
])
def test_fused_unsupported_shapes(pkg, ws, stride, pad):
    x = torch.zeros((1, 32, 4, 8, 8), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((ws[0], ws[2], ws[3], ws[4], ws[1]), dtype=torch.float8_e4m3fn,
                     device="cuda")
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_ncdhw_fp8(x, qw, stride, pad, 1)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    # C not a multiple of 16
    x = torch.zeros((1, 24, 4, 8, 8), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((32, 1, 3, 3, 24), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_fwd_ncdhw_fp8(x, qw, 1, (0, 1, 1), 1)
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED


def _fuzz_cases(n=16, seed=20261):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        N, D = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        C = 16 * int(rng.integers(1, 11))                 # up to 160: partial 128-channel chunks
        H, W = int(rng.integers(1, 25)), int(rng.integers(1, 25))
        K = 32 * int(rng.integers(1, 9))                  # up to 256: partial column tiles
        R, S = (int(v) for v in rng.choice([1, 3, 5], size=2))
        cases.append(((N, C, D, H, W), (K, C, 1, R, S), int(rng.integers(0, 2)),
                      int(rng.choice([128, 256])), bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("i", range(16))
def test_fused_loader_fuzz(pkg, i):
    """Seeded random problems (N, D up to 2 / 3, C up to 160, H and W 1..24,
    K up to 256, 1 / 3 / 5-tap filter rows and columns), each with a random
    CTA-pair choice, one or two taps per weight stage and either workspace
    mode, against the oracle's pack + conv."""
    xs, ws, pair, k_bytes, small_ws = _fuzz_cases()[i]
    with pkg.overrides(pair=pair, k_bytes=k_bytes):
        _, _, _, _, y, ref, _ = _run(pkg, xs, ws, 100 + i, small_ws=small_ws)
    assert_close(as_f64(y), ref, f"fuzz {i}: x {xs} w {ws} pair={pair} k_bytes={k_bytes} "
                                 f"small_ws={small_ws}")
