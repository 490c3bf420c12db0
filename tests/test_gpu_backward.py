"""GPU parity of the point-output backward passes (MIOpen PR #10912:
backward data and backward weights of patch-embedding shapes, each one GEMM)
against the fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import conv_workloads as cw
import oracle
from _gpu_util import as_f64, assert_close, bits16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


# (x [N,D,H,W,C], K): the filter equals x's spatial extent, stride = filter
CASES = [
    ((9500, 1, 14, 14, 3), 1280),    # the page's patch embedding, in full
    ((37, 1, 14, 14, 3), 100),       # odd batch, K % 8 != 0
    ((130, 2, 4, 4, 8), 96),         # 3-D filter
    ((9, 1, 16, 16, 3), 64),
    ((1, 1, 2, 2, 4), 8),            # one image
]


def _operands(xs, K, seed):
    N = xs[0]
    ws = (K, xs[1], xs[2], xs[3], xs[4])
    J = xs[1] * xs[2] * xs[3] * xs[4]
    x = cw.randn_bf16(xs, 700 + seed, 1.0, "cuda")
    w = cw.randn_bf16(ws, 800 + seed, 1.0 / np.sqrt(J), "cuda")
    dy = cw.randn_bf16((N, 1, 1, 1, K), 900 + seed, 1.0 / np.sqrt(max(N, K)), "cuda")
    return x, w, dy, ws, (xs[1], xs[2], xs[3])


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_backward_data(pkg, case):
    xs, K = case
    x, w, dy, ws, st = _operands(xs, K, CASES.index(case))
    dx = pkg.conv_bwd_data_point(dy, w, xs, st)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d_bwd_data(bits16(dy), bits16(w), xs, st)
    assert_close(as_f64(dx), ref, f"dgrad {case}")


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_backward_weight(pkg, case):
    xs, K = case
    x, w, dy, ws, st = _operands(xs, K, CASES.index(case))
    dw = pkg.conv_bwd_weight_point(x, dy, ws, st)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d_bwd_weight(bits16(x), bits16(dy), ws, st)
    assert_close(as_f64(dw), ref, f"wgrad {case}")


def test_backward_weight_without_split_k(pkg):
    """A workspace that holds only the transposes: the GEMM runs unsplit."""
    xs, K = (300, 1, 14, 14, 3), 64
    x, w, dy, ws, st = _operands(xs, K, 11)
    Np = (xs[0] + 7) // 8 * 8
    J = 588
    head = (K * Np * 2 + 255) // 256 * 256 + (J * Np * 2 + 255) // 256 * 256
    assert pkg.conv_bwd_point_workspace_bytes(xs, ws, st, 0, 1, 1) > head   # split-K wanted
    wsp = torch.empty(head, dtype=torch.uint8, device="cuda")
    dw = pkg.conv_bwd_weight_point(x, dy, ws, st, workspace=wsp)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    ref = oracle.conv3d_bwd_weight(bits16(x), bits16(dy), ws, st)
    assert_close(as_f64(dw), ref, "wgrad unsplit")


def test_backward_rejects_other_shapes(pkg):
    x = torch.zeros((2, 1, 8, 8, 16), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((32, 1, 3, 3, 16), dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros((2, 1, 6, 6, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_bwd_data_point(dy, w, tuple(x.shape), 1,
                                workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == pkg.CONV_ERR_UNSUPPORTED
    xs = (4, 1, 4, 4, 8)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.ConvError) as e:
        pkg.conv_bwd_data_point(torch.zeros((4, 1, 1, 1, 8), dtype=torch.bfloat16, device="cuda"),
                                torch.zeros((8, 1, 4, 4, 8), dtype=torch.bfloat16, device="cuda"),
                                xs, (1, 4, 4), workspace=small)
    assert e.value.status == pkg.CONV_ERR_INVALID


def test_backward_odd_extents(pkg):
    """J = T*R*S*C = 27 and K = 7 / 8: the transposes move single elements and
    the outputs leave through 2-byte stores."""
    xs = (21, 1, 3, 3, 3)
    x, w, dy, ws, st = _operands(xs, 8, 12)
    dx = pkg.conv_bwd_data_point(dy, w, xs, st)
    torch.cuda.synchronize()
    assert_close(as_f64(dx), oracle.conv3d_bwd_data(bits16(dy), bits16(w), xs, st), "dgrad odd J")
    x, w, dy, ws, st = _operands(xs, 7, 13)
    dw = pkg.conv_bwd_weight_point(x, dy, ws, st)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert_close(as_f64(dw), oracle.conv3d_bwd_weight(bits16(x), bits16(dy), ws, st), "wgrad odd")


@pytest.mark.parametrize("amn", ["0", "1"])
def test_backward_weight_both_operand_paths(pkg, amn):
    """dW with dy read in place as an MN-major operand (K % 8 == 0, the default)
    and through the transposed copy (the dy_in_place override 0): both against the oracle,
    with split-K and without (a workspace holding only the copies)."""
    xs, K = (700, 1, 14, 14, 3), 256
    x, w, dy, ws, st = _operands(xs, K, 14)
    with pkg.overrides(dy_in_place=int(amn)):
        for small in (False, True):
            wsp = None
            if small:
                Np = (xs[0] + 7) // 8 * 8
                wsp = torch.empty(((K * Np * 2 + 255) // 256 + (588 * Np * 2 + 255) // 256) * 256,
                                  dtype=torch.uint8, device="cuda")
            dw = pkg.conv_bwd_weight_point(x, dy, ws, st, workspace=wsp)
            torch.cuda.synchronize()
            assert pkg.conv_get_device_status() == 0
            assert_close(as_f64(dw), oracle.conv3d_bwd_weight(bits16(x), bits16(dy), ws, st),
                         f"wgrad amn={amn} small_ws={small}")
