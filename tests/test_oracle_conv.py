"""Pins of the CPU oracle's convolution (no GPU).

Each test checks the oracle against something other than itself: the torch CPU
fp64 library convolution, a scatter-form brute force, an explicit im2col GEMM,
and the closed forms the method's pages rely on (1x1x1 conv == matmul,
point-output conv == one GEMM over reshaped patches, delta filter == shifted
copy, linearity).  A dropped tap, a wrong sign in the padding offset, a
transposed operand or a swapped stride/dilation each fails at least one.
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _torch_conv_ndhwc(x, w, stride, pad, dil):
    """torch CPU fp64 F.conv3d in NDHWC/KTRSC terms (library routine)."""
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(0, 4, 1, 2, 3)
    wt = torch.from_numpy(np.ascontiguousarray(w)).permute(0, 4, 1, 2, 3)
    y = F.conv3d(xt, wt, stride=tuple(stride), padding=tuple(pad), dilation=tuple(dil))
    return y.permute(0, 2, 3, 4, 1).contiguous().numpy()


def _random_case(rng):
    N = int(rng.integers(1, 3))
    C = int(rng.integers(1, 9))
    K = int(rng.integers(1, 9))
    T, R, S = (int(v) for v in rng.integers(1, 5, size=3))
    stride = [int(v) for v in rng.integers(1, 4, size=3)]
    dil = [int(v) for v in rng.integers(1, 3, size=3)]
    pad = [int(rng.integers(0, f)) if f > 1 else int(rng.integers(0, 2)) for f in (T, R, S)]
    # input extents large enough to give at least one output position
    ext = []
    for f, p, d in zip((T, R, S), pad, dil):
        need = d * (f - 1) + 1 - 2 * p
        ext.append(max(1, need) + int(rng.integers(0, 5)))
    D, H, W = ext
    return (N, D, H, W, C), (K, T, R, S, C), stride, pad, dil


def test_oracle_matches_torch_conv3d_fp64_random_shapes():
    rng = np.random.default_rng(12345)
    for _ in range(220):
        xs, ws, stride, pad, dil = _random_case(rng)
        x = rng.standard_normal(xs)
        w = rng.standard_normal(ws)
        ref = _torch_conv_ndhwc(x, w, stride, pad, dil)
        got = oracle.conv3d(x, w, stride, pad, dil)
        assert got.shape == ref.shape, (xs, ws, stride, pad, dil)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_oracle_bf16_inputs_match_torch_on_decoded_values():
    rng = np.random.default_rng(7)
    for _ in range(20):
        xs, ws, stride, pad, dil = _random_case(rng)
        xb = torch.randn(xs, dtype=torch.float32).to(torch.bfloat16)
        wb = torch.randn(ws, dtype=torch.float32).to(torch.bfloat16)
        ref = _torch_conv_ndhwc(xb.double().numpy(), wb.double().numpy(), stride, pad, dil)
        got = oracle.conv3d(xb.view(torch.int16).numpy().view(np.uint16),
                            wb.view(torch.int16).numpy().view(np.uint16), stride, pad, dil)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _scatter_conv(x, w, stride, pad, dil):
    """Brute force, second formulation: walk every input pixel and every tap
    and scatter-add its contribution into the output it feeds."""
    N, D, H, W, C = x.shape
    K, T, R, S, _ = w.shape
    Do = (D + 2 * pad[0] - dil[0] * (T - 1) - 1) // stride[0] + 1
    Ho = (H + 2 * pad[1] - dil[1] * (R - 1) - 1) // stride[1] + 1
    Wo = (W + 2 * pad[2] - dil[2] * (S - 1) - 1) // stride[2] + 1
    y = np.zeros((N, Do, Ho, Wo, K))
    for n, d, h, ww in itertools.product(range(N), range(D), range(H), range(W)):
        for t, r, s in itertools.product(range(T), range(R), range(S)):
            # input d feeds output od when od*stride - pad + t*dil == d
            qd, qh, qw = d + pad[0] - t * dil[0], h + pad[1] - r * dil[1], ww + pad[2] - s * dil[2]
            if qd % stride[0] or qh % stride[1] or qw % stride[2]:
                continue
            od, oh, ow = qd // stride[0], qh // stride[1], qw // stride[2]
            if not (0 <= od < Do and 0 <= oh < Ho and 0 <= ow < Wo):
                continue
            y[n, od, oh, ow, :] += w[:, t, r, s, :] @ x[n, d, h, ww, :]
    return y


def test_oracle_matches_scatter_brute_force_tiny():
    rng = np.random.default_rng(99)
    cases = [((1, 3, 4, 5, 2), (3, 2, 3, 2, 2), (1, 2, 1), (1, 1, 0), (1, 1, 2)),
             ((2, 4, 3, 3, 3), (2, 3, 1, 3, 3), (2, 1, 1), (2, 0, 1), (1, 1, 1)),
             ((1, 5, 5, 5, 1), (1, 3, 3, 3, 1), (3, 3, 3), (1, 1, 1), (1, 1, 1)),
             ((1, 2, 6, 7, 4), (5, 1, 2, 3, 4), (1, 3, 2), (0, 1, 2), (1, 2, 1))]
    for xs, ws, stride, pad, dil in cases:
        x = rng.standard_normal(xs)
        w = rng.standard_normal(ws)
        np.testing.assert_allclose(oracle.conv3d(x, w, stride, pad, dil),
                                   _scatter_conv(x, w, stride, pad, dil), rtol=1e-12, atol=1e-12)


def _im2col_gemm(x, w, stride, pad, dil):
    """Third formulation: materialise the im2col matrix A[M, T*R*S*C] (zeros
    at padding) and multiply by W[K, T*R*S*C]^T -- the GEMM view with
    M = output positions, N = filters, reduction over (t, r, s, c)."""
    N, D, H, W, C = x.shape
    K, T, R, S, _ = w.shape
    xp = np.pad(x, ((0, 0), (pad[0], pad[0]), (pad[1], pad[1]), (pad[2], pad[2]), (0, 0)))
    Do = (D + 2 * pad[0] - dil[0] * (T - 1) - 1) // stride[0] + 1
    Ho = (H + 2 * pad[1] - dil[1] * (R - 1) - 1) // stride[1] + 1
    Wo = (W + 2 * pad[2] - dil[2] * (S - 1) - 1) // stride[2] + 1
    cols = []
    for t, r, s in itertools.product(range(T), range(R), range(S)):
        sl = xp[:, t * dil[0]: t * dil[0] + (Do - 1) * stride[0] + 1: stride[0],
                r * dil[1]: r * dil[1] + (Ho - 1) * stride[1] + 1: stride[1],
                s * dil[2]: s * dil[2] + (Wo - 1) * stride[2] + 1: stride[2], :]
        cols.append(sl.reshape(-1, C))
    A = np.concatenate(cols, axis=1)
    return (A @ w.reshape(K, -1).T).reshape(N, Do, Ho, Wo, K)


def test_oracle_matches_im2col_gemm():
    rng = np.random.default_rng(5)
    for _ in range(30):
        xs, ws, stride, pad, dil = _random_case(rng)
        x = rng.standard_normal(xs)
        w = rng.standard_normal(ws)
        np.testing.assert_allclose(oracle.conv3d(x, w, stride, pad, dil),
                                   _im2col_gemm(x, w, stride, pad, dil), rtol=1e-12, atol=1e-12)


def test_1x1x1_conv_is_matmul():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, 4, 5, 12))
    w = rng.standard_normal((7, 1, 1, 1, 12))
    got = oracle.conv3d(x, w)
    ref = (x.reshape(-1, 12) @ w.reshape(7, 12).T).reshape(2, 3, 4, 5, 7)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_point_output_conv_is_one_gemm():
    """Patch-embedding shape (stride == filter, no pad, 1x1 output): every
    batch row of x and every row of w enumerate (t, r, s, c) in the same
    order, so the conv is x.reshape(N, TRSC) @ w.reshape(K, TRSC)^T
    (MIOpen PR #10912, description)."""
    rng = np.random.default_rng(2)
    xb = torch.randn((37, 1, 14, 14, 3)).to(torch.bfloat16)
    wb = (torch.randn((48, 1, 14, 14, 3)) / np.sqrt(588)).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    wbits = wb.view(torch.int16).numpy().view(np.uint16)
    got = oracle.conv3d(xbits, wbits, stride=(1, 14, 14))
    assert got.shape == (37, 1, 1, 1, 48)
    ref = xb.double().numpy().reshape(37, 588) @ wb.double().numpy().reshape(48, 588).T
    np.testing.assert_allclose(got.reshape(37, 48), ref, rtol=1e-12, atol=1e-12)
    # the 3D form with a temporal extent as well
    x = rng.standard_normal((5, 2, 4, 4, 3))
    w = rng.standard_normal((6, 2, 4, 4, 3))
    got = oracle.conv3d(x, w, stride=(2, 4, 4))
    np.testing.assert_allclose(got.reshape(5, 6), x.reshape(5, -1) @ w.reshape(6, -1).T,
                               rtol=1e-12, atol=1e-12)


def test_delta_filter_is_shifted_copy_exactly():
    """w[k,t,r,s,c] = [c == k] * [(t,r,s) == tap] gives out[n,od,oh,ow,k] =
    x[n, od*sd-pd+t0*dd, ...,  k] or 0 out of range: exact equality."""
    xb = torch.randn((2, 5, 6, 7, 4)).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    x = xb.double().numpy()
    for (T, R, S), tap, stride, pad, dil in [((3, 3, 3), (2, 0, 1), (1, 1, 1), (1, 1, 1), (1, 1, 1)),
                                            ((1, 3, 3), (0, 2, 2), (1, 2, 1), (0, 1, 1), (1, 1, 2)),
                                            ((3, 1, 1), (0, 0, 0), (2, 1, 1), (1, 0, 0), (2, 1, 1))]:
        w = torch.zeros((4, T, R, S, 4), dtype=torch.bfloat16)
        for k in range(4):
            w[k, tap[0], tap[1], tap[2], k] = 1.0
        wbits = w.view(torch.int16).numpy().view(np.uint16)
        got = oracle.conv3d(xbits, wbits, stride, pad, dil)
        N, Do, Ho, Wo, K = got.shape
        ref = np.zeros_like(got)
        for od, oh, ow in itertools.product(range(Do), range(Ho), range(Wo)):
            d = od * stride[0] - pad[0] + tap[0] * dil[0]
            h = oh * stride[1] - pad[1] + tap[1] * dil[1]
            ww = ow * stride[2] - pad[2] + tap[2] * dil[2]
            if 0 <= d < 5 and 0 <= h < 6 and 0 <= ww < 7:
                ref[:, od, oh, ow, :] = x[:, d, h, ww, :]
        assert np.array_equal(got, ref)


def test_linearity_in_x_and_w():
    rng = np.random.default_rng(3)
    xs, ws, stride, pad, dil = (2, 4, 5, 6, 5), (3, 3, 2, 3, 5), (1, 2, 1), (1, 0, 1), (1, 1, 2)
    x1, x2 = rng.standard_normal(xs), rng.standard_normal(xs)
    w1, w2 = rng.standard_normal(ws), rng.standard_normal(ws)
    a, b = 0.75, -1.5
    lhs = oracle.conv3d(a * x1 + b * x2, w1, stride, pad, dil)
    rhs = a * oracle.conv3d(x1, w1, stride, pad, dil) + b * oracle.conv3d(x2, w1, stride, pad, dil)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    lhs = oracle.conv3d(x1, a * w1 + b * w2, stride, pad, dil)
    rhs = a * oracle.conv3d(x1, w1, stride, pad, dil) + b * oracle.conv3d(x1, w2, stride, pad, dil)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def test_scales_multiply_the_sum():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 3, 3, 3, 2))
    w = rng.standard_normal((2, 3, 3, 3, 2))
    base = oracle.conv3d(x, w, pad=(1, 1, 1))
    np.testing.assert_allclose(oracle.conv3d(x, w, pad=(1, 1, 1), scale_x=0.5, scale_w=3.0),
                               1.5 * base, rtol=1e-15, atol=0)


def test_points_equal_full_evaluation():
    xb = torch.randn((2, 5, 6, 7, 8)).to(torch.bfloat16)
    wb = torch.randn((9, 3, 3, 3, 8)).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    wbits = wb.view(torch.int16).numpy().view(np.uint16)
    full = oracle.conv3d(xbits, wbits, (1, 2, 1), (1, 1, 0), (1, 1, 2))
    idx = np.random.default_rng(0).integers(0, full.size, size=500)
    pts = oracle.conv3d_points(xbits, wbits, idx, (1, 2, 1), (1, 1, 0), (1, 1, 2))
    assert np.array_equal(pts, full.ravel()[idx])


def test_points_on_channel_major_x_match_torch():
    """The channel-major (NCDHW) evaluation against torch CPU fp64 F.conv3d
    on the same array, in torch's own layout (no permutation of x), over
    random geometries; a swapped stride of the NCDHW indexing (c vs w, d vs
    h) fails it.  Outputs are compared at every flat NDHWC index."""
    rng = np.random.default_rng(606)
    for _ in range(60):
        (N, D, H, W, C), ws, stride, pad, dil = _random_case(rng)
        x = rng.standard_normal((N, C, D, H, W))
        w = rng.standard_normal(ws)
        wt = torch.from_numpy(np.ascontiguousarray(w)).permute(0, 4, 1, 2, 3)
        ref = F.conv3d(torch.from_numpy(x), wt, stride=tuple(stride), padding=tuple(pad),
                       dilation=tuple(dil)).permute(0, 2, 3, 4, 1).contiguous().numpy()
        idx = np.arange(ref.size, dtype=np.int64)
        got = oracle.conv3d_points(x, w, idx, stride, pad, dil, x_layout="ncdhw")
        np.testing.assert_allclose(got, ref.ravel(), rtol=1e-12, atol=1e-12)
        # and the same numbers as the channel-last evaluation of the permuted x
        nd = oracle.conv3d_points(np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1)), w, idx,
                                  stride, pad, dil)
        assert np.array_equal(got, nd)


def test_activations_match_torch_fp64():
    """The epilogue activations against torch's own fp64 relu / silu / gelu
    (erf form) on values spanning the tails, plus exact special values."""
    rng = np.random.default_rng(77)
    v = np.concatenate([rng.standard_normal(5000) * 4, np.linspace(-40, 40, 801),
                        [0.0, -0.0, 1e-30, -1e-30]])
    tv = torch.from_numpy(v)
    ref = {"relu": F.relu(tv), "silu": F.silu(tv), "gelu": F.gelu(tv)}
    for act, r in ref.items():
        got = oracle.activate(v, act)
        np.testing.assert_allclose(got, r.numpy(), rtol=1e-12, atol=1e-15, err_msg=act)
    assert np.array_equal(oracle.activate(v, "none"), v)
    assert oracle.activate(np.array([-2.0, 0.0, 3.0]), "relu").tolist() == [0.0, 0.0, 3.0]
    assert oracle.activate(np.array([0.0]), "silu")[0] == 0.0
    assert oracle.activate(np.array([0.0]), "gelu")[0] == 0.0
    # far tails: silu and gelu approach the identity above and zero below
    big = oracle.activate(np.array([60.0, -60.0]), "gelu")
    assert big[0] == 60.0 and abs(big[1]) < 1e-300
    with pytest.raises(ValueError):
        oracle.activate(v, "tanh")


def test_conv_with_bias_and_activation_matches_torch():
    """conv + bias + activation against torch CPU fp64 F.conv3d (with its own
    bias) followed by torch's activation."""
    rng = np.random.default_rng(78)
    x = rng.standard_normal((2, 4, 5, 6, 7))
    w = rng.standard_normal((9, 3, 2, 3, 7)) / 8
    b = rng.standard_normal(9)
    xt = torch.from_numpy(x).permute(0, 4, 1, 2, 3)
    wt = torch.from_numpy(w).permute(0, 4, 1, 2, 3)
    y = F.conv3d(xt, wt, bias=torch.from_numpy(b), stride=(1, 2, 1), padding=(1, 1, 0))
    for act, fn in (("relu", F.relu), ("silu", F.silu), ("gelu", F.gelu)):
        ref = fn(y).permute(0, 2, 3, 4, 1).contiguous().numpy()
        got = oracle.conv3d(x, w, (1, 2, 1), (1, 1, 0), (1, 1, 1), bias=b, act=act)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12, err_msg=act)
        idx = np.arange(ref.size, dtype=np.int64)[::7]
        pts = oracle.conv3d_points(x, w, idx, (1, 2, 1), (1, 1, 0), (1, 1, 1), bias=b, act=act)
        assert np.array_equal(pts, got.ravel()[idx])


def test_points_reject_out_of_range_index():
    x = np.zeros((1, 2, 2, 2, 1))
    w = np.zeros((1, 1, 1, 1, 1))
    with pytest.raises(ValueError):
        oracle.conv3d_points(x, w, np.array([8], dtype=np.int64))


def test_out_extent_matches_torch_shape_rule():
    for inp, f, s, p, d in itertools.product(range(1, 9), range(1, 4), range(1, 4), range(0, 3),
                                              range(1, 3)):
        span = inp + 2 * p - d * (f - 1)
        if span < 1:
            continue
        x = torch.zeros((1, 1, inp))
        w = torch.zeros((1, 1, f))
        ref = F.conv1d(x, w, stride=s, padding=p, dilation=d).shape[-1]
        assert oracle.out_extent(inp, f, s, p, d) == ref


def test_bias_special_cases():
    """A per-filter bias (FlyDSL PR #860 lists a bias case among the fp8 conv
    tests): with zero weights, or a zero input, every output of filter k is
    exactly bias[k]; the sampled evaluation adds the same entry."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 3, 5, 4, 6))
    w = rng.standard_normal((7, 3, 2, 2, 6))
    b = rng.standard_normal(7)
    out0 = oracle.conv3d(x, np.zeros_like(w), (1, 2, 1), (1, 0, 1), (1, 1, 2), bias=b)
    assert np.array_equal(out0, np.broadcast_to(b, out0.shape))
    outz = oracle.conv3d(np.zeros_like(x), w, (1, 2, 1), (1, 0, 1), (1, 1, 2), 0.5, 3.0, bias=b)
    assert np.array_equal(outz, np.broadcast_to(b, outz.shape))
    full = oracle.conv3d(x, w, (1, 2, 1), (1, 0, 1), (1, 1, 2), 0.5, 3.0, bias=b)
    idx = rng.integers(0, full.size, size=50)
    pts = oracle.conv3d_points(x, w, idx, (1, 2, 1), (1, 0, 1), (1, 1, 2), 0.5, 3.0, bias=b)
    assert np.array_equal(pts, full.reshape(-1)[idx])


# ------------------------------------------------------------ backward passes

def _torch_grads(x, w, dy, stride, pad, dil):
    """fp64 gradients of sum(conv3d(x, w) * dy) by torch autograd on the CPU
    (a library routine), in the NDHWC / KTRSC layouts."""
    xt = torch.from_numpy(np.transpose(x, (0, 4, 1, 2, 3)).copy()).requires_grad_(True)
    wt = torch.from_numpy(np.transpose(w, (0, 4, 1, 2, 3)).copy()).requires_grad_(True)
    y = torch.nn.functional.conv3d(xt, wt, stride=stride, padding=pad, dilation=dil)
    y.backward(torch.from_numpy(np.transpose(dy, (0, 4, 1, 2, 3)).copy()))
    return (np.transpose(xt.grad.numpy(), (0, 2, 3, 4, 1)),
            np.transpose(wt.grad.numpy(), (0, 2, 3, 4, 1)))


def test_backward_matches_torch_autograd():
    rng = np.random.default_rng(31)
    done = 0
    while done < 40:
        T, R, S = (int(v) for v in rng.integers(1, 4, size=3))
        st = tuple(int(v) for v in rng.integers(1, 4, size=3))
        pa = tuple(int(rng.integers(0, f)) if f > 1 else 0 for f in (T, R, S))
        di = tuple(int(v) for v in rng.integers(1, 3, size=3))
        xs = (int(rng.integers(1, 3)), int(rng.integers(1, 6)), int(rng.integers(1, 7)),
              int(rng.integers(1, 7)), int(rng.integers(1, 5)))
        ws = (int(rng.integers(1, 6)), T, R, S, xs[4])
        od = oracle.out_dims(xs, ws, st, pa, di)
        if min(od) < 1:
            continue
        x = rng.standard_normal(xs)
        w = rng.standard_normal(ws)
        dy = rng.standard_normal(od)
        gx, gw = _torch_grads(x, w, dy, st, pa, di)
        np.testing.assert_allclose(oracle.conv3d_bwd_data(dy, w, xs, st, pa, di), gx,
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(oracle.conv3d_bwd_weight(x, dy, ws, st, pa, di), gw,
                                   rtol=1e-12, atol=1e-12)
        done += 1


def test_backward_adjoint_identity():
    """<conv(x, w), dy> = <x, dx(dy, w)> = <w, dw(x, dy)>: the three share one
    trilinear form."""
    rng = np.random.default_rng(32)
    xs, ws, st, pa, di = (2, 5, 6, 7, 3), (4, 3, 2, 3, 3), (2, 1, 2), (1, 1, 0), (1, 2, 1)
    x, w = rng.standard_normal(xs), rng.standard_normal(ws)
    dy = rng.standard_normal(oracle.out_dims(xs, ws, st, pa, di))
    fwd = np.sum(oracle.conv3d(x, w, st, pa, di) * dy)
    assert np.isclose(fwd, np.sum(x * oracle.conv3d_bwd_data(dy, w, xs, st, pa, di)), rtol=1e-12)
    assert np.isclose(fwd, np.sum(w * oracle.conv3d_bwd_weight(x, dy, ws, st, pa, di)), rtol=1e-12)


def test_backward_point_output_is_one_gemm():
    """Point-output shapes (MIOpen PR #10912): dx = dy @ W and dW = dy^T @ x
    over the flattened (t, r, s, c) axis, at the patch-embedding geometry."""
    rng = np.random.default_rng(33)
    xs, ws, st = (37, 1, 14, 14, 3), (20, 1, 14, 14, 3), (1, 14, 14)
    x, w = rng.standard_normal(xs), rng.standard_normal(ws)
    dy = rng.standard_normal((37, 1, 1, 1, 20))
    dx = oracle.conv3d_bwd_data(dy, w, xs, st)
    np.testing.assert_allclose(dx.reshape(37, -1), dy.reshape(37, 20) @ w.reshape(20, -1),
                               rtol=1e-12, atol=1e-12)
    dw = oracle.conv3d_bwd_weight(x, dy, ws, st)
    np.testing.assert_allclose(dw.reshape(20, -1), dy.reshape(37, 20).T @ x.reshape(37, -1),
                               rtol=1e-12, atol=1e-12)
