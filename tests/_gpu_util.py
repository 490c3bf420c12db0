"""Helpers shared by the GPU parity tests: host copies of device tensors as
raw bits, the per-element tolerance check, and oracle calls on the exact bytes
the GPU consumed."""
import numpy as np
import torch

import oracle

RTOL = 1e-2   # |out - ref| <= RTOL*|ref| + ATOL for every checked element
ATOL = 1e-2


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bytes8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def as_f64(out_bf16: torch.Tensor) -> np.ndarray:
    return out_bf16.detach().float().cpu().double().numpy()


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    excess = np.abs(got - ref) - (RTOL * np.abs(ref) + ATOL)
    bad = excess > 0
    if bad.any():
        i = int(np.argmax(excess))
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside tolerance; worst at flat "
            f"{i}: got {got.ravel()[i]!r} ref {ref.ravel()[i]!r}")


def oracle_conv(x: torch.Tensor, w: torch.Tensor, stride, pad, dil, scale_x=1.0, scale_w=1.0):
    if x.dtype == torch.bfloat16:
        xb, wb = bits16(x), bits16(w)
    else:
        xb, wb = bytes8(x), bytes8(w)
    return oracle.conv3d(xb, wb, stride, pad, dil, scale_x, scale_w)


def oracle_points(x_host: np.ndarray, w_host: np.ndarray, idx: np.ndarray, stride, pad, dil,
                  scale_x=1.0, scale_w=1.0):
    return oracle.conv3d_points(x_host, w_host, idx, stride, pad, dil, scale_x, scale_w)
