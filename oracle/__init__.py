"""CPU oracle for the forward implicit-GEMM convolution and the fp8 pack.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports it and shares no code
with it.

The arithmetic lives in ``conv_oracle.c`` (plain C, fp64, OpenMP), compiled
with gcc into ``liboracle.so`` beside it.  This module only marshals numpy
arrays into that library.

Sources followed (each C function cites its passage):
  * FlyDSL PR #860 "fp8 conv3d: 8-wave GEMM pipeline + BIG_IN fix" -- PR
    summary (GEMM view M x K-filters x crs, KTRSC weight, E4M3FN inputs,
    fp8-cast conv reference) and the commit verifying against
    torch.nn.functional.conv3d (torch conv semantics).
  * MIOpen PR #10912 "Use a single GEMM for point-output conv ..." --
    description (point-output conv == one GEMM over channel-last rows).

Pins: every function here is pinned by ``tests/test_oracle_*.py`` against
torch CPU fp64 ``F.conv3d``, a scatter-form brute force, closed forms
(1x1x1 == matmul, point-output == GEMM, delta filter == shifted copy,
linearity) and the E4M3FN format definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ELEM_BF16 = 0
ELEM_E4M3 = 1
ELEM_F64 = 2

_I64P = ctypes.POINTER(ctypes.c_int64)
_I32P = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into liboracle.so with gcc (-O2 -fopenmp)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_amax_bf16.restype = ctypes.c_float
        lib.oracle_amax_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_fp8_scale.restype = ctypes.c_float
        lib.oracle_fp8_scale.argtypes = [ctypes.c_float]
        lib.oracle_quantize_e4m3.restype = ctypes.c_uint8
        lib.oracle_quantize_e4m3.argtypes = [ctypes.c_uint16, ctypes.c_float]
        lib.oracle_pack_ncdhw_to_ndhwc_bf16.restype = None
        lib.oracle_pack_ncdhw_to_ndhwc_bf16.argtypes = [ctypes.c_void_p, _I64P, ctypes.c_void_p]
        lib.oracle_pack_ncdhw_to_ndhwc_fp8.restype = None
        lib.oracle_pack_ncdhw_to_ndhwc_fp8.argtypes = [
            ctypes.c_void_p, _I64P, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
        lib.oracle_out_extent.restype = ctypes.c_int64
        lib.oracle_out_extent.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int]
        conv_args = [ctypes.c_void_p, _I64P, ctypes.c_void_p, _I64P, _I32P, _I32P, _I32P,
                     ctypes.c_int, ctypes.c_double, ctypes.c_double]
        lib.oracle_conv3d_fwd.restype = ctypes.c_int
        lib.oracle_conv3d_fwd.argtypes = conv_args + [ctypes.c_void_p]
        lib.oracle_conv3d_fwd_points.restype = ctypes.c_int
        lib.oracle_conv3d_fwd_points.argtypes = conv_args + [_I64P, ctypes.c_int64,
                                                             ctypes.c_void_p]
        lib.oracle_conv3d_fwd_points_ncdhw.restype = ctypes.c_int
        lib.oracle_conv3d_fwd_points_ncdhw.argtypes = lib.oracle_conv3d_fwd_points.argtypes
        bwd_args = [ctypes.c_void_p, _I64P, ctypes.c_void_p, _I64P, _I32P, _I32P, _I32P,
                    ctypes.c_int, ctypes.c_void_p]
        lib.oracle_conv3d_bwd_data.restype = ctypes.c_int
        lib.oracle_conv3d_bwd_data.argtypes = bwd_args
        lib.oracle_conv3d_bwd_weight.restype = ctypes.c_int
        lib.oracle_conv3d_bwd_weight.argtypes = bwd_args
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        _lib = lib
        return lib


def _dims(v, n):
    arr = (ctypes.c_int64 * n)(*[int(a) for a in v])
    return arr


def _ints3(v):
    return (ctypes.c_int * 3)(*[int(a) for a in v])


def _elem_of(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return ELEM_BF16
    if a.dtype == np.uint8:
        return ELEM_E4M3
    if a.dtype == np.float64:
        return ELEM_F64
    raise TypeError(f"oracle takes bf16 bits (uint16), e4m3 bytes (uint8) or float64, got {a.dtype}")


# ---------------------------------------------------------------- decoders

def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(int(code))


def f32_to_e4m3(v: float) -> int:
    return int(_load().oracle_f32_to_e4m3(float(v)))


def e4m3_decode_table() -> np.ndarray:
    """float64[256]: the value of every E4M3FN code (NaN for 0x7F/0xFF)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)


def quantize_e4m3(xbits: np.ndarray, scale: float) -> np.ndarray:
    """Elementwise q = E4M3FN_satfinite_rne(f32(x)/scale) (small arrays only)."""
    lib = _load()
    flat = np.ascontiguousarray(xbits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_quantize_e4m3(int(b), float(scale)) for b in flat),
                      dtype=np.uint8, count=flat.size)
    return out.reshape(np.shape(xbits))


def amax_bf16(xbits: np.ndarray) -> float:
    a = np.ascontiguousarray(xbits, dtype=np.uint16)
    return float(_load().oracle_amax_bf16(a.ctypes.data, a.size))


def fp8_scale(amax: float) -> float:
    return float(_load().oracle_fp8_scale(float(amax)))


# ---------------------------------------------------------------- pack

def pack_ncdhw_to_ndhwc_bf16(xbits: np.ndarray) -> np.ndarray:
    """[N,C,D,H,W] bf16 bits -> [N,D,H,W,C] bf16 bits."""
    a = np.ascontiguousarray(xbits, dtype=np.uint16)
    N, C, D, H, W = a.shape
    out = np.empty((N, D, H, W, C), dtype=np.uint16)
    _load().oracle_pack_ncdhw_to_ndhwc_bf16(a.ctypes.data, _dims(a.shape, 5), out.ctypes.data)
    return out


def pack_ncdhw_to_ndhwc_fp8(xbits: np.ndarray):
    """[N,C,D,H,W] bf16 bits -> ([N,D,H,W,C] e4m3 bytes, binary32 scale)."""
    a = np.ascontiguousarray(xbits, dtype=np.uint16)
    N, C, D, H, W = a.shape
    out = np.empty((N, D, H, W, C), dtype=np.uint8)
    scale = ctypes.c_float(0.0)
    _load().oracle_pack_ncdhw_to_ndhwc_fp8(a.ctypes.data, _dims(a.shape, 5), out.ctypes.data,
                                           ctypes.byref(scale))
    return out, float(np.float32(scale.value))


# ---------------------------------------------------------------- conv

def out_extent(inp: int, filt: int, stride: int, pad: int, dil: int) -> int:
    return int(_load().oracle_out_extent(inp, filt, stride, pad, dil))


def out_dims(x_shape, w_shape, stride, pad, dil):
    N, D, H, W, C = x_shape
    K, T, R, S, _ = w_shape
    return (N, out_extent(D, T, stride[0], pad[0], dil[0]),
            out_extent(H, R, stride[1], pad[1], dil[1]),
            out_extent(W, S, stride[2], pad[2], dil[2]), K)


ACTIVATIONS = ("none", "relu", "silu", "gelu")


def activate(v: np.ndarray, act: str = "none") -> np.ndarray:
    """The epilogue activation in fp64, each its textbook definition: relu =
    max(v, 0); silu = v * sigmoid(v) = v / (1 + e^-v); gelu = v * Phi(v) with
    Phi the standard normal CDF, v/2 * (1 + erf(v / sqrt 2)).  (The pages name
    no activation; FlyDSL PR #860's fp8 conv tests stop at a bias.)"""
    v = np.asarray(v, dtype=np.float64)
    if act == "none":
        return v
    if act == "relu":
        return np.maximum(v, 0.0)
    if act == "silu":
        with np.errstate(over="ignore"):
            return v / (1.0 + np.exp(-v))
    if act == "gelu":
        try:
            from scipy.special import erf
        except ImportError:   # scipy-less hosts: the scalar library erf
            import math
            erf = np.vectorize(math.erf, otypes=[np.float64])
        return 0.5 * v * (1.0 + erf(v / np.sqrt(2.0)))
    raise ValueError(f"act must be one of {ACTIVATIONS}")


def conv3d(x: np.ndarray, w: np.ndarray, stride=(1, 1, 1), pad=(0, 0, 0), dil=(1, 1, 1),
           scale_x: float = 1.0, scale_w: float = 1.0, bias=None,
           act: str = "none") -> np.ndarray:
    """Full fp64 forward conv.  x [N,D,H,W,C], w [K,T,R,S,C]; both bf16 bits
    (uint16), e4m3 bytes (uint8) or float64.  Returns fp64 [N,Do,Ho,Wo,K]:
    scale_x * scale_w * (the sum), plus bias[k] (a per-filter vector, FlyDSL
    PR #860's fp8 conv tests include a bias case) when given, then the
    activation ``act``."""
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    elem = _elem_of(x)
    if _elem_of(w) != elem:
        raise TypeError("x and w must have the same element type")
    od = out_dims(x.shape, w.shape, stride, pad, dil)
    out = np.zeros(od, dtype=np.float64)
    rc = _load().oracle_conv3d_fwd(x.ctypes.data, _dims(x.shape, 5), w.ctypes.data,
                                   _dims(w.shape, 5), _ints3(stride), _ints3(pad), _ints3(dil),
                                   elem, float(scale_x), float(scale_w), out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_conv3d_fwd: bad shapes")
    if bias is not None:
        out += np.asarray(bias, dtype=np.float64).reshape(-1)
    return activate(out, act)


def conv3d_points(x: np.ndarray, w: np.ndarray, idx: np.ndarray, stride=(1, 1, 1),
                  pad=(0, 0, 0), dil=(1, 1, 1), scale_x: float = 1.0,
                  scale_w: float = 1.0, bias=None, x_layout: str = "ndhwc",
                  act: str = "none") -> np.ndarray:
    """fp64 conv evaluated at flat NDHWC output indices ``idx`` (int64), plus
    bias[k] of each index's filter k when given, then the activation ``act``.
    ``x_layout="ncdhw"``: x is stored channel-major [N,C,D,H,W] (the output
    indices stay NDHWC)."""
    if x_layout not in ("ndhwc", "ncdhw"):
        raise ValueError("x_layout must be 'ndhwc' or 'ncdhw'")
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    elem = _elem_of(x)
    if _elem_of(w) != elem:
        raise TypeError("x and w must have the same element type")
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float64)
    fn = (_load().oracle_conv3d_fwd_points if x_layout == "ndhwc"
          else _load().oracle_conv3d_fwd_points_ncdhw)
    rc = fn(
        x.ctypes.data, _dims(x.shape, 5), w.ctypes.data, _dims(w.shape, 5), _ints3(stride),
        _ints3(pad), _ints3(dil), elem, float(scale_x), float(scale_w),
        idx.ctypes.data_as(_I64P), idx.size, vals.ctypes.data)
    if rc != 0:
        raise ValueError("oracle conv3d points: bad shapes or index out of range")
    if bias is not None:
        vals += np.asarray(bias, dtype=np.float64).reshape(-1)[idx % w.shape[0]]
    return activate(vals, act)


def conv3d_bwd_data(dy: np.ndarray, w: np.ndarray, x_shape, stride=(1, 1, 1), pad=(0, 0, 0),
                    dil=(1, 1, 1)) -> np.ndarray:
    """fp64 gradient of sum(conv3d(x, w) * dy) with respect to x (MIOpen PR
    #10912, backward data).  dy [N,Do,Ho,Wo,K], w [K,T,R,S,C], both bf16 bits
    or float64; returns dx [N,D,H,W,C] = x_shape."""
    dy = np.ascontiguousarray(dy)
    w = np.ascontiguousarray(w)
    elem = _elem_of(dy)
    if _elem_of(w) != elem:
        raise TypeError("dy and w must have the same element type")
    od = out_dims(x_shape, w.shape, stride, pad, dil)
    if tuple(dy.shape) != tuple(od):
        raise ValueError(f"dy must have the output shape {od}")
    dx = np.empty(tuple(x_shape), dtype=np.float64)
    rc = _load().oracle_conv3d_bwd_data(dy.ctypes.data, _dims(x_shape, 5), w.ctypes.data,
                                        _dims(w.shape, 5), _ints3(stride), _ints3(pad),
                                        _ints3(dil), elem, dx.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_conv3d_bwd_data: bad shapes")
    return dx


def conv3d_bwd_weight(x: np.ndarray, dy: np.ndarray, w_shape, stride=(1, 1, 1), pad=(0, 0, 0),
                      dil=(1, 1, 1)) -> np.ndarray:
    """fp64 gradient of sum(conv3d(x, w) * dy) with respect to w (MIOpen PR
    #10912, backward weights).  x [N,D,H,W,C], dy [N,Do,Ho,Wo,K], both bf16
    bits or float64; returns dw [K,T,R,S,C] = w_shape."""
    x = np.ascontiguousarray(x)
    dy = np.ascontiguousarray(dy)
    elem = _elem_of(x)
    if _elem_of(dy) != elem:
        raise TypeError("x and dy must have the same element type")
    od = out_dims(x.shape, w_shape, stride, pad, dil)
    if tuple(dy.shape) != tuple(od):
        raise ValueError(f"dy must have the output shape {od}")
    dw = np.empty(tuple(w_shape), dtype=np.float64)
    rc = _load().oracle_conv3d_bwd_weight(x.ctypes.data, _dims(x.shape, 5), dy.ctypes.data,
                                          _dims(w_shape, 5), _ints3(stride), _ints3(pad),
                                          _ints3(dil), elem, dw.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_conv3d_bwd_weight: bad shapes")
    return dw


def num_threads() -> int:
    return int(_load().oracle_num_threads())
