"""Forward implicit-GEMM convolution for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libconv3d.so`` (C ABI in ``include/conv3d.h``).
It only marshals arguments: shapes, device pointers and the current CUDA
stream of torch tensors.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and every call
raises if the library is missing or returns an error.

Names follow the C ABI (``conv_fwd``, ``pack_ncdhw_bf16_to_ndhwc``,
``pack_ncdhw_bf16_to_ndhwc_fp8``, ...).  ``conv3d``, ``conv2d`` and
``conv1d`` are the convenience wrappers: 2-D and 1-D convolutions run as the
degenerate 3-D forms D=T=1 (and H=R=1 for 1-D), as the FlyDSL PR #860
conv2d/conv1d wrapper commit does.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libconv3d.so")

CONV_OK = 0
CONV_ERR_INVALID = 1
CONV_ERR_UNSUPPORTED = 2
CONV_ERR_CUDA = 3
CONV_ERR_TIMEOUT = 4

CONV_DTYPE_BF16 = 0
CONV_DTYPE_FP8_E4M3 = 1

CLASS_NAMES = {0: "generic", 1: "temporal", 2: "point_gemm", 3: "patch_gemm"}

# epilogue activations (conv_fwd_bias_act)
CONV_ACT_NONE, CONV_ACT_RELU, CONV_ACT_SILU, CONV_ACT_GELU = 0, 1, 2, 3
ACT_CODES = {"none": CONV_ACT_NONE, "relu": CONV_ACT_RELU, "silu": CONV_ACT_SILU,
             "gelu": CONV_ACT_GELU}

# conv_overrides (include/conv3d.h), field order as declared there
OVERRIDE_FIELDS = ("tile_n", "k_bytes", "stages", "group_m", "splits", "pair", "msub", "slices",
                   "epilogue", "hw_major", "two_phase", "repack", "dy_in_place", "pdl",
                   "weight_groups", "ncdhw_in_place", "pack_lanes", "log")


class _Overrides(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int) for f in OVERRIDE_FIELDS]


_I64_5 = ctypes.c_int64 * 5
_I32_3 = ctypes.c_int * 3
_lock = threading.Lock()
_lib = None


class ConvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {_status_string(status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def _status_string(s: int) -> str:
    lib = _lib
    if lib is None:
        return f"status {s}"
    return lib.conv_status_string(int(s)).decode()


def load_library(path: str = LIB_PATH):
    """Load libconv3d.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -m implicit_gemm_convolution_conv3d_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, i64p, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int)
        lib.conv_out_dims.argtypes = [i64p, i64p, i32p, i32p, i32p, i64p]
        lib.conv_out_dims.restype = ctypes.c_int
        lib.conv_fwd_plan.argtypes = [i64p, i64p, i32p, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                      i32p, i32p, i32p, i32p, i32p, i32p,
                                      ctypes.POINTER(ctypes.c_size_t)]
        lib.conv_fwd_plan.restype = ctypes.c_int
        lib.conv_fwd.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, ctypes.c_int, vp, vp, vp,
                                 vp, ctypes.c_size_t, vp]
        lib.conv_fwd.restype = ctypes.c_int
        lib.conv_fwd_bias.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, ctypes.c_int, vp, vp,
                                      vp, vp, vp, ctypes.c_size_t, vp]
        lib.conv_fwd_bias.restype = ctypes.c_int
        lib.conv_fwd_bias_act.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, ctypes.c_int, vp,
                                          vp, vp, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
        lib.conv_fwd_bias_act.restype = ctypes.c_int
        lib.conv_fwd_ncdhw_plan.argtypes = lib.conv_fwd_plan.argtypes
        lib.conv_fwd_ncdhw_plan.restype = ctypes.c_int
        lib.conv_fwd_ncdhw.argtypes = lib.conv_fwd_bias.argtypes
        lib.conv_fwd_ncdhw.restype = ctypes.c_int
        lib.conv_bwd_point_workspace_bytes.argtypes = [i64p, i64p, i32p, i32p, i32p, ctypes.c_int,
                                                       ctypes.POINTER(ctypes.c_size_t)]
        lib.conv_bwd_point_workspace_bytes.restype = ctypes.c_int
        for fn in (lib.conv_bwd_data_point, lib.conv_bwd_weight_point):
            fn.argtypes = [vp, vp, i64p, i64p, i32p, i32p, i32p, vp, vp, ctypes.c_size_t, vp]
            fn.restype = ctypes.c_int
        lib.conv_fwd_kernel_launches.argtypes = [i64p, i64p, i32p, i32p, i32p, ctypes.c_int,
                                                 ctypes.c_size_t, i32p]
        lib.conv_fwd_kernel_launches.restype = ctypes.c_int
        lib.conv_fwd_noalloc.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, ctypes.c_int, vp,
                                         vp, vp, vp]
        lib.conv_fwd_noalloc.restype = ctypes.c_int
        lib.conv_fwd_from_host.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, ctypes.c_int,
                                           vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                           ctypes.c_int, vp]
        lib.conv_fwd_from_host.restype = ctypes.c_int
        lib.pack_ncdhw_bf16_to_ndhwc.argtypes = [vp, i64p, vp, vp]
        lib.pack_ncdhw_bf16_to_ndhwc.restype = ctypes.c_int
        lib.pack_fp8_workspace_size.argtypes = []
        lib.pack_fp8_workspace_size.restype = ctypes.c_size_t
        lib.pack_ncdhw_bf16_to_ndhwc_fp8.argtypes = [vp, i64p, vp, vp, vp, ctypes.c_size_t, vp]
        lib.pack_ncdhw_bf16_to_ndhwc_fp8.restype = ctypes.c_int
        lib.conv_fwd_ncdhw_fp8.argtypes = [vp, i64p, vp, i64p, i32p, i32p, i32p, vp, vp, vp, vp,
                                           vp, ctypes.c_size_t, vp]
        lib.conv_fwd_ncdhw_fp8.restype = ctypes.c_int
        lib.conv_fwd_ncdhw_fp8_workspace_size.argtypes = [i64p, i64p, i32p, i32p, i32p,
                                                          ctypes.POINTER(ctypes.c_size_t)]
        lib.conv_fwd_ncdhw_fp8_workspace_size.restype = ctypes.c_int
        lib.conv_fwd_workspace_size.argtypes = [i64p, i64p, i32p, i32p, i32p, ctypes.c_int]
        lib.conv_fwd_workspace_size.restype = ctypes.c_size_t
        lib.conv_get_device_status_stream.argtypes = [vp, i32p]
        lib.conv_get_device_status_stream.restype = ctypes.c_int
        lib.conv_default_overrides.argtypes = [ctypes.POINTER(_Overrides)]
        lib.conv_default_overrides.restype = None
        lib.conv_set_overrides.argtypes = [ctypes.POINTER(_Overrides)]
        lib.conv_set_overrides.restype = ctypes.c_int
        lib.conv_get_device_status.argtypes = [i32p]
        lib.conv_get_device_status.restype = ctypes.c_int
        lib.conv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.conv_set_wait_limit_ns.restype = None
        lib.conv_status_string.argtypes = [ctypes.c_int]
        lib.conv_status_string.restype = ctypes.c_char_p
        lib.conv_last_error.argtypes = []
        lib.conv_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(rc: int, where: str):
    if rc != CONV_OK:
        detail = _lib.conv_last_error().decode() if _lib is not None else ""
        raise ConvError(rc, where, detail)


def _triple(v: Union[int, Sequence[int]]) -> Tuple[int, int, int]:
    if isinstance(v, int):
        return (v, v, v)
    t = tuple(int(a) for a in v)
    if len(t) != 3:
        raise ValueError("expected an int or a 3-sequence")
    return t


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CONV_DTYPE_BF16
    if t.dtype == torch.float8_e4m3fn:
        return CONV_DTYPE_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or float8_e4m3fn")


# the current stream's raw handle without building a Stream object (torch's
# own accessor where it exists; the public API otherwise)
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream: Optional[torch.cuda.Stream], device: Optional[int] = None):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_current_stream is not None and device is not None:
        return ctypes.c_void_p(_raw_current_stream(device))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ------------------------------------------------------------------ host-only

def conv_out_dims(x_shape, w_shape, stride=1, pad=0, dil=1) -> Tuple[int, ...]:
    """(N, Do, Ho, Wo, K) of the forward conv of x [N,D,H,W,C] by w [K,T,R,S,C]."""
    lib = load_library()
    out = _I64_5()
    _check(lib.conv_out_dims(_I64_5(*x_shape), _I64_5(*w_shape), _I32_3(*_triple(stride)),
                             _I32_3(*_triple(pad)), _I32_3(*_triple(dil)), out), "conv_out_dims")
    return tuple(int(v) for v in out)


def conv_fwd_plan(x_shape, w_shape, stride=1, pad=0, dil=1, dtype: int = CONV_DTYPE_BF16,
                  num_sms: int = 0) -> dict:
    """The plan conv_fwd runs: class, tile N, k-step bytes, stages, split-K, CTAs,
    workspace bytes.  ``num_sms > 0`` plans host-only for that SM count."""
    lib = load_library()
    v = [ctypes.c_int(0) for _ in range(6)]
    ws = ctypes.c_size_t(0)
    _check(lib.conv_fwd_plan(_I64_5(*x_shape), _I64_5(*w_shape), _I32_3(*_triple(stride)),
                             _I32_3(*_triple(pad)), _I32_3(*_triple(dil)), int(dtype),
                             int(num_sms), *[ctypes.byref(a) for a in v], ctypes.byref(ws)),
           "conv_fwd_plan")
    cls, bn, bk, st, sp, ctas = (a.value for a in v)
    return {"class": CLASS_NAMES.get(cls, str(cls)), "tile_n": bn, "k_bytes": bk, "stages": st,
            "splits": sp, "ctas": ctas, "workspace_bytes": int(ws.value)}


def conv_fwd_ncdhw_plan(x_shape, w_shape, stride=1, pad=0, dil=1,
                        dtype: int = CONV_DTYPE_BF16, num_sms: int = 0) -> dict:
    """conv_fwd_plan for conv_fwd_ncdhw: x_shape is (N, C, D, H, W)."""
    lib = load_library()
    v = [ctypes.c_int(0) for _ in range(6)]
    ws = ctypes.c_size_t(0)
    _check(lib.conv_fwd_ncdhw_plan(_I64_5(*x_shape), _I64_5(*w_shape), _I32_3(*_triple(stride)),
                                   _I32_3(*_triple(pad)), _I32_3(*_triple(dil)), int(dtype),
                                   int(num_sms), *[ctypes.byref(a) for a in v], ctypes.byref(ws)),
           "conv_fwd_ncdhw_plan")
    cls, bn, bk, st, sp, ctas = (a.value for a in v)
    return {"class": CLASS_NAMES.get(cls, str(cls)), "tile_n": bn, "k_bytes": bk, "stages": st,
            "splits": sp, "ctas": ctas, "workspace_bytes": int(ws.value)}


def conv_fwd_from_host_slices(x_shape, w_shape, stride=1, pad=0, dil=1,
                              dtype: int = CONV_DTYPE_BF16, num_sms: int = 0,
                              workspace_bytes: int = 0, chunks: int = 0) -> dict:
    """The slices conv_fwd_from_host cuts this problem into: per slice its
    output rows (lo, hi) and the input it reads, (whole, part, rows) = (n, d)
    planes [0, whole) entirely and rows [0, rows) of planes [whole, part);
    and the first slice's weight groups.  ``num_sms > 0`` plans host-only."""
    lib = load_library()
    n = ctypes.c_int(0)
    groups = ctypes.c_int(0)
    rows = (ctypes.c_int64 * 64)()
    reach = (ctypes.c_int64 * 96)()
    _check(lib.conv_fwd_from_host_slices(_I64_5(*x_shape), _I64_5(*w_shape),
                                         _I32_3(*_triple(stride)), _I32_3(*_triple(pad)),
                                         _I32_3(*_triple(dil)), int(dtype), int(num_sms),
                                         ctypes.c_size_t(int(workspace_bytes)), int(chunks),
                                         ctypes.byref(n), rows, reach, ctypes.byref(groups)),
           "conv_fwd_from_host_slices")
    k = n.value
    return {"rows": [(rows[2 * i], rows[2 * i + 1]) for i in range(k)],
            "reach": [(reach[3 * i], reach[3 * i + 1], reach[3 * i + 2]) for i in range(k)],
            "weight_groups": groups.value}


def conv_fwd_workspace_size(x_shape, w_shape, stride=1, pad=0, dil=1,
                            dtype: int = CONV_DTYPE_BF16) -> int:
    """Workspace bytes conv_fwd uses for this problem on the current device
    (0: none needed, or the problem is invalid / unsupported)."""
    lib = load_library()
    return int(lib.conv_fwd_workspace_size(_I64_5(*x_shape), _I64_5(*w_shape),
                                           _I32_3(*_triple(stride)), _I32_3(*_triple(pad)),
                                           _I32_3(*_triple(dil)), int(dtype)))


def conv_fwd_kernel_launches(x_shape, w_shape, stride=1, pad=0, dil=1,
                             dtype: int = CONV_DTYPE_BF16, workspace_bytes: int = 0) -> int:
    """Kernels one conv_fwd call launches for this problem and workspace."""
    lib = load_library()
    n = ctypes.c_int(0)
    _check(lib.conv_fwd_kernel_launches(_I64_5(*x_shape), _I64_5(*w_shape),
                                        _I32_3(*_triple(stride)), _I32_3(*_triple(pad)),
                                        _I32_3(*_triple(dil)), int(dtype), int(workspace_bytes),
                                        ctypes.byref(n)), "conv_fwd_kernel_launches")
    return int(n.value)


_current_overrides: dict = {}


def set_overrides(**fields) -> dict:
    """Install plan / path overrides for every later call (conv_set_overrides);
    no arguments restores the library's own choices.  Fields are those of
    conv_overrides; ``tile="BN,BK,stages,group_m,splits"`` is shorthand for
    the first five (0 or -1 in it keeps the plan's value).  Returns the
    overrides that were installed before."""
    global _current_overrides
    lib = load_library()
    vals = dict(fields)
    tile = vals.pop("tile", None)
    if tile is not None:
        for name, v in zip(OVERRIDE_FIELDS[:5], str(tile).split(",")):
            v = int(v)
            vals[name] = v if v > 0 else -1
    unknown = set(vals) - set(OVERRIDE_FIELDS)
    if unknown:
        raise ValueError(f"unknown override fields {sorted(unknown)}")
    o = _Overrides()
    lib.conv_default_overrides(ctypes.byref(o))
    for k, v in vals.items():
        setattr(o, k, -1 if v is None else int(v))
    _check(lib.conv_set_overrides(ctypes.byref(o)), "conv_set_overrides")
    old, _current_overrides = _current_overrides, {k: v for k, v in vals.items() if v is not None}
    _shape_cache.clear()   # plans (and so workspace sizes) may change with the overrides
    return old


@contextlib.contextmanager
def overrides(**fields):
    """Context manager: the given overrides on top of those already installed,
    restored on exit (for sweeps and tests)."""
    merged = dict(_current_overrides)
    tile = fields.pop("tile", None)
    if tile is not None:
        for name, v in zip(OVERRIDE_FIELDS[:5], str(tile).split(",")):
            merged[name] = int(v) if int(v) > 0 else None
    merged.update(fields)
    old = set_overrides(**merged)
    try:
        yield
    finally:
        set_overrides(**old)


def conv_set_wait_limit_ns(ns: int) -> None:
    load_library().conv_set_wait_limit_ns(int(ns))


def conv_get_device_status() -> int:
    """Synchronise the device, then read and clear its status word."""
    lib = load_library()
    v = ctypes.c_int(0)
    _check(lib.conv_get_device_status(ctypes.byref(v)), "conv_get_device_status")
    return int(v.value)


def conv_get_device_status_stream(stream: Optional[torch.cuda.Stream] = None) -> int:
    """After the work queued on ``stream`` (default: the current stream),
    read and clear the device status word; synchronises that stream only."""
    lib = load_library()
    v = ctypes.c_int(0)
    _check(lib.conv_get_device_status_stream(_stream_handle(stream), ctypes.byref(v)),
           "conv_get_device_status_stream")
    return int(v.value)


# ------------------------------------------------------------------ per-shape cache
# A forward call's output dims, its marshalled shape arguments and (when the
# caller gives no workspace) the plan's workspace size depend only on the
# shapes, stride / pad / dilation, dtype and device (and on the overrides,
# whose change clears the cache), so they are computed once per problem.
# A stale size could not change a result: the library plans within the
# workspace it is given.

class _FwdShape:
    __slots__ = ("od", "xd", "wd", "st", "pa", "di", "need")

    def __init__(self, x_shape, w_shape, st, pa, di):
        self.od = conv_out_dims(x_shape, w_shape, st, pa, di)
        self.xd, self.wd = _I64_5(*x_shape), _I64_5(*w_shape)
        self.st, self.pa, self.di = _I32_3(*st), _I32_3(*pa), _I32_3(*di)
        self.need = None


_shape_cache: dict = {}
_SHAPE_CACHE_MAX = 256


def _fwd_shape(x: torch.Tensor, w: torch.Tensor, stride, pad, dil, dtype: int) -> _FwdShape:
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    key = (tuple(x.shape), tuple(w.shape), st, pa, di, dtype, x.device.index)
    e = _shape_cache.get(key)
    if e is None:
        e = _FwdShape(key[0], key[1], st, pa, di)
        if len(_shape_cache) >= _SHAPE_CACHE_MAX:
            _shape_cache.clear()
        _shape_cache[key] = e
    return e


# ------------------------------------------------------------------ device calls

def conv_fwd(x: torch.Tensor, w: torch.Tensor, stride=1, pad=0, dil=1,
             scale_x: Optional[torch.Tensor] = None, scale_w: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None, split_k: bool = True,
             bias: Optional[torch.Tensor] = None, act: str = "none") -> torch.Tensor:
    """Forward conv: x NDHWC [N,D,H,W,C], w KTRSC [K,T,R,S,C] (both bf16, or
    both float8_e4m3fn with fp32 device scales) -> out NDHWC [N,Do,Ho,Wo,K]
    bf16, plus ``bias`` (fp32 [K], through conv_fwd_bias) when given, then
    ``act`` ("relu", "silu" or "gelu", through conv_fwd_bias_act).  A
    split-K workspace is taken from torch's allocator when the plan wants one
    and none is given (``split_k=False`` runs without)."""
    if act not in ACT_CODES:
        raise ValueError(f"act must be one of {sorted(ACT_CODES)}")
    lib = _lib or load_library()
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x must be [N,D,H,W,C] and w [K,T,R,S,C]")
    dtype = _dtype_code(x)
    if _dtype_code(w) != dtype:
        raise TypeError("x and w must have the same dtype")
    for s in (scale_x, scale_w):
        if s is not None and (s.dtype != torch.float32 or s.numel() < 1):
            raise TypeError("scales must be float32 device tensors")
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (w.shape[0],)):
        raise TypeError("bias must be a float32 device tensor of shape [K]")
    _require_cuda(x, w, scale_x, scale_w, out, workspace, bias)
    e = _fwd_shape(x, w, stride, pad, dil, dtype)
    if out is None:
        out = torch.empty(e.od, dtype=torch.bfloat16, device=x.device)
    elif tuple(out.shape) != e.od or out.dtype != torch.bfloat16:
        raise ValueError(f"out must be bf16 {e.od}")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    elif split_k:
        if e.need is None:
            e.need = conv_fwd_plan(tuple(x.shape), tuple(w.shape), stride, pad, dil,
                                   dtype)["workspace_bytes"]
        if e.need:
            workspace = torch.empty(e.need, dtype=torch.uint8, device=x.device)
            ws_ptr, ws_bytes = workspace.data_ptr(), e.need
    if act != "none":
        rc = lib.conv_fwd_bias_act(x.data_ptr(), e.xd, w.data_ptr(), e.wd, e.st, e.pa, e.di,
                                   dtype, _ptr(scale_x), _ptr(scale_w), _ptr(bias),
                                   ACT_CODES[act], out.data_ptr(), ws_ptr, ws_bytes,
                                   _stream_handle(stream, x.device.index))
        _check(rc, "conv_fwd_bias_act")
    elif bias is None:
        rc = lib.conv_fwd(x.data_ptr(), e.xd, w.data_ptr(), e.wd, e.st, e.pa, e.di, dtype,
                          _ptr(scale_x), _ptr(scale_w), out.data_ptr(), ws_ptr, ws_bytes,
                          _stream_handle(stream, x.device.index))
        _check(rc, "conv_fwd")
    else:
        rc = lib.conv_fwd_bias(x.data_ptr(), e.xd, w.data_ptr(), e.wd, e.st, e.pa, e.di, dtype,
                               _ptr(scale_x), _ptr(scale_w), bias.data_ptr(), out.data_ptr(),
                               ws_ptr, ws_bytes, _stream_handle(stream, x.device.index))
        _check(rc, "conv_fwd_bias")
    return out


def conv_fwd_ncdhw(x: torch.Tensor, w: torch.Tensor, stride=1, pad=0, dil=1,
                   scale_x: Optional[torch.Tensor] = None, scale_w: Optional[torch.Tensor] = None,
                   bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None,
                   split_k: bool = True) -> torch.Tensor:
    """Forward conv of a channel-major activation read in place: x NCDHW
    [N,C,D,H,W] bf16, w KTRSC [K,T,1,1,C] bf16 -> out NDHWC [N,Do,H,W,K] bf16
    (T x 1 x 1 filters, unit H/W stride, no H/W padding; H*W and C multiples
    of 8).  Other arguments as for conv_fwd."""
    lib = load_library()
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x must be [N,C,D,H,W] and w [K,T,R,S,C]")
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("conv_fwd_ncdhw takes bf16 x and w")
    for s in (scale_x, scale_w):
        if s is not None and (s.dtype != torch.float32 or s.numel() < 1):
            raise TypeError("scales must be float32 device tensors")
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (w.shape[0],)):
        raise TypeError("bias must be a float32 device tensor of shape [K]")
    _require_cuda(x, w, scale_x, scale_w, out, workspace, bias)
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    n, c, d, h, wd = (int(v) for v in x.shape)
    od = conv_out_dims((n, d, h, wd, c), tuple(w.shape), st, pa, di)
    if out is None:
        out = torch.empty(od, dtype=torch.bfloat16, device=x.device)
    elif tuple(out.shape) != od or out.dtype != torch.bfloat16:
        raise ValueError(f"out must be bf16 {od}")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    elif split_k:
        need = conv_fwd_ncdhw_plan(tuple(x.shape), tuple(w.shape), st, pa, di)["workspace_bytes"]
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
            ws_ptr, ws_bytes = workspace.data_ptr(), need
    rc = lib.conv_fwd_ncdhw(x.data_ptr(), _I64_5(*x.shape), w.data_ptr(), _I64_5(*w.shape),
                            _I32_3(*st), _I32_3(*pa), _I32_3(*di), CONV_DTYPE_BF16,
                            _ptr(scale_x), _ptr(scale_w), _ptr(bias), out.data_ptr(), ws_ptr,
                            ws_bytes, _stream_handle(stream))
    _check(rc, "conv_fwd_ncdhw")
    return out


def conv_fwd_ncdhw_fp8_workspace_size(x_shape, w_shape, stride=1, pad=0, dil=1) -> int:
    """Preferred workspace bytes of conv_fwd_ncdhw_fp8 (x_shape = N, C, D, H, W)."""
    lib = load_library()
    b = ctypes.c_size_t(0)
    _check(lib.conv_fwd_ncdhw_fp8_workspace_size(
        _I64_5(*x_shape), _I64_5(*w_shape), _I32_3(*_triple(stride)), _I32_3(*_triple(pad)),
        _I32_3(*_triple(dil)), ctypes.byref(b)), "conv_fwd_ncdhw_fp8_workspace_size")
    return int(b.value)


def conv_fwd_ncdhw_fp8(x: torch.Tensor, w: torch.Tensor, stride=1, pad=0, dil=1,
                       scale_w: Optional[torch.Tensor] = None,
                       scale_x: Optional[torch.Tensor] = None,
                       bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None):
    """e4m3 conv of a bf16 channel-major activation quantised while it is
    loaded: x NCDHW [N,C,D,H,W] bf16, w e4m3 KTRSC [K,1,R,S,C] with its fp32
    scale -> (out NDHWC [N,D,H,W,K] bf16, scale_x fp32[1] = amax(x)/448)."""
    lib = load_library()
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x must be [N,C,D,H,W] and w [K,T,R,S,C]")
    if x.dtype != torch.bfloat16 or w.dtype != torch.float8_e4m3fn:
        raise TypeError("conv_fwd_ncdhw_fp8 takes bf16 x and float8_e4m3fn w")
    for s in (scale_w, scale_x):
        if s is not None and (s.dtype != torch.float32 or s.numel() < 1):
            raise TypeError("scales must be float32 device tensors")
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (w.shape[0],)):
        raise TypeError("bias must be a float32 device tensor of shape [K]")
    _require_cuda(x, w, scale_w, scale_x, bias, out, workspace)
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    n, c, d, h, wd = (int(v) for v in x.shape)
    od = conv_out_dims((n, d, h, wd, c), tuple(w.shape), st, pa, di)
    if out is None:
        out = torch.empty(od, dtype=torch.bfloat16, device=x.device)
    elif tuple(out.shape) != od or out.dtype != torch.bfloat16:
        raise ValueError(f"out must be bf16 {od}")
    if scale_x is None:
        scale_x = torch.empty(1, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(conv_fwd_ncdhw_fp8_workspace_size(tuple(x.shape), tuple(w.shape),
                                                                  st, pa, di),
                                dtype=torch.uint8, device=x.device)
    rc = lib.conv_fwd_ncdhw_fp8(x.data_ptr(), _I64_5(*x.shape), w.data_ptr(), _I64_5(*w.shape),
                                _I32_3(*st), _I32_3(*pa), _I32_3(*di), _ptr(scale_w),
                                scale_x.data_ptr(), _ptr(bias), out.data_ptr(),
                                workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    _check(rc, "conv_fwd_ncdhw_fp8")
    return out, scale_x


def conv_fwd_noalloc(x: torch.Tensor, w: torch.Tensor, stride=1, pad=0, dil=1,
                     scale_x: Optional[torch.Tensor] = None,
                     scale_w: Optional[torch.Tensor] = None, out: torch.Tensor = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """conv_fwd for callers that cannot allocate device memory: the caller
    passes ``out`` (bf16, the output shape) and the library keeps any split-K
    partials in its own static device scratch (see include/conv3d.h for the
    size limit and the rule that overlapping calls race on that scratch)."""
    lib = load_library()
    if out is None:
        raise ValueError("conv_fwd_noalloc writes into a caller-provided out tensor")
    dtype = _dtype_code(x)
    if _dtype_code(w) != dtype:
        raise TypeError("x and w must have the same dtype")
    _require_cuda(x, w, scale_x, scale_w, out)
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    rc = lib.conv_fwd_noalloc(x.data_ptr(), _I64_5(*x.shape), w.data_ptr(), _I64_5(*w.shape),
                              _I32_3(*st), _I32_3(*pa), _I32_3(*di), dtype, _ptr(scale_x),
                              _ptr(scale_w), out.data_ptr(), _stream_handle(stream))
    _check(rc, "conv_fwd_noalloc")
    return out


def conv_fwd_from_host(x_host: torch.Tensor, w_host: torch.Tensor, stride=1, pad=0, dil=1,
                       scale_x: Optional[torch.Tensor] = None,
                       scale_w: Optional[torch.Tensor] = None,
                       out_host: Optional[torch.Tensor] = None,
                       x_dev: Optional[torch.Tensor] = None, w_dev: Optional[torch.Tensor] = None,
                       out_dev: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, chunks: int = 0,
                       stream: Optional[torch.cuda.Stream] = None,
                       device: Optional[torch.device] = None) -> torch.Tensor:
    """conv_fwd with x, w and the result in host memory (CPU tensors, pinned
    for the copies to overlap the convolution): the output rows are computed
    in slices whose input copies and output copies overlap the other slices'
    kernels.  Device buffers of the operands' sizes (and a workspace when the
    plan wants one) are taken from torch's allocator when not given.  Returns
    ``out_host``; synchronise the stream before reading it."""
    lib = load_library()
    if x_host.dim() != 5 or w_host.dim() != 5:
        raise ValueError("x must be [N,D,H,W,C] and w [K,T,R,S,C]")
    for t in (x_host, w_host, out_host):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host operands must be contiguous CPU tensors")
    dtype = _dtype_code(x_host)
    if _dtype_code(w_host) != dtype:
        raise TypeError("x and w must have the same dtype")
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    od = conv_out_dims(tuple(x_host.shape), tuple(w_host.shape), st, pa, di)
    if out_host is None:
        out_host = torch.empty(od, dtype=torch.bfloat16, pin_memory=True)
    elif tuple(out_host.shape) != od or out_host.dtype != torch.bfloat16:
        raise ValueError(f"out_host must be bf16 {od}")
    if x_dev is None:
        x_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
    if w_dev is None:
        w_dev = torch.empty(w_host.shape, dtype=w_host.dtype, device=dev)
    if out_dev is None:
        out_dev = torch.empty(od, dtype=torch.bfloat16, device=dev)
    for dv, h in ((x_dev, x_host), (w_dev, w_host), (out_dev, out_host)):
        if dv.numel() * dv.element_size() != h.numel() * h.element_size():
            raise ValueError("device buffers must match the host tensors' sizes")
    _require_cuda(x_dev, w_dev, out_dev, scale_x, scale_w, workspace)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    else:
        need = conv_fwd_plan(tuple(x_host.shape), tuple(w_host.shape), st, pa, di,
                             dtype)["workspace_bytes"]
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            ws_ptr, ws_bytes = workspace.data_ptr(), need
    rc = lib.conv_fwd_from_host(
        x_host.data_ptr(), _I64_5(*x_host.shape), w_host.data_ptr(), _I64_5(*w_host.shape),
        _I32_3(*st), _I32_3(*pa), _I32_3(*di), dtype, _ptr(scale_x), _ptr(scale_w),
        out_host.data_ptr(), x_dev.data_ptr(), w_dev.data_ptr(), out_dev.data_ptr(), ws_ptr,
        ws_bytes, int(chunks), _stream_handle(stream))
    _check(rc, "conv_fwd_from_host")
    return out_host


def conv_bwd_point_workspace_bytes(x_shape, w_shape, stride=1, pad=0, dil=1,
                                   which: int = 0) -> int:
    """Preferred workspace of conv_bwd_data_point (which=0) or
    conv_bwd_weight_point (which=1) on the current device."""
    lib = load_library()
    b = ctypes.c_size_t(0)
    _check(lib.conv_bwd_point_workspace_bytes(
        _I64_5(*x_shape), _I64_5(*w_shape), _I32_3(*_triple(stride)), _I32_3(*_triple(pad)),
        _I32_3(*_triple(dil)), int(which), ctypes.byref(b)), "conv_bwd_point_workspace_bytes")
    return int(b.value)


def _bwd_call(name, a, b, x_shape, w_shape, stride, pad, dil, out, workspace, stream, which):
    lib = load_library()
    for t in (a, b):
        if t.dtype != torch.bfloat16:
            raise TypeError("backward passes take bf16 tensors")
    _require_cuda(a, b, out, workspace)
    st, pa, di = _triple(stride), _triple(pad), _triple(dil)
    if workspace is None:
        need = conv_bwd_point_workspace_bytes(x_shape, w_shape, st, pa, di, which)
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    rc = getattr(lib, name)(a.data_ptr(), b.data_ptr(), _I64_5(*x_shape), _I64_5(*w_shape),
                            _I32_3(*st), _I32_3(*pa), _I32_3(*di), out.data_ptr(),
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream_handle(stream))
    _check(rc, name)
    return out


def conv_bwd_data_point(dy: torch.Tensor, w: torch.Tensor, x_shape, stride=1, pad=0, dil=1,
                        dx: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Backward data of a point-output conv: dx (x_shape, bf16) from dy
    [N,1,1,1,K] and w [K,T,R,S,C]."""
    if dx is None:
        dx = torch.empty(tuple(x_shape), dtype=torch.bfloat16, device=dy.device)
    return _bwd_call("conv_bwd_data_point", dy, w, x_shape, tuple(w.shape), stride, pad, dil,
                     dx, workspace, stream, 0)


def conv_bwd_weight_point(x: torch.Tensor, dy: torch.Tensor, w_shape, stride=1, pad=0, dil=1,
                          dw: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Backward weights of a point-output conv: dw (w_shape, bf16) from x
    [N,D,H,W,C] and dy [N,1,1,1,K]."""
    if dw is None:
        dw = torch.empty(tuple(w_shape), dtype=torch.bfloat16, device=x.device)
    return _bwd_call("conv_bwd_weight_point", x, dy, tuple(x.shape), w_shape, stride, pad, dil,
                     dw, workspace, stream, 1)


def pack_ncdhw_bf16_to_ndhwc(x: torch.Tensor, out: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """bf16 NCDHW [N,C,D,H,W] -> bf16 NDHWC [N,D,H,W,C] (a torch weight
    [K,C,T,R,S] gives the KTRSC weight)."""
    lib = load_library()
    if x.dim() != 5 or x.dtype != torch.bfloat16:
        raise ValueError("x must be a bf16 [N,C,D,H,W] tensor")
    N, C, D, H, W = x.shape
    if out is None:
        out = torch.empty((N, D, H, W, C), dtype=torch.bfloat16, device=x.device)
    _require_cuda(x, out)
    _check(lib.pack_ncdhw_bf16_to_ndhwc(x.data_ptr(), _I64_5(*x.shape), out.data_ptr(),
                                        _stream_handle(stream)), "pack_ncdhw_bf16_to_ndhwc")
    return out


def pack_ncdhw_bf16_to_ndhwc_fp8(x: torch.Tensor, out: Optional[torch.Tensor] = None,
                                 scale: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None,
                                 stream: Optional[torch.cuda.Stream] = None):
    """bf16 NCDHW -> (e4m3 NDHWC, fp32 scale[1]) with scale = amax/448."""
    lib = load_library()
    if x.dim() != 5 or x.dtype != torch.bfloat16:
        raise ValueError("x must be a bf16 [N,C,D,H,W] tensor")
    N, C, D, H, W = x.shape
    if out is None:
        out = torch.empty((N, D, H, W, C), dtype=torch.float8_e4m3fn, device=x.device)
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
    wsb = int(lib.pack_fp8_workspace_size())
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    _require_cuda(x, out, scale, workspace)
    _check(lib.pack_ncdhw_bf16_to_ndhwc_fp8(
        x.data_ptr(), _I64_5(*x.shape), out.data_ptr(), scale.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream)),
        "pack_ncdhw_bf16_to_ndhwc_fp8")
    return out, scale


# ------------------------------------------------------------------ wrappers

def conv3d(x, w, stride=1, padding=0, dilation=1, scale_x=None, scale_w=None, **kw):
    """conv_fwd under its usual name (NDHWC x, KTRSC w)."""
    return conv_fwd(x, w, stride, padding, dilation, scale_x, scale_w, **kw)


def conv2d(x, w, stride=1, padding=0, dilation=1, scale_x=None, scale_w=None, **kw):
    """NHWC x [N,H,W,C], KRSC w [K,R,S,C] -> NHWC [N,Ho,Wo,K], as the D=T=1 conv3d."""
    s = (stride, stride) if isinstance(stride, int) else tuple(stride)
    p = (padding, padding) if isinstance(padding, int) else tuple(padding)
    d = (dilation, dilation) if isinstance(dilation, int) else tuple(dilation)
    y = conv_fwd(x.unsqueeze(1), w.unsqueeze(1), (1,) + s, (0,) + p, (1,) + d, scale_x, scale_w,
                 **kw)
    return y.squeeze(1)


def conv1d(x, w, stride=1, padding=0, dilation=1, scale_x=None, scale_w=None, **kw):
    """NWC x [N,W,C], KSC w [K,S,C] -> NWC [N,Wo,K], as the D=T=H=R=1 conv3d."""
    s = stride if isinstance(stride, int) else int(stride[0])
    p = padding if isinstance(padding, int) else int(padding[0])
    d = dilation if isinstance(dilation, int) else int(dilation[0])
    y = conv_fwd(x[:, None, None], w[:, None, None], (1, 1, s), (0, 0, p), (1, 1, d), scale_x,
                 scale_w, **kw)
    return y[:, 0, 0]


__all__ = [
    "conv_fwd", "conv_fwd_noalloc", "conv_fwd_plan", "conv_out_dims", "conv_get_device_status",
    "conv_set_wait_limit_ns", "pack_ncdhw_bf16_to_ndhwc", "pack_ncdhw_bf16_to_ndhwc_fp8",
    "conv3d", "conv2d", "conv1d", "load_library", "ConvError", "LIB_PATH",
    "conv_fwd_from_host", "conv_fwd_from_host_slices", "conv_fwd_kernel_launches",
    "conv_fwd_ncdhw",
    "conv_fwd_ncdhw_plan", "conv_bwd_point_workspace_bytes", "conv_bwd_data_point",
    "conv_bwd_weight_point", "conv_fwd_workspace_size", "conv_get_device_status_stream",
    "set_overrides", "overrides", "conv_fwd_ncdhw_fp8", "conv_fwd_ncdhw_fp8_workspace_size",
]
