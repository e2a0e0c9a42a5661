"""ctypes binding of libim2win.so: argument marshalling only.

The functions named like the C entry points take torch tensors (device memory
owned by torch) and pass their data pointers, the shape arguments and the
current CUDA stream to the library; every step of the computation runs in the
library's kernels. There is no CPU path: if the library is missing, or the
tensors are not CUDA tensors, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)
OP_TRANSFORM, OP_CONV, OP_CONV_FUSED, OP_CONV_NHWC, OP_CONV_FUSED_NHWC = 0, 1, 2, 3, 4
F32, F16, BF16 = 0, 1, 2
NCHW, NHWC = 0, 1
_DTYPE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

EXPORTS = ("im2win_workspace_size", "im2win_transform", "im2win_conv", "im2win_conv_fused",
           "im2win_status_string", "im2win_device_status", "im2win_conv_fused_noalloc",
           "im2win_transform_nhwc", "im2win_conv_nhwc", "im2win_conv_fused_nhwc",
           "im2win_workspace_size_ex", "im2win_transform_ex", "im2win_conv_ex", "im2win_conv_fused_ex",
           "im2win_plan")
NOALLOC_SCRATCH_BYTES = 16 << 20
KERNEL_F32, KERNEL_TAP, KERNEL_EXPAND = 0, 1, 2


class PlanInfo(ctypes.Structure):
    """im2win_plan_info: the kernel and tiling a convolution call launches."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "kernel", "tap_mode", "stacked", "rows_per_tile", "pitch", "tmem_columns", "tmem_read_end",
        "smem_bytes", "filter_stage_taps", "filter_stages", "slab_stages", "reserved")] + [
        ("tiles", ctypes.c_int64), ("grid", ctypes.c_int64)]

_lock = threading.Lock()
_lib = None


class Im2winError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libim2win.so (built in-tree by build.build()); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with memory_efficient_cnn_gb300.build.build() "
                    "(nvcc, sm_103a); there is no fallback implementation")
            L = ctypes.CDLL(path)
            i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
            shp = [i64] * 9
            L.im2win_workspace_size.argtypes = [ctypes.c_int] + shp + [ctypes.c_int, ctypes.POINTER(sz)]
            L.im2win_transform.argtypes = [vp, vp] + shp + [ctypes.c_int, vp]
            L.im2win_conv.argtypes = [vp, vp, vp, vp, sz] + shp + [ctypes.c_int, vp]
            L.im2win_conv_fused.argtypes = [vp, vp, vp, vp, sz] + shp + [ctypes.c_int, vp]
            L.im2win_status_string.argtypes = [ctypes.c_int]
            L.im2win_status_string.restype = ctypes.c_char_p
            L.im2win_device_status.argtypes = [vp, sz, vp]
            L.im2win_conv_fused_noalloc.argtypes = [vp, vp, vp] + shp + [ctypes.c_int, vp]
            L.im2win_transform_nhwc.argtypes = [vp, vp] + shp + [ctypes.c_int, vp]
            L.im2win_conv_nhwc.argtypes = [vp, vp, vp, vp, sz] + shp + [ctypes.c_int, vp]
            L.im2win_conv_fused_nhwc.argtypes = [vp, vp, vp, vp, sz] + shp + [ctypes.c_int, vp]
            pd = [i64] * 4 + [ctypes.c_int, ctypes.c_int]  # p_h, p_w, d_h, d_w, layout, dtype
            L.im2win_workspace_size_ex.argtypes = [ctypes.c_int] + shp + pd + [ctypes.POINTER(sz)]
            L.im2win_transform_ex.argtypes = [vp, vp] + shp + pd + [vp]
            L.im2win_conv_ex.argtypes = [vp, vp, vp, vp, sz] + shp + pd + [vp]
            L.im2win_conv_fused_ex.argtypes = [vp, vp, vp, vp, sz] + shp + pd + [vp]
            L.im2win_plan.argtypes = [ctypes.c_int] + shp + pd + [ctypes.c_int, ctypes.POINTER(PlanInfo)]
            for f in ("im2win_workspace_size", "im2win_transform", "im2win_conv",
                      "im2win_conv_fused", "im2win_device_status", "im2win_conv_fused_noalloc",
                      "im2win_transform_nhwc", "im2win_conv_nhwc", "im2win_conv_fused_nhwc",
                      "im2win_workspace_size_ex", "im2win_transform_ex", "im2win_conv_ex",
                      "im2win_conv_fused_ex", "im2win_plan"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().im2win_status_string(int(status)).decode()


im2win_status_string = status_string


def _check(fn, status):
    if status != OK:
        raise Im2winError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32, float16 or bfloat16") from None


def _cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("im2win tensors must be CUDA tensors (no CPU implementation exists)")
        if not t.is_contiguous():
            raise ValueError("im2win tensors must be contiguous")


def _same_device(fn, *ts):
    dev = ts[0].device
    for t in ts[1:]:
        if t.device != dev:
            raise ValueError(f"{fn}: every tensor must be on one device ({dev} and {t.device} given)")


def _check_conv(fn, src, filt, out, ws, dims, C_o, H_f, W_f, stride, pad=(0, 0), dil=(1, 1),
                layout=NCHW, window=False):
    """Shape and device checks of a convolution call, made before anything is
    launched: the filter must be C_o x C_i x H_f x W_f, `out` must have the
    output's exact shape in `layout`, the source must hold at least the input
    (fused) or window tensor (window=True) of `dims` = (N, C_i, H_i, W_i), and
    every tensor must be on one device. A mismatch raises ValueError; the
    library itself checks the workspace size. An empty batch (N = 0) reads and
    writes nothing, so its buffers are not checked."""
    N, C_i, H_i, W_i = (int(v) for v in dims)
    if filt.dim() != 4 or tuple(filt.shape) != (C_o, C_i, H_f, W_f):
        raise ValueError(f"{fn}: filt has shape {tuple(filt.shape)}, expected {(C_o, C_i, H_f, W_f)}")
    H_o, W_o = out_hw_pd(H_i, W_i, H_f, W_f, stride, pad, dil)
    if N > 0 and H_o >= 1 and W_o >= 1:
        want = (N, H_o, W_o, C_o) if layout == NHWC else (N, C_o, H_o, W_o)
        if tuple(out.shape) != want:
            raise ValueError(f"{fn}: out has shape {tuple(out.shape)}, expected {want}")
        elems = N * C_i * H_o * (W_i + 2 * pad[1]) * H_f if window else N * C_i * H_i * W_i
        if src.numel() < elems:
            what = "window tensor" if window else "input"
            raise ValueError(f"{fn}: the {what} has {src.numel()} elements, expected {elems}")
    _same_device(fn, src, filt, out, *([ws] if ws is not None else []))


def _check_transform(fn, x, win, dims):
    if x.numel() < int(dims[0]) * int(dims[1]) * int(dims[2]) * int(dims[3]):
        raise ValueError(f"{fn}: x has {x.numel()} elements, expected N*C_i*H_i*W_i of {tuple(dims)}")
    _same_device(fn, x, win)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def out_hw(H_i, W_i, H_f, W_f, s_h, s_w):
    """Valid-convolution output extent (no padding)."""
    return (H_i - H_f) // s_h + 1, (W_i - W_f) // s_w + 1


def im2win_workspace_size(op: int, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    _check("im2win_workspace_size",
           lib().im2win_workspace_size(op, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, dtype,
                                       ctypes.byref(out)))
    return out.value


def im2win_transform(x: torch.Tensor, win: torch.Tensor, C_o, H_f, W_f, s_h, s_w) -> None:
    N, C_i, H_i, W_i = x.shape
    _check_transform("im2win_transform", x, win, x.shape)
    _cuda(x, win)
    if win.dtype != x.dtype:
        raise TypeError("win must have the dtype of x")
    need = im2win_workspace_size(OP_TRANSFORM, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                                 _dtype_code(x))
    if win.numel() * win.element_size() < need:
        raise ValueError("win is smaller than the window tensor")
    _check("im2win_transform",
           lib().im2win_transform(x.data_ptr(), win.data_ptr(), N, C_i, H_i, W_i, C_o, H_f, W_f,
                                  s_h, s_w, _dtype_code(x), _stream(x)))


def im2win_conv(win: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w) -> None:
    _check_conv("im2win_conv", win, filt, out, ws, (N, C_i, H_i, W_i), C_o, H_f, W_f, (s_h, s_w),
                window=True)
    _cuda(win, filt, out, ws)
    if not (win.dtype == filt.dtype == out.dtype):
        raise TypeError("win, filt and out must share a dtype")
    _check("im2win_conv",
           lib().im2win_conv(win.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                             ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f, W_f,
                             s_h, s_w, _dtype_code(win), _stream(win)))


def im2win_conv_fused(x: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                      s_h, s_w) -> None:
    N, C_i, H_i, W_i = x.shape
    C_o, _, H_f, W_f = filt.shape
    _check_conv("im2win_conv_fused", x, filt, out, ws, x.shape, C_o, H_f, W_f, (s_h, s_w))
    _cuda(x, filt, out, ws)
    if not (x.dtype == filt.dtype == out.dtype):
        raise TypeError("x, filt and out must share a dtype")
    _check("im2win_conv_fused",
           lib().im2win_conv_fused(x.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                   ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f,
                                   W_f, s_h, s_w, _dtype_code(x), _stream(x)))


def im2win_conv_fused_noalloc(x: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, s_h, s_w) -> None:
    """Fused convolution for callers that cannot allocate a workspace: the
    scratch is the library's built-in array (see include/im2win.h)."""
    N, C_i, H_i, W_i = x.shape
    C_o, _, H_f, W_f = filt.shape
    _check_conv("im2win_conv_fused_noalloc", x, filt, out, None, x.shape, C_o, H_f, W_f, (s_h, s_w))
    _cuda(x, filt, out)
    if not (x.dtype == filt.dtype == out.dtype):
        raise TypeError("x, filt and out must share a dtype")
    _check("im2win_conv_fused_noalloc",
           lib().im2win_conv_fused_noalloc(x.data_ptr(), filt.data_ptr(), out.data_ptr(), N, C_i,
                                           H_i, W_i, C_o, H_f, W_f, s_h, s_w, _dtype_code(x),
                                           _stream(x)))


def im2win_transform_nhwc(x: torch.Tensor, win: torch.Tensor, C_o, H_f, W_f, s_h, s_w) -> None:
    """Channels-last window transform: x[N][H_i][W_i][C_i] -> win[N][H_o][W_i*H_f][C_i]."""
    N, H_i, W_i, C_i = x.shape
    _check_transform("im2win_transform_nhwc", x, win, x.shape)
    _cuda(x, win)
    if win.dtype != x.dtype:
        raise TypeError("win must have the dtype of x")
    need = im2win_workspace_size(OP_TRANSFORM, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                                 _dtype_code(x))
    if win.numel() * win.element_size() < need:
        raise ValueError("win is smaller than the window tensor")
    _check("im2win_transform_nhwc",
           lib().im2win_transform_nhwc(x.data_ptr(), win.data_ptr(), N, C_i, H_i, W_i, C_o, H_f,
                                       W_f, s_h, s_w, _dtype_code(x), _stream(x)))


def im2win_conv_nhwc(win: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                     N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w) -> None:
    """Convolution from the channels-last window tensor into out[N][H_o][W_o][C_o]."""
    _check_conv("im2win_conv_nhwc", win, filt, out, ws, (N, C_i, H_i, W_i), C_o, H_f, W_f, (s_h, s_w),
                layout=NHWC, window=True)
    _cuda(win, filt, out, ws)
    if not (win.dtype == filt.dtype == out.dtype):
        raise TypeError("win, filt and out must share a dtype")
    _check("im2win_conv_nhwc",
           lib().im2win_conv_nhwc(win.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f, W_f,
                                  s_h, s_w, _dtype_code(win), _stream(win)))


def im2win_conv_fused_nhwc(x: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                           s_h, s_w) -> None:
    """Fused convolution of x[N][H_i][W_i][C_i] into out[N][H_o][W_o][C_o]."""
    N, H_i, W_i, C_i = x.shape
    C_o, _, H_f, W_f = filt.shape
    _check_conv("im2win_conv_fused_nhwc", x, filt, out, ws, (N, C_i, H_i, W_i), C_o, H_f, W_f, (s_h, s_w),
                layout=NHWC)
    _cuda(x, filt, out, ws)
    if not (x.dtype == filt.dtype == out.dtype):
        raise TypeError("x, filt and out must share a dtype")
    _check("im2win_conv_fused_nhwc",
           lib().im2win_conv_fused_nhwc(x.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                        ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f,
                                        W_f, s_h, s_w, _dtype_code(x), _stream(x)))


def im2win_workspace_size_ex(op: int, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w,
                             layout: int, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    _check("im2win_workspace_size_ex",
           lib().im2win_workspace_size_ex(op, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w,
                                          layout, dtype, ctypes.byref(out)))
    return out.value


def im2win_transform_ex(x: torch.Tensor, win: torch.Tensor, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                        p_h, p_w, d_h, d_w, layout: int) -> None:
    _check_transform("im2win_transform_ex", x, win, (N, C_i, H_i, W_i))
    _cuda(x, win)
    if win.dtype != x.dtype:
        raise TypeError("win must have the dtype of x")
    need = im2win_workspace_size_ex(OP_TRANSFORM, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w,
                                    d_h, d_w, layout, _dtype_code(x))
    if win.numel() * win.element_size() < need:
        raise ValueError("win is smaller than the window tensor")
    _check("im2win_transform_ex",
           lib().im2win_transform_ex(x.data_ptr(), win.data_ptr(), N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                                     p_h, p_w, d_h, d_w, layout, _dtype_code(x), _stream(x)))


def im2win_conv_ex(win: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                   N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w, layout: int) -> None:
    _check_conv("im2win_conv_ex", win, filt, out, ws, (N, C_i, H_i, W_i), C_o, H_f, W_f, (s_h, s_w),
                (p_h, p_w), (d_h, d_w), layout, window=True)
    _cuda(win, filt, out, ws)
    if not (win.dtype == filt.dtype == out.dtype):
        raise TypeError("win, filt and out must share a dtype")
    _check("im2win_conv_ex",
           lib().im2win_conv_ex(win.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                                p_h, p_w, d_h, d_w, layout, _dtype_code(win), _stream(win)))


def im2win_conv_fused_ex(x: torch.Tensor, filt: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                         N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w, layout: int) -> None:
    _check_conv("im2win_conv_fused_ex", x, filt, out, ws, (N, C_i, H_i, W_i), C_o, H_f, W_f, (s_h, s_w),
                (p_h, p_w), (d_h, d_w), layout)
    _cuda(x, filt, out, ws)
    if not (x.dtype == filt.dtype == out.dtype):
        raise TypeError("x, filt and out must share a dtype")
    _check("im2win_conv_fused_ex",
           lib().im2win_conv_fused_ex(x.data_ptr(), filt.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                      ws.numel() * ws.element_size(), N, C_i, H_i, W_i, C_o, H_f, W_f, s_h,
                                      s_w, p_h, p_w, d_h, d_w, layout, _dtype_code(x), _stream(x)))


def im2win_plan(op: int, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h=0, p_w=0, d_h=1, d_w=1,
                layout: int = NCHW, dtype: int = F16, sms: int = 0) -> dict:
    """Kernel and tiling of a convolution call (host only, no device needed);
    op OP_CONV (from the window tensor) or OP_CONV_FUSED. Raises Im2winError
    where the call would fail."""
    info = PlanInfo()
    _check("im2win_plan", lib().im2win_plan(op, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w,
                                            layout, dtype, sms, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_ if name != "reserved"}


def im2win_device_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream and return the status word of `ws`."""
    _cuda(ws)
    return lib().im2win_device_status(ws.data_ptr(), ws.numel() * ws.element_size(), _stream(ws))


# ---------------------------------------------------------------- conveniences
def workspace(op: int, x_shape, w_shape, stride, dtype: torch.dtype, device) -> torch.Tensor:
    """Allocate (through torch) the workspace `op` needs; x_shape is given as
    (N, C_i, H_i, W_i) in either layout."""
    N, C_i, H_i, W_i = x_shape
    C_o, _, H_f, W_f = w_shape
    b = im2win_workspace_size(op, N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0], stride[1],
                              _DTYPE[dtype])
    return torch.empty(max(b, 16), dtype=torch.uint8, device=device)


def transform(x: torch.Tensor, H_f: int, s_h: int = 1) -> torch.Tensor:
    """Window tensor win[N][C_i][H_o][W_i*H_f] of x."""
    N, C_i, H_i, W_i = x.shape
    H_o = (H_i - H_f) // s_h + 1
    win = torch.empty((N, C_i, H_o, W_i * H_f), dtype=x.dtype, device=x.device)
    im2win_transform(x, win, 1, H_f, 1, s_h, 1)
    return win


def conv(win: torch.Tensor, filt: torch.Tensor, stride=(1, 1), ws: torch.Tensor | None = None,
         out: torch.Tensor | None = None) -> torch.Tensor:
    """Convolution from a window tensor produced by transform()."""
    N, C_i, H_o, L = win.shape
    C_o, _, H_f, W_f = filt.shape
    W_i = L // H_f
    H_i = (H_o - 1) * stride[0] + H_f
    _, W_o = out_hw(H_i, W_i, H_f, W_f, *stride)
    if ws is None:
        ws = workspace(OP_CONV, (N, C_i, H_i, W_i), filt.shape, stride, win.dtype, win.device)
    if out is None:
        out = torch.empty((N, C_o, H_o, W_o), dtype=win.dtype, device=win.device)
    im2win_conv(win, filt, out, ws, N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0], stride[1])
    return out


def conv_fused(x: torch.Tensor, filt: torch.Tensor, stride=(1, 1), ws: torch.Tensor | None = None,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """Fused im2win convolution straight from the NCHW input."""
    N, C_i, H_i, W_i = x.shape
    C_o, _, H_f, W_f = filt.shape
    H_o, W_o = out_hw(H_i, W_i, H_f, W_f, *stride)
    if ws is None:
        ws = workspace(OP_CONV_FUSED, x.shape, filt.shape, stride, x.dtype, x.device)
    if out is None:
        out = torch.empty((N, C_o, H_o, W_o), dtype=x.dtype, device=x.device)
    im2win_conv_fused(x, filt, out, ws, stride[0], stride[1])
    return out


def transform_nhwc(x: torch.Tensor, H_f: int, s_h: int = 1) -> torch.Tensor:
    """Channels-last window tensor win[N][H_o][W_i*H_f][C_i] of x[N][H_i][W_i][C_i]."""
    N, H_i, W_i, C_i = x.shape
    H_o = (H_i - H_f) // s_h + 1
    win = torch.empty((N, H_o, W_i * H_f, C_i), dtype=x.dtype, device=x.device)
    im2win_transform_nhwc(x, win, 1, H_f, 1, s_h, 1)
    return win


def conv_nhwc(win: torch.Tensor, filt: torch.Tensor, stride=(1, 1), ws: torch.Tensor | None = None,
              out: torch.Tensor | None = None) -> torch.Tensor:
    """Convolution from a channels-last window tensor produced by transform_nhwc()."""
    N, H_o, L, C_i = win.shape
    C_o, _, H_f, W_f = filt.shape
    W_i = L // H_f
    H_i = (H_o - 1) * stride[0] + H_f
    _, W_o = out_hw(H_i, W_i, H_f, W_f, *stride)
    if ws is None:
        ws = workspace(OP_CONV_NHWC, (N, C_i, H_i, W_i), filt.shape, stride, win.dtype, win.device)
    if out is None:
        out = torch.empty((N, H_o, W_o, C_o), dtype=win.dtype, device=win.device)
    im2win_conv_nhwc(win, filt, out, ws, N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0], stride[1])
    return out


def conv_fused_nhwc(x: torch.Tensor, filt: torch.Tensor, stride=(1, 1), ws: torch.Tensor | None = None,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """Fused im2win convolution straight from the NHWC input; out[N][H_o][W_o][C_o]."""
    N, H_i, W_i, C_i = x.shape
    C_o, _, H_f, W_f = filt.shape
    H_o, W_o = out_hw(H_i, W_i, H_f, W_f, *stride)
    if ws is None:
        ws = workspace(OP_CONV_FUSED_NHWC, (N, C_i, H_i, W_i), filt.shape, stride, x.dtype, x.device)
    if out is None:
        out = torch.empty((N, H_o, W_o, C_o), dtype=x.dtype, device=x.device)
    im2win_conv_fused_nhwc(x, filt, out, ws, stride[0], stride[1])
    return out


# ---------------------------------------------------------------- padding / dilation
def _pd_dims(x_shape, layout):
    if layout == NHWC:
        N, H_i, W_i, C_i = x_shape
    else:
        N, C_i, H_i, W_i = x_shape
    return N, C_i, H_i, W_i


def out_hw_pd(H_i, W_i, H_f, W_f, stride, pad, dil):
    """Output extent with zero padding and dilation."""
    return ((H_i + 2 * pad[0] - dil[0] * (H_f - 1) - 1) // stride[0] + 1,
            (W_i + 2 * pad[1] - dil[1] * (W_f - 1) - 1) // stride[1] + 1)


def transform_ex(x: torch.Tensor, H_f: int, W_f: int, stride=(1, 1), pad=(0, 0), dil=(1, 1),
                 layout: int = NCHW) -> torch.Tensor:
    """Window tensor of the padded input with row dilation (W_i + 2 p_w columns)."""
    N, C_i, H_i, W_i = _pd_dims(x.shape, layout)
    H_o, _ = out_hw_pd(H_i, W_i, H_f, W_f, stride, pad, dil)
    L = (W_i + 2 * pad[1]) * H_f
    shape = (N, H_o, L, C_i) if layout == NHWC else (N, C_i, H_o, L)
    win = torch.empty(shape, dtype=x.dtype, device=x.device)
    im2win_transform_ex(x, win, N, C_i, H_i, W_i, 1, H_f, W_f, stride[0], stride[1], pad[0], pad[1],
                        dil[0], dil[1], layout)
    return win


def conv_ex(win: torch.Tensor, filt: torch.Tensor, x_shape, stride=(1, 1), pad=(0, 0), dil=(1, 1),
            layout: int = NCHW, ws: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Convolution from a window tensor produced by transform_ex(); x_shape is the
    input's shape in `layout`."""
    N, C_i, H_i, W_i = _pd_dims(x_shape, layout)
    C_o, _, H_f, W_f = filt.shape
    H_o, W_o = out_hw_pd(H_i, W_i, H_f, W_f, stride, pad, dil)
    args = (N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1])
    if ws is None:
        b = im2win_workspace_size_ex(OP_CONV, *args, layout, _DTYPE[win.dtype])
        ws = torch.empty(max(b, 16), dtype=torch.uint8, device=win.device)
    if out is None:
        shape = (N, H_o, W_o, C_o) if layout == NHWC else (N, C_o, H_o, W_o)
        out = torch.empty(shape, dtype=win.dtype, device=win.device)
    im2win_conv_ex(win, filt, out, ws, *args, layout)
    return out


def conv_fused_ex(x: torch.Tensor, filt: torch.Tensor, stride=(1, 1), pad=(0, 0), dil=(1, 1),
                  layout: int = NCHW, ws: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Fused convolution with zero padding and dilation, straight from x."""
    N, C_i, H_i, W_i = _pd_dims(x.shape, layout)
    C_o, _, H_f, W_f = filt.shape
    H_o, W_o = out_hw_pd(H_i, W_i, H_f, W_f, stride, pad, dil)
    args = (N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1])
    if ws is None:
        b = im2win_workspace_size_ex(OP_CONV_FUSED, *args, layout, _DTYPE[x.dtype])
        ws = torch.empty(max(b, 16), dtype=torch.uint8, device=x.device)
    if out is None:
        shape = (N, H_o, W_o, C_o) if layout == NHWC else (N, C_o, H_o, W_o)
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    im2win_conv_fused_ex(x, filt, out, ws, *args, layout)
    return out
