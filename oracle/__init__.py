"""CPU oracle for im2win convolution -- test infrastructure only.

Plain fp64 C (``oracle.c``) behind ctypes. Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package; the product library never does, and shares no code with it.

Each wrapper names the passage of the method it follows:

* ``conv_direct`` / ``conv_points`` -- direct convolution, the left column of
  Fig. 1 of "Enabling Memory-efficient Im2win Convolution with Multi-precision
  Support on GPU CUDA and Tensor Cores" (valid convolution, Table I shapes).
* ``im2win`` -- the im2win transformation, Abstract of "Im2win: Memory
  Efficient Convolution On SIMD Architectures" and Fig. 1 middle column.
* ``conv_im2win`` -- convolution as dot products over window segments (same).
* ``conv_im2col`` -- im2col + GEMM, Fig. 1 right column.
* ``im2win_nhwc`` / ``conv_im2win_nhwc`` -- the same two steps with channels
  innermost (x[N][H_i][W_i][C_i], win[N][H_o][W_i*H_f][C_i],
  out[N][H_o][W_o][C_o]); the [SIMD] page names a successor work on three
  tensor layouts by title only, and this is the plainest reading of it.
* ``conv_direct_nhwc`` / ``conv_points_nhwc`` -- the direct sums above on
  channels-last tensors: a transpose to NCHW, the NCHW routine, a transpose back.
* ``conv_direct_pd`` / ``conv_points_pd`` / ``im2win_pd`` / ``conv_im2win_pd``
  -- zero padding (p_h, p_w) and dilation (d_h, d_w), in either layout: the
  usual definitions of the two options (the pages' layers use neither), with
  the window row running over the W_i + 2 p_w padded columns.

Inputs are numpy arrays; floating inputs are widened to float64 exactly before
the call (the caller has already rounded them to the dtype under test).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_PD = ctypes.POINTER(ctypes.c_double)
_PI = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:3] + ["-fopenmp"] + base[3:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            shp = [_I64] * 9
            lib.oracle_conv_direct.argtypes = [_PD, _PD, _PD, _PD] + shp
            lib.oracle_conv_points.argtypes = [_PD, _PD, _PI, _I64, _PD, _PD] + shp
            lib.oracle_conv_im2win.argtypes = [_PD, _PD, _PD] + shp
            lib.oracle_conv_im2col.argtypes = [_PD, _PD, _PD] + shp
            lib.oracle_im2win.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [_I64] * 6
            lib.oracle_im2win_nhwc.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [_I64] * 6
            lib.oracle_conv_im2win_nhwc.argtypes = [_PD, _PD, _PD] + shp
            ci = ctypes.c_int
            lib.oracle_conv_direct_pd.argtypes = [_PD, _PD, _PD, _PD, ci] + shp + [_I64] * 4
            lib.oracle_conv_points_pd.argtypes = [_PD, _PD, _PI, _I64, _PD, _PD, ci] + shp + [_I64] * 4
            lib.oracle_im2win_pd.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64, ci] + [_I64] * 12
            lib.oracle_conv_im2win_pd.argtypes = [_PD, _PD, _PD, ci] + shp + [_I64] * 4
            for f in (lib.oracle_conv_direct, lib.oracle_conv_points, lib.oracle_conv_im2win,
                      lib.oracle_conv_im2col, lib.oracle_im2win, lib.oracle_im2win_nhwc,
                      lib.oracle_conv_im2win_nhwc, lib.oracle_conv_direct_pd, lib.oracle_conv_points_pd,
                      lib.oracle_im2win_pd, lib.oracle_conv_im2win_pd):
                f.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (1 without OpenMP)."""
    return int(_load().oracle_num_threads())


def out_shape(x_shape, w_shape, stride):
    n, ci, hi, wi = x_shape
    co, ci2, hf, wf = w_shape
    if ci != ci2:
        raise ValueError("channel mismatch")
    sh, sw = stride
    return (n, co, (hi - hf) // sh + 1, (wi - wf) // sw + 1)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _dp(a):
    return a.ctypes.data_as(_PD)


def _args(x, w, stride):
    n, ci, hi, wi = x.shape
    co, _, hf, wf = w.shape
    return [n, ci, hi, wi, co, hf, wf, stride[0], stride[1]]


def conv_direct(x, w, stride=(1, 1)):
    """Direct convolution in fp64; returns (out, S) with S = sum |x||w| per output."""
    x, w = _f64(x), _f64(w)
    shp = out_shape(x.shape, w.shape, stride)
    out = np.empty(shp, np.float64)
    scale = np.empty(shp, np.float64)
    rc = _load().oracle_conv_direct(_dp(x), _dp(w), _dp(out), _dp(scale), *_args(x, w, stride))
    if rc:
        raise ValueError("oracle_conv_direct: bad shape")
    return out, scale


def conv_points(x, w, idx, stride=(1, 1)):
    """Direct-sum outputs at coordinates idx[t] = (n, co, ho, wo); returns (vals, S)."""
    x, w = _f64(x), _f64(w)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1, 4))
    out = np.empty(len(idx), np.float64)
    scale = np.empty(len(idx), np.float64)
    rc = _load().oracle_conv_points(_dp(x), _dp(w), idx.ctypes.data_as(_PI), len(idx),
                                    _dp(out), _dp(scale), *_args(x, w, stride))
    if rc:
        raise ValueError("oracle_conv_points: bad shape or index")
    return out, scale


def im2win(x, H_f, s_h):
    """Window tensor win[n][ci][ho][w*H_f + r] = x[n][ci][ho*s_h + r][w], same dtype, byte copy."""
    x = np.ascontiguousarray(x)
    n, ci, hi, wi = x.shape
    ho = (hi - H_f) // s_h + 1
    win = np.empty((n, ci, ho, wi * H_f), dtype=x.dtype)
    rc = _load().oracle_im2win(x.ctypes.data, win.ctypes.data, x.dtype.itemsize,
                               n, ci, hi, wi, H_f, s_h)
    if rc:
        raise ValueError("oracle_im2win: bad shape")
    return win


def conv_im2win(x, w, stride=(1, 1)):
    """Convolution through the fp64 window tensor and the re-laid filter."""
    x, w = _f64(x), _f64(w)
    win = im2win(x, w.shape[2], stride[0])
    out = np.empty(out_shape(x.shape, w.shape, stride), np.float64)
    rc = _load().oracle_conv_im2win(_dp(win), _dp(w), _dp(out), *_args(x, w, stride))
    if rc:
        raise ValueError("oracle_conv_im2win: bad shape")
    return out


def conv_im2col(x, w, stride=(1, 1)):
    """Brute-force im2col + GEMM convolution in fp64 (small inputs)."""
    x, w = _f64(x), _f64(w)
    out = np.empty(out_shape(x.shape, w.shape, stride), np.float64)
    rc = _load().oracle_conv_im2col(_dp(x), _dp(w), _dp(out), *_args(x, w, stride))
    if rc:
        raise ValueError("oracle_conv_im2col: bad shape")
    return out


def workspace_elems(x_shape, w_shape, stride):
    """Element counts (input, window tensor, im2col matrix) for one problem."""
    n, ci, hi, wi = x_shape
    _, _, hf, wf = w_shape
    _, _, ho, wo = out_shape(x_shape, w_shape, stride)
    return n * ci * hi * wi, n * ci * ho * wi * hf, n * ci * hf * wf * ho * wo


# ---- channels-last (NHWC) layouts

def _nchw(a):
    return np.ascontiguousarray(np.transpose(a, (0, 3, 1, 2)))


def _nhwc(a):
    return np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))


def out_shape_nhwc(x_shape, w_shape, stride):
    n, hi, wi, ci = x_shape
    n2, co, ho, wo = out_shape((n, ci, hi, wi), w_shape, stride)
    return (n2, ho, wo, co)


def conv_direct_nhwc(x, w, stride=(1, 1)):
    """conv_direct on x[N][H_i][W_i][C_i]; returns (out, S) as [N][H_o][W_o][C_o]."""
    out, scale = conv_direct(_nchw(_f64(x)), w, stride)
    return _nhwc(out), _nhwc(scale)


def conv_points_nhwc(x, w, idx, stride=(1, 1)):
    """conv_points on x[N][H_i][W_i][C_i] at coordinates idx[t] = (n, ho, wo, co)."""
    idx = np.asarray(idx, dtype=np.int64).reshape(-1, 4)
    return conv_points(_nchw(_f64(x)), w, idx[:, [0, 3, 1, 2]], stride)


def im2win_nhwc(x, H_f, s_h):
    """Window tensor win[n][ho][w*H_f + r][c] = x[n][ho*s_h + r][w][c], same dtype, byte copy."""
    x = np.ascontiguousarray(x)
    n, hi, wi, ci = x.shape
    ho = (hi - H_f) // s_h + 1
    win = np.empty((n, ho, wi * H_f, ci), dtype=x.dtype)
    rc = _load().oracle_im2win_nhwc(x.ctypes.data, win.ctypes.data, x.dtype.itemsize,
                                    n, ci, hi, wi, H_f, s_h)
    if rc:
        raise ValueError("oracle_im2win_nhwc: bad shape")
    return win


def conv_im2win_nhwc(x, w, stride=(1, 1)):
    """Convolution through the fp64 channels-last window tensor; out[N][H_o][W_o][C_o]."""
    x, w = _f64(x), _f64(w)
    n, hi, wi, ci = x.shape
    win = im2win_nhwc(x, w.shape[2], stride[0])
    out = np.empty(out_shape_nhwc(x.shape, w.shape, stride), np.float64)
    co, _, hf, wf = w.shape
    rc = _load().oracle_conv_im2win_nhwc(_dp(win), _dp(w), _dp(out), n, ci, hi, wi, co, hf, wf,
                                         stride[0], stride[1])
    if rc:
        raise ValueError("oracle_conv_im2win_nhwc: bad shape")
    return out


# ---- zero padding and dilation (either layout)

def _dims(x_shape, layout):
    if layout == "nhwc":
        n, hi, wi, ci = x_shape
    else:
        n, ci, hi, wi = x_shape
    return n, ci, hi, wi


def out_shape_pd(x_shape, w_shape, stride, pad, dil, layout="nchw"):
    n, ci, hi, wi = _dims(x_shape, layout)
    co, ci2, hf, wf = w_shape
    if ci != ci2:
        raise ValueError("channel mismatch")
    ho = (hi + 2 * pad[0] - dil[0] * (hf - 1) - 1) // stride[0] + 1
    wo = (wi + 2 * pad[1] - dil[1] * (wf - 1) - 1) // stride[1] + 1
    return (n, ho, wo, co) if layout == "nhwc" else (n, co, ho, wo)


def _pd_args(x, w, stride, pad, dil, layout):
    n, ci, hi, wi = _dims(x.shape, layout)
    co, _, hf, wf = w.shape
    return [n, ci, hi, wi, co, hf, wf, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1]]


def conv_direct_pd(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), layout="nchw"):
    """Padded, dilated direct convolution in fp64; returns (out, S) in the layout of x."""
    x, w = _f64(x), _f64(w)
    shp = out_shape_pd(x.shape, w.shape, stride, pad, dil, layout)
    out = np.empty(shp, np.float64)
    scale = np.empty(shp, np.float64)
    rc = _load().oracle_conv_direct_pd(_dp(x), _dp(w), _dp(out), _dp(scale), int(layout == "nhwc"),
                                       *_pd_args(x, w, stride, pad, dil, layout))
    if rc:
        raise ValueError("oracle_conv_direct_pd: bad shape")
    return out, scale


def conv_points_pd(x, w, idx, stride=(1, 1), pad=(0, 0), dil=(1, 1), layout="nchw"):
    """The padded, dilated direct sum at idx[t] = (n, co, ho, wo) (NCHW output coordinates)."""
    x, w = _f64(x), _f64(w)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1, 4))
    out = np.empty(len(idx), np.float64)
    scale = np.empty(len(idx), np.float64)
    rc = _load().oracle_conv_points_pd(_dp(x), _dp(w), idx.ctypes.data_as(_PI), len(idx), _dp(out),
                                       _dp(scale), int(layout == "nhwc"),
                                       *_pd_args(x, w, stride, pad, dil, layout))
    if rc:
        raise ValueError("oracle_conv_points_pd: bad shape or index")
    return out, scale


def im2win_pd(x, w_shape, stride=(1, 1), pad=(0, 0), dil=(1, 1), layout="nchw"):
    """Window tensor of the padded input with row dilation, same dtype, byte copy:
    NCHW win[n][ci][ho][w*H_f + r], NHWC win[n][ho][w*H_f + r][ci], w < W_i + 2 p_w."""
    x = np.ascontiguousarray(x)
    n, ci, hi, wi = _dims(x.shape, layout)
    _, _, hf, wf = w_shape
    ho = (hi + 2 * pad[0] - dil[0] * (hf - 1) - 1) // stride[0] + 1
    wp = wi + 2 * pad[1]
    shp = (n, ho, wp * hf, ci) if layout == "nhwc" else (n, ci, ho, wp * hf)
    win = np.empty(shp, dtype=x.dtype)
    rc = _load().oracle_im2win_pd(x.ctypes.data, win.ctypes.data, x.dtype.itemsize, int(layout == "nhwc"),
                                  n, ci, hi, wi, hf, wf, stride[0], stride[1], pad[0], pad[1],
                                  dil[0], dil[1])
    if rc:
        raise ValueError("oracle_im2win_pd: bad shape")
    return win


def conv_im2win_pd(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), layout="nchw"):
    """Convolution through the fp64 padded window tensor (column runs at dilation d_w)."""
    x, w = _f64(x), _f64(w)
    win = im2win_pd(x, w.shape, stride, pad, dil, layout)
    out = np.empty(out_shape_pd(x.shape, w.shape, stride, pad, dil, layout), np.float64)
    rc = _load().oracle_conv_im2win_pd(_dp(win), _dp(w), _dp(out), int(layout == "nhwc"),
                                       *_pd_args(x, w, stride, pad, dil, layout))
    if rc:
        raise ValueError("oracle_conv_im2win_pd: bad shape")
    return out
