"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every entry point include/im2win.h declares; workspace sizes and
argument errors are answered on the host without touching a device."""
import ctypes
import os
import re

import pytest

import memory_efficient_cnn_gb300 as mec
from memory_efficient_cnn_gb300 import build as mbuild
from memory_efficient_cnn_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "im2win.h")


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mec.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(im2win_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(mec.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert mec.status_string(0) == "ok"
    assert "timed out" in mec.status_string(mec._binding.ERR_TIMEOUT)
    assert mec.status_string(999) == "unknown status"


def _win_elems(layer):
    ho = (layer.H_i - layer.H_f) // layer.s_h + 1
    return layer.N * layer.C_i * ho * layer.W_i * layer.H_f


@pytest.mark.parametrize("layer", wl.ALL, ids=lambda l: l.name)
def test_transform_size_is_the_window_tensor(lib, layer):
    for dt, esz in ((mec.F32, 4), (mec.F16, 2), (mec.BF16, 2)):
        b = mec.im2win_workspace_size(mec.OP_TRANSFORM, *layer.shape_args, dt)
        assert b == _win_elems(layer) * esz


@pytest.mark.parametrize("layer", wl.ALL, ids=lambda l: l.name)
def test_conv_workspaces_hold_status_and_filter_only(lib, layer):
    for dt, esz in ((mec.F32, 4), (mec.F16, 2), (mec.BF16, 2)):
        for op in (mec.OP_CONV, mec.OP_CONV_FUSED, mec.OP_CONV_NHWC, mec.OP_CONV_FUSED_NHWC):
            b = mec.im2win_workspace_size(op, *layer.shape_args, dt)
            filt = layer.C_o * layer.C_i * layer.H_f * layer.W_f * esz
            assert b % 256 == 0 and b >= 256 + filt
            # far below the window tensor on every benchmark layer but 1x1
            if layer.H_f > 1:
                assert b < _win_elems(layer) * esz


def test_argument_errors_on_host(lib):
    L = lib
    sz = ctypes.c_size_t()
    args = [1, 3, 8, 8, 4, 3, 3, 1, 1]
    assert L.im2win_workspace_size(0, *args, 0, None) == mec._binding.ERR_INVALID_ARG
    assert L.im2win_workspace_size(7, *args, 0, ctypes.byref(sz)) == mec._binding.ERR_INVALID_ARG
    assert L.im2win_workspace_size(0, *args, 9, ctypes.byref(sz)) == mec._binding.ERR_INVALID_ARG
    bad = [1, 3, 8, 8, 4, 9, 3, 1, 1]  # H_f > H_i
    assert L.im2win_workspace_size(0, *bad, 0, ctypes.byref(sz)) == mec._binding.ERR_INVALID_ARG
    zero_stride = [1, 3, 8, 8, 4, 3, 3, 0, 1]
    assert L.im2win_workspace_size(0, *zero_stride, 0, ctypes.byref(sz)) == mec._binding.ERR_INVALID_ARG
    # null / misaligned pointers are rejected before any device work
    assert L.im2win_transform(None, 256, *args, 0, None) == mec._binding.ERR_INVALID_ARG
    assert L.im2win_transform(1024 + 4, 2048, *args, 0, None) == mec._binding.ERR_MISALIGNED
    assert L.im2win_conv(1024, 2048, 4096, None, 0, *args, 1, None) == mec._binding.ERR_WORKSPACE
    assert L.im2win_conv_fused(1024, 2048, 4096, 8192, 16, *args, 1, None) == mec._binding.ERR_WORKSPACE
    assert L.im2win_conv(1024, 2050, 4096, 8192, 1 << 20, *args, 0, None) == mec._binding.ERR_MISALIGNED
    assert L.im2win_device_status(None, 256, None) == mec._binding.ERR_WORKSPACE


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 3, 8, 8)
    with pytest.raises(ValueError, match="CUDA"):
        mec.transform(x, 3, 1)


def test_ex_workspace_sizes_and_argument_errors(lib):
    sz = ctypes.c_size_t()
    L = lib
    base = [2, 16, 20, 21, 32, 3, 3, 1, 1]
    # padding widens the window rows: N*C_i*H_o*(W_i + 2 p_w)*H_f elements
    b = mec.im2win_workspace_size_ex(mec.OP_TRANSFORM, *base, 1, 2, 1, 1, mec.NCHW, mec.F16)
    assert b == 2 * 16 * 20 * (21 + 4) * 3 * 2
    b = mec.im2win_workspace_size_ex(mec.OP_TRANSFORM, *base, 0, 0, 2, 1, mec.NHWC, mec.F32)
    assert b == 2 * 16 * 16 * 21 * 3 * 4  # dilation 2: H_o = 20 - 4
    # with p = 0 and d = 1 the sizes equal the valid calls'
    for op, op_plain in ((mec.OP_CONV, mec.OP_CONV), (mec.OP_CONV_FUSED, mec.OP_CONV_FUSED)):
        for dt in (mec.F32, mec.F16):
            assert (mec.im2win_workspace_size_ex(op, *base, 0, 0, 1, 1, mec.NCHW, dt)
                    == mec.im2win_workspace_size(op_plain, *base, dt))
    for op in (mec.OP_CONV, mec.OP_CONV_FUSED):
        for lo in (mec.NCHW, mec.NHWC):
            for dt in (mec.F32, mec.F16, mec.BF16):
                b = mec.im2win_workspace_size_ex(op, *base, 1, 1, 2, 2, lo, dt)
                assert b % 256 == 0 and b >= 256 + 32 * 16 * 9 * (4 if dt == mec.F32 else 2)
    bad = mec._binding.ERR_INVALID_ARG
    pd = [ctypes.c_int64(v) for v in (1, 1, 1, 1)]
    assert L.im2win_workspace_size_ex(0, *base, *pd, 7, 0, ctypes.byref(sz)) == bad   # layout
    assert L.im2win_workspace_size_ex(0, *base, -1, 0, 1, 1, 0, 0, ctypes.byref(sz)) == bad
    assert L.im2win_workspace_size_ex(0, *base, 0, 0, 0, 1, 0, 0, ctypes.byref(sz)) == bad
    # the dilated filter (7 rows) does not fit 20 + 2*0 rows? it does; 11 rows of d=10 do not
    assert L.im2win_workspace_size_ex(0, *base[:5], 3, 3, 1, 1, 0, 0, 10, 1, 0, 0,
                                      ctypes.byref(sz)) == bad
    assert L.im2win_transform_ex(None, 256, *base, 0, 0, 1, 1, 0, 0, None) == bad
    assert L.im2win_conv_fused_ex(1024 + 4, 2048, 4096, 8192, 1 << 20, *base, 0, 0, 1, 1, 0, 1,
                                  None) == mec._binding.ERR_MISALIGNED


def test_binding_refuses_mismatched_shapes_before_launching(lib):
    """A filter, output or source of the wrong size is refused on the host, before
    the C ABI (and so any kernel) is reached: these are CPU tensors, which the
    binding would otherwise refuse for not being on the GPU."""
    import torch
    x = torch.zeros(2, 3, 9, 9)
    w = torch.zeros(4, 3, 3, 3)
    out = torch.zeros(2, 4, 7, 7)
    ws = torch.zeros(1 << 12, dtype=torch.uint8)
    with pytest.raises(ValueError, match="out has shape"):
        mec.im2win_conv_fused(x, w, torch.zeros(2, 4, 7, 6), ws, 1, 1)
    with pytest.raises(ValueError, match="out has shape"):
        mec.im2win_conv_fused_noalloc(x, w, torch.zeros(2, 4, 6, 7), 1, 1)
    with pytest.raises(ValueError, match="filt has shape"):
        mec.im2win_conv_fused(x, torch.zeros(4, 2, 3, 3), out, ws, 1, 1)
    with pytest.raises(ValueError, match="window tensor has"):
        mec.im2win_conv(torch.zeros(2 * 3 * 7 * 27 - 1), w, out, ws, 2, 3, 9, 9, 4, 3, 3, 1, 1)
    with pytest.raises(ValueError, match="filt has shape"):
        mec.im2win_conv(torch.zeros(2 * 3 * 7 * 27), w, out, ws, 2, 3, 9, 9, 5, 3, 3, 1, 1)
    with pytest.raises(ValueError, match="out has shape"):
        mec.im2win_conv_fused_nhwc(x.permute(0, 2, 3, 1).contiguous(), w, out, ws, 1, 1)
    with pytest.raises(ValueError, match="out has shape"):
        mec.im2win_conv_fused_ex(x, w, out, ws, 2, 3, 9, 9, 4, 3, 3, 1, 1, 1, 1, 1, 1, mec.NCHW)
    with pytest.raises(ValueError, match="x has"):
        mec.im2win_transform_ex(x[:1], torch.zeros(10 ** 4), 2, 3, 9, 9, 4, 3, 3, 1, 1, 0, 0, 1, 1, mec.NCHW)
    # the right shapes pass the shape checks and stop at the device check
    with pytest.raises(ValueError, match="CUDA"):
        mec.im2win_conv_fused(x, w, out, ws, 1, 1)
    with pytest.raises(ValueError, match="CUDA"):
        mec.im2win_conv_fused_ex(x, w, torch.zeros(2, 4, 9, 9), ws, 2, 3, 9, 9, 4, 3, 3, 1, 1, 1, 1, 1, 1,
                                 mec.NCHW)


def test_workspace_query_refuses_shapes_whose_sizes_would_wrap(lib):
    """Each factor below passes the per-dimension limits, but the window tensor
    (N*C_i*H_o*W_i*H_f elements) would exceed 2^64 bytes: UNSUPPORTED, not a
    wrapped-around size."""
    sz = ctypes.c_size_t()
    big = [1 << 20, 1 << 20, 1 << 19, 1 << 19, 1, 1 << 10, 1, 1, 1]
    assert lib.im2win_workspace_size(0, *big, 0, ctypes.byref(sz)) == mec._binding.ERR_UNSUPPORTED
    assert lib.im2win_workspace_size_ex(0, *big, 0, 0, 1, 1, 0, 0, ctypes.byref(sz)) == \
        mec._binding.ERR_UNSUPPORTED
    # just under the limit the size is exact
    ok = [1, 1 << 10, 1 << 10, 1 << 10, 1, 1, 1, 1, 1]
    assert lib.im2win_workspace_size(0, *ok, 1, ctypes.byref(sz)) == 0
    assert sz.value == (1 << 30) * 2
