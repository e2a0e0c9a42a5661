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
