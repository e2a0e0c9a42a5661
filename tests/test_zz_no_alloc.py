"""The fused convolution for callers that cannot allocate a workspace.

Some callers hold only their input and output buffers (a plugin slot that is
handed tensor pointers and nothing else, or code that must not call cudaMalloc
because it may synchronise the device). im2win_conv_fused_noalloc serves them
from a scratch array built into the library. Its results must match the
workspace-taking entry point's on the same inputs, also on the second of two
calls in a row that share (and overwrite) that array.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl
from parity import TOL, to_f64

pytestmark = pytest.mark.gpu

# two different problems so that the second call overwrites the first's scratch
CASES = [
    ("bf16", wl.Layer("a", 2, 96, 24, 24, 256, 5, 5, 1, 1, seed=31)),
    ("f16", wl.Layer("b", 2, 3, 47, 45, 96, 11, 11, 4, 4, seed=32)),
    ("f32", wl.Layer("c", 2, 8, 20, 21, 40, 3, 3, 1, 2, seed=33)),
]


def _noalloc(x, w, stride):
    N, C_i, H_i, W_i = x.shape
    C_o, _, H_f, W_f = w.shape
    H_o, W_o = mec.out_hw(H_i, W_i, H_f, W_f, *stride)
    out = torch.full((N, C_o, H_o, W_o), float("nan"), dtype=x.dtype, device=x.device)
    st = mec.lib().im2win_conv_fused_noalloc(
        x.data_ptr(), w.data_ptr(), out.data_ptr(), N, C_i, H_i, W_i, C_o, H_f, W_f, stride[0],
        stride[1], mec._binding._dtype_code(x), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, mec.status_string(st)
    return out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    for _ in range(2):
        for dt, layer in CASES:
            x, w = wl.make_inputs(layer, dt)
            x, w = x.cuda(), w.cuda()
            stride = (layer.s_h, layer.s_w)
            got = _noalloc(x, w, stride)
            want = mec.conv_fused(x, w, stride)  # the entry point that takes a workspace
            torch.cuda.synchronize()
            _, scale = oracle.conv_direct(to_f64(x), to_f64(w), stride)
            err = np.abs(to_f64(got) - to_f64(want))
            assert np.all(err <= TOL[x.dtype] * scale), (dt, layer.name, err.max())


def test_noalloc_call_allocates_no_device_memory():
    """What the entry point exists for: once its kernels are loaded (the first
    call), a call takes no device memory -- neither from torch's allocator nor
    from the driver (free bytes of the device unchanged)."""
    dt, layer = CASES[0]
    x, w = wl.make_inputs(layer, dt)
    x, w = x.cuda(), w.cuda()
    stride = (layer.s_h, layer.s_w)
    _noalloc(x, w, stride)  # loads the kernels, looks up the scratch address
    torch.cuda.synchronize()
    H_o, W_o = mec.out_hw(layer.H_i, layer.W_i, layer.H_f, layer.W_f, *stride)
    out = torch.empty((layer.N, layer.C_o, H_o, W_o), dtype=x.dtype, device=x.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        st = mec.lib().im2win_conv_fused_noalloc(
            x.data_ptr(), w.data_ptr(), out.data_ptr(), layer.N, layer.C_i, layer.H_i, layer.W_i, layer.C_o,
            layer.H_f, layer.W_f, stride[0], stride[1], mec._binding._dtype_code(x), stream)
        assert st == 0, mec.status_string(st)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 512 x 512 channels of 11 x 11 taps: the re-laid fp32 filter alone is 121 MiB
    big = (1, 512, 16, 16, 512, 11, 11, 1, 1)
    need = mec.im2win_workspace_size(mec.OP_CONV_FUSED, *big, mec.F32)
    assert need > mec.NOALLOC_SCRATCH_BYTES
    st = mec.lib().im2win_conv_fused_noalloc(16, 16, 16, *big, mec.F32, None)
    assert st == mec._binding.ERR_WORKSPACE
