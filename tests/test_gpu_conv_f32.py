"""GPU parity of the fp32 CUDA-core convolution (from the window tensor and fused)."""
import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl
from parity import check_full, check_sampled, to_f64

pytestmark = pytest.mark.gpu

SMALL = [  # N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w
    (1, 3, 32, 32, 8, 3, 3, 1, 1), (2, 3, 47, 45, 96, 11, 11, 4, 4), (2, 5, 30, 33, 37, 3, 7, 1, 2),
    (3, 17, 12, 14, 130, 1, 1, 1, 1), (1, 64, 20, 21, 64, 7, 7, 2, 2), (2, 2, 9, 9, 5, 9, 9, 1, 1),
    (1, 1, 50, 3, 1, 2, 3, 3, 1), (2, 8, 24, 24, 33, 5, 5, 1, 1),
]


def _run(x, w, stride, fused):
    xd, wd = x.cuda(), w.cuda()
    if fused:
        return mec.conv_fused(xd, wd, stride)
    win = mec.transform(xd, w.shape[2], stride[0])
    return mec.conv(win, wd, stride)


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_conv_f32_small(case, fused):
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("t", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=sum(case))
    x, w = wl.make_inputs(layer, "f32")
    out = _run(x, w, (s_h, s_w), fused)
    torch.cuda.synchronize()
    check_full(out, x, w, (s_h, s_w), f"f32 {case} fused={fused}")


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
def test_conv_f32_exact_on_integers(fused):
    """Integer inputs make every fp32 partial sum exact: any summation order must
    reproduce the oracle bit for bit."""
    layer = wl.Layer("int", 2, 7, 40, 43, 70, 5, 3, 2, 3, seed=5)
    x, w = wl.make_int_inputs(layer, "f32", seed=21)
    out = _run(x, w, (2, 3), fused)
    want, _ = oracle.conv_direct(to_f64(x), to_f64(w), (2, 3))
    np.testing.assert_array_equal(to_f64(out), want)


def test_conv_f32_tiny_config():
    layer = wl.TINY
    x, w = wl.make_inputs(layer, "f32")
    for fused in (False, True):
        out = _run(x, w, (1, 1), fused)
        check_full(out, x, w, (1, 1), f"tiny fused={fused}")


@pytest.mark.parametrize("layer", [wl.CV1, wl.CV2, wl.CV3] + list(wl.SWEEP), ids=lambda l: l.name)
def test_conv_f32_full_size_sampled(layer):
    x, w = wl.make_inputs(layer, "f32")
    stride = (layer.s_h, layer.s_w)
    for fused in (False, True):
        out = _run(x, w, stride, fused)
        torch.cuda.synchronize()
        check_sampled(out, x, w, stride, images=(0, -1), n_points=2048,
                      what=f"{layer.name} f32 fused={fused}")


def test_conv_workspace_status_is_ok_after_f32_call():
    x, w = wl.make_inputs(wl.TINY, "f32")
    ws = mec.workspace(mec.OP_CONV_FUSED, x.shape, w.shape, (1, 1), torch.float32, "cuda")
    mec.conv_fused(x.cuda(), w.cuda(), (1, 1), ws=ws)
    assert mec.im2win_device_status(ws) == 0
