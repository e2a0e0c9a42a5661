"""GPU parity of the fp16/bf16 tensor-core (tcgen05) convolution, from the
window tensor and fused, against the fp64 oracle."""
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
    (1, 1, 50, 3, 1, 2, 3, 3, 1), (2, 96, 24, 24, 256, 5, 5, 1, 1), (1, 16, 40, 40, 200, 3, 3, 1, 1),
    # many input channels: the fused call takes the tap kernel (vector and scalar slab fills,
    # one or two MMA halves, several row tiles, strides 1-3, channel counts not a multiple of 16)
    (2, 32, 30, 64, 128, 3, 5, 3, 2), (1, 48, 60, 56, 64, 11, 11, 1, 1), (2, 128, 30, 56, 128, 3, 3, 1, 1),
    (1, 24, 100, 16, 40, 2, 2, 2, 2), (2, 40, 33, 35, 136, 4, 3, 2, 1), (1, 64, 9, 600, 16, 3, 3, 1, 2),
    # 1x1 filters at stride 1 on rows of whole 8-position groups: the input tile copied
    # MN-major into the slab (channels past C_i and positions past the plane read as zero)
    (2, 40, 12, 16, 72, 1, 1, 1, 1), (1, 32, 40, 24, 64, 1, 1, 1, 1), (1, 16, 5, 8, 128, 1, 1, 1, 1),
    # ... in 64-position blocks with the copy's 128-byte swizzle (planes and tiles whole
    # blocks): a tile of one block (no second accumulator), a ragged last tile, three chunks
    (3, 24, 8, 32, 200, 1, 1, 1, 1), (2, 48, 16, 64, 130, 1, 1, 1, 1), (2, 96, 10, 32, 96, 1, 1, 1, 1),
]


def _run(x, w, stride, fused):
    xd, wd = x.cuda(), w.cuda()
    if fused:
        return mec.conv_fused(xd, wd, stride)
    win = mec.transform(xd, w.shape[2], stride[0])
    return mec.conv(win, wd, stride)


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_conv_tc_small(case, dt, fused):
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("t", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=sum(case))
    x, w = wl.make_inputs(layer, dt)
    out = _run(x, w, (s_h, s_w), fused)
    torch.cuda.synchronize()
    check_full(out, x, w, (s_h, s_w), f"{dt} {case} fused={fused}")


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("dt,bound", [("f16", 2048), ("bf16", 256)])
def test_conv_tc_exact_on_sparse_integers(dt, bound, fused):
    """Sparse +-1 inputs keep |out| small enough to be exact in the output dtype,
    and every fp32 partial sum is an exact integer: the result must equal the
    oracle exactly, whatever the summation order."""
    layer = wl.Layer("int", 2, 24, 30, 31, 150, 5, 3, 1, 2, seed=5)
    x, w = wl.make_int_inputs(layer, dt, seed=22, x_range=1, w_range=1, density=0.5)
    out = _run(x, w, (1, 2), fused)
    want, _ = oracle.conv_direct(to_f64(x), to_f64(w), (1, 2))
    assert np.abs(want).max() <= bound
    np.testing.assert_array_equal(to_f64(out), want)


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("case", [(2, 40, 12, 16, 72), (2, 48, 16, 64, 130),
                                  (64, 40, 16, 56, 64), (40, 32, 24, 56, 136)],
                         ids=lambda c: "x".join(map(str, c)))
def test_conv_tc_1x1_exact_on_integers(case, fused):
    """1x1 filters: the MN-major slab, without swizzle (16-position rows) and with the
    128-byte swizzle (whole 64-position blocks). Sparse integer inputs make every
    partial sum exact, so the result must equal the oracle exactly: a position or
    channel read from the wrong place of the slab shows as a mismatch."""
    N, C_i, H_i, W_i, C_o = case
    layer = wl.Layer("mn", N, C_i, H_i, W_i, C_o, 1, 1, 1, 1, seed=12)
    x, w = wl.make_int_inputs(layer, "bf16", seed=24, x_range=1, w_range=1, density=0.5)
    out = _run(x, w, (1, 1), fused)
    want, _ = oracle.conv_direct(to_f64(x), to_f64(w), (1, 1))
    assert np.abs(want).max() <= 256
    np.testing.assert_array_equal(to_f64(out), want)


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("case", [(2, 24, 30, 33, 40, 5, 3, 1, 2), (1, 40, 21, 29, 64, 7, 7, 2, 2),
                                  (2, 17, 19, 40, 8, 3, 4, 1, 1),
                                  # tiles of two M blocks (positions past 128) with positions
                                  # along M: the shifted add crosses lane quarters and blocks
                                  (1, 24, 12, 150, 40, 5, 3, 1, 2), (2, 16, 9, 200, 64, 3, 4, 1, 1),
                                  (1, 32, 17, 224, 64, 7, 7, 2, 2),
                                  # 1120 tiles: every CTA reuses both TMEM buffers several times
                                  (160, 8, 9, 200, 16, 3, 4, 1, 1)],
                         ids=lambda c: "x".join(map(str, c)))
def test_conv_tc_stacked_taps_exact_on_integers(case, fused):
    """Output channels <= 64: two filter taps share one MMA (the second tap's sum is
    taken one column to the left and added back in the epilogue). On sparse integer
    inputs every partial sum is exact, so the result must equal the oracle exactly."""
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("stk", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=8)
    x, w = wl.make_int_inputs(layer, "f16", seed=23, x_range=1, w_range=1, density=0.5)
    out = _run(x, w, (s_h, s_w), fused)
    want, _ = oracle.conv_direct(to_f64(x), to_f64(w), (s_h, s_w))
    assert np.abs(want).max() <= 2048
    np.testing.assert_array_equal(to_f64(out), want)


@pytest.mark.parametrize("r0,j0", [(3, 2), (5, 6), (0, 0), (6, 5)])
def test_conv_tc_stacked_one_hot_is_exact_crop(r0, j0):
    """A single non-zero filter tap with C_o <= 64 at a pair's top (j=0), bottom
    (j=2: partner of 0 at stride 2), the last column's unpaired tap (j=6 at W_f=7,
    s_w=2 pairs with nothing) and the other row/column phases."""
    layer = wl.Layer("hot2", 2, 20, 33, 37, 48, 7, 7, 2, 2, seed=10)
    x, _ = wl.make_inputs(layer, "bf16")
    w = torch.zeros((48, 20, 7, 7), dtype=torch.bfloat16)
    w[41, 13, r0, j0] = 1.0
    for fused in (False, True):
        out = _run(x, w, (2, 2), fused)
        ho, wo = out.shape[2:]
        crop = x[:, 13, r0:r0 + (ho - 1) * 2 + 1:2, j0:j0 + (wo - 1) * 2 + 1:2]
        assert torch.equal(out[:, 41].cpu(), crop), f"fused={fused}"
        assert not out[:, :41].any() and not out[:, 42:].any()


def test_conv_tc_one_hot_filter_is_exact_crop():
    layer = wl.Layer("hot", 2, 20, 33, 37, 130, 4, 5, 2, 3, seed=9)
    x, _ = wl.make_inputs(layer, "bf16")
    w = torch.zeros((130, 20, 4, 5), dtype=torch.bfloat16)
    w[77, 13, 2, 3] = 1.0
    for fused in (False, True):
        out = _run(x, w, (2, 3), fused)
        ho, wo = out.shape[2:]
        crop = x[:, 13, 2:2 + (ho - 1) * 2 + 1:2, 3:3 + (wo - 1) * 3 + 1:3]
        assert torch.equal(out[:, 77].cpu(), crop)
        assert not out[:, :77].any() and not out[:, 78:].any()


@pytest.mark.parametrize("layer,dt", [(wl.CV1, "f16"), (wl.CV2, "f16"), (wl.CV3, "f16"), (wl.CV4, "f16"),
                                      (wl.CV5, "bf16")]
                         + [(l, "bf16") for l in wl.SWEEP], ids=lambda v: getattr(v, "name", v))
def test_conv_tc_full_size_sampled(layer, dt):
    x, w = wl.make_inputs(layer, dt)
    stride = (layer.s_h, layer.s_w)
    for fused in (False, True):
        out = _run(x, w, stride, fused)
        torch.cuda.synchronize()
        check_sampled(out, x, w, stride, images=(0, -1), n_points=2048,
                      what=f"{layer.name} {dt} fused={fused}")
        del out
        torch.cuda.empty_cache()


def test_conv_tc_status_ok_and_no_write_past_output():
    layer = wl.Layer("g", 3, 8, 19, 23, 70, 3, 3, 1, 1, seed=4)
    x, w = wl.make_inputs(layer, "f16")
    ho, wo = 17, 21
    n_out = 3 * 70 * ho * wo
    buf = torch.full((n_out + 256,), 5.0, dtype=torch.float16, device="cuda")
    out = buf[:n_out].view(3, 70, ho, wo)
    ws = mec.workspace(mec.OP_CONV_FUSED, x.shape, w.shape, (1, 1), torch.float16, "cuda")
    mec.conv_fused(x.cuda(), w.cuda(), (1, 1), ws=ws, out=out)
    assert mec.im2win_device_status(ws) == 0
    assert torch.all(buf[n_out:] == 5.0)
    check_full(out, x, w, (1, 1), "guarded")
