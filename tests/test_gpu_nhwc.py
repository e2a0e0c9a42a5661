"""GPU parity of the channels-last (NHWC) calls against the oracle: the window
transform bit for bit, the convolutions (fp32 CUDA cores, fp16/bf16 tensor
cores; from the window tensor and fused) within the tolerance of their dtype.

Inputs are the NCHW draws of the workload recipe with the channel axis moved
innermost, so every NHWC case sees the same values as its NCHW counterpart."""
import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl
from parity import TOL, assert_within, check_sampled, to_f64

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
RAW = {torch.float32: np.uint32, torch.float16: np.uint16, torch.bfloat16: np.uint16}


def _raw(t: torch.Tensor) -> np.ndarray:
    v = t.detach().cpu().contiguous()
    bits = v.view(torch.int32 if v.element_size() == 4 else torch.int16).numpy()
    return bits.view(RAW[t.dtype])


def _cl(x: torch.Tensor) -> torch.Tensor:
    return x.permute(0, 2, 3, 1).contiguous()


def _run(x_cl, w, stride, fused):
    xd, wd = x_cl.cuda(), w.cuda()
    if fused:
        return mec.conv_fused_nhwc(xd, wd, stride)
    win = mec.transform_nhwc(xd, w.shape[2], stride[0])
    return mec.conv_nhwc(win, wd, stride)


def _check_full(out, x_cl, w, stride, what):
    want, scale = oracle.conv_direct_nhwc(to_f64(x_cl), to_f64(w), stride)
    assert tuple(out.shape) == want.shape, (tuple(out.shape), want.shape)
    assert_within(to_f64(out), want, scale, TOL[out.dtype], what)


# ---------------------------------------------------------------- transform
T_CASES = [  # N, C_i, H_i, W_i, H_f, s_h
    (2, 3, 32, 32, 3, 1), (3, 5, 37, 45, 11, 4), (2, 8, 20, 21, 3, 2), (1, 64, 17, 19, 7, 2),
    (2, 12, 9, 13, 9, 1), (1, 1, 40, 5, 1, 1), (2, 4, 50, 17, 3, 5), (1, 96, 24, 24, 5, 1),
    # input rows too long to stage a band in shared memory: element-wise path
    (1, 3, 12, 12000, 3, 2),
    # channel runs of whole 16-byte vectors, window rows in several column chunks
    # with a short last one (tensor-copy path)
    (1, 64, 12, 301, 5, 2), (2, 32, 9, 130, 3, 1),
    # more channels than a tensor copy's box holds (256): the vector-copy kernel
    (1, 264, 6, 8, 3, 1),
]


@pytest.mark.parametrize("case", T_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_transform_nhwc_small_bit_exact(case, dt):
    N, C_i, H_i, W_i, H_f, s_h = case
    g = torch.Generator().manual_seed(sum(case))
    x = (torch.rand((N, H_i, W_i, C_i), generator=g) * 2 - 1).to(DT[dt])
    win = mec.transform_nhwc(x.cuda(), H_f, s_h)
    torch.cuda.synchronize()
    want = oracle.im2win_nhwc(_raw(x), H_f, s_h)
    got = _raw(win)
    assert got.shape == want.shape
    assert got.tobytes() == want.tobytes()


def test_transform_nhwc_does_not_write_past_the_window():
    x = torch.randn(2, 31, 45, 3, dtype=torch.float16)  # 3 channels: staged bands, unaligned band ends
    H_f, s_h = 11, 4
    H_o = (31 - H_f) // s_h + 1
    n = 2 * H_o * 45 * H_f * 3
    buf = torch.full((n + 64,), 7, dtype=torch.float16, device="cuda")
    mec.im2win_transform_nhwc(x.cuda(), buf, 1, H_f, 1, s_h, 1)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7)
    assert _raw(buf[:n]).tobytes() == oracle.im2win_nhwc(_raw(x), H_f, s_h).tobytes()


@pytest.mark.parametrize("layer,dt", [(wl.CV1, "f16"), (wl.CV1, "f32"), (wl.CV5, "bf16"), (wl.SWEEP[1], "bf16")],
                         ids=lambda v: getattr(v, "name", v))
def test_transform_nhwc_full_size_bit_exact(layer, dt):
    x, _ = wl.make_inputs(layer, dt)
    x = _cl(x)
    win = mec.transform_nhwc(x.cuda(), layer.H_f, layer.s_h)
    torch.cuda.synchronize()
    assert _raw(win).tobytes() == oracle.im2win_nhwc(_raw(x), layer.H_f, layer.s_h).tobytes()


# ---------------------------------------------------------------- convolutions
SMALL = [  # N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w
    # C_i a multiple of 8: channel-group copies straight into the tensor-core slab
    (2, 16, 19, 40, 8, 3, 4, 1, 1), (1, 64, 20, 21, 64, 7, 7, 2, 2), (2, 96, 24, 24, 256, 5, 5, 1, 1),
    (2, 128, 30, 56, 128, 3, 3, 1, 1), (2, 32, 30, 64, 130, 3, 5, 3, 2), (1, 24, 100, 16, 40, 2, 2, 2, 2),
    (1, 40, 21, 29, 60, 7, 7, 2, 2), (1, 8, 9, 600, 16, 3, 3, 1, 2),
    # other channel counts: the input seen as one channel of W_i*C_i columns
    (1, 3, 32, 32, 8, 3, 3, 1, 1), (2, 3, 47, 45, 96, 11, 11, 4, 4), (2, 5, 30, 33, 37, 3, 7, 1, 2),
    (2, 12, 19, 40, 20, 3, 4, 1, 1), (1, 100, 12, 13, 30, 3, 3, 1, 1), (1, 1, 50, 3, 1, 2, 3, 3, 1),
    (3, 17, 12, 14, 130, 1, 1, 1, 1),
    # 1x1 filters with channels in whole 64s: 64-channel chunks copied K-major with the
    # copy's 128-byte swizzle (tiles past the last row, positions past a box, no second
    # accumulator, three chunks, 256-position rows)
    (2, 64, 12, 16, 72, 1, 1, 1, 1), (3, 128, 9, 24, 200, 1, 1, 1, 1), (1, 192, 5, 40, 64, 1, 1, 1, 1),
    (2, 64, 7, 8, 130, 1, 1, 1, 1), (1, 64, 3, 256, 96, 1, 1, 1, 1),
]


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_conv_nhwc_small(case, dt, fused):
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("t", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=sum(case) + 1)
    x, w = wl.make_inputs(layer, dt)
    x = _cl(x)
    out = _run(x, w, (s_h, s_w), fused)
    torch.cuda.synchronize()
    _check_full(out, x, w, (s_h, s_w), f"{dt} {case} fused={fused}")


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("case", [(2, 24, 30, 31, 150, 5, 3, 1, 2), (2, 24, 30, 33, 40, 5, 3, 1, 2),
                                  (1, 40, 21, 29, 64, 7, 7, 2, 2), (2, 12, 19, 40, 20, 3, 4, 1, 1),
                                  # stacked tiles of two M blocks; many tiles per CTA
                                  (1, 24, 12, 150, 48, 5, 3, 1, 2), (2, 16, 9, 200, 64, 3, 4, 1, 1),
                                  (160, 8, 9, 200, 16, 3, 4, 1, 1),
                                  # 1x1, 64-channel swizzled K-major chunks; several tiles per CTA
                                  (2, 64, 12, 16, 72, 1, 1, 1, 1), (40, 64, 24, 56, 136, 1, 1, 1, 1)],
                         ids=lambda c: "x".join(map(str, c)))
def test_conv_nhwc_exact_on_sparse_integers(case, fused):
    """Sparse +-1 inputs: every fp32 partial sum is an exact small integer and the
    result is exact in fp16, so it must equal the oracle exactly in any order
    (covers the stacked-tap epilogue for C_o <= 64)."""
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("int", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=5)
    x, w = wl.make_int_inputs(layer, "f16", seed=31, x_range=1, w_range=1, density=0.5)
    x = _cl(x)
    out = _run(x, w, (s_h, s_w), fused)
    want, _ = oracle.conv_direct_nhwc(to_f64(x), to_f64(w), (s_h, s_w))
    assert np.abs(want).max() <= 2048
    np.testing.assert_array_equal(to_f64(out), want)


def test_conv_nhwc_one_hot_filter_is_exact_crop():
    layer = wl.Layer("hot", 2, 24, 33, 37, 130, 4, 5, 2, 3, seed=9)
    x, _ = wl.make_inputs(layer, "bf16")
    x = _cl(x)
    w = torch.zeros((130, 24, 4, 5), dtype=torch.bfloat16)
    w[77, 13, 2, 3] = 1.0
    for fused in (False, True):
        out = _run(x, w, (2, 3), fused)
        ho, wo = out.shape[1:3]
        crop = x[:, 2:2 + (ho - 1) * 2 + 1:2, 3:3 + (wo - 1) * 3 + 1:3, 13]
        assert torch.equal(out[..., 77].cpu(), crop), f"fused={fused}"
        assert not out[..., :77].any() and not out[..., 78:].any()


def test_conv_nhwc_status_ok_and_no_write_past_output():
    layer = wl.Layer("g", 3, 16, 19, 23, 70, 3, 3, 1, 1, seed=4)
    x, w = wl.make_inputs(layer, "f16")
    x = _cl(x)
    ho, wo = 17, 21
    n_out = 3 * ho * wo * 70
    buf = torch.full((n_out + 256,), 5.0, dtype=torch.float16, device="cuda")
    out = buf[:n_out].view(3, ho, wo, 70)
    ws = mec.workspace(mec.OP_CONV_FUSED_NHWC, (3, 16, 19, 23), w.shape, (1, 1), torch.float16, "cuda")
    mec.conv_fused_nhwc(x.cuda(), w.cuda(), (1, 1), ws=ws, out=out)
    assert mec.im2win_device_status(ws) == 0
    assert torch.all(buf[n_out:] == 5.0)
    _check_full(out, x, w, (1, 1), "guarded")


@pytest.mark.parametrize("layer,dt", [(wl.CV1, "f16"), (wl.CV1, "f32"), (wl.CV4, "f16"), (wl.CV5, "bf16"),
                                      (wl.SWEEP[0], "bf16"), (wl.SWEEP[1], "bf16"), (wl.SWEEP[4], "bf16")],
                         ids=lambda v: getattr(v, "name", v))
def test_conv_nhwc_full_size_sampled(layer, dt):
    x, w = wl.make_inputs(layer, dt)
    stride = (layer.s_h, layer.s_w)
    xc = _cl(x)
    for fused in (False, True):
        out = _run(xc, w, stride, fused)
        torch.cuda.synchronize()
        # the NCHW view of the channels-last output against the NCHW draw
        check_sampled(out.permute(0, 3, 1, 2), x, w, stride, images=(0, -1), n_points=2048,
                      what=f"{layer.name} {dt} nhwc fused={fused}")
        del out
        torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
def test_stacked_taps_ignore_what_earlier_kernels_left_in_shared_memory(layout, fused):
    """With tap stacking (C_o <= 64) a group without a second tap multiplies zero
    filter rows by slab entries past the input's last column, which no fill
    writes. Convolutions of all-NaN inputs of wider shapes first leave NaN bit
    patterns in the SMs' shared memory; the exact integer result must follow."""
    cl = layout == "nhwc"
    for wi in (40, 48, 64, 96):
        xn = torch.full((2, 24, 30, wi), float("nan"), dtype=torch.float16)
        wn = torch.ones((40, 24, 5, 3), dtype=torch.float16)
        xn = _cl(xn) if cl else xn
        if cl:
            _run(xn, wn, (1, 2), fused)
        else:
            xd = xn.cuda()
            mec.conv_fused(xd, wn.cuda(), (1, 2)) if fused else mec.conv(mec.transform(xd, 5, 1), wn.cuda(), (1, 2))
    layer = wl.Layer("stale", 2, 24, 30, 33, 40, 5, 3, 1, 2, seed=5)
    x, w = wl.make_int_inputs(layer, "f16", seed=31, x_range=1, w_range=1, density=0.5)
    if cl:
        x = _cl(x)
        out = _run(x, w, (1, 2), fused)
        want, _ = oracle.conv_direct_nhwc(to_f64(x), to_f64(w), (1, 2))
    else:
        xd = x.cuda()
        out = (mec.conv_fused(xd, w.cuda(), (1, 2)) if fused
               else mec.conv(mec.transform(xd, 5, 1), w.cuda(), (1, 2)))
        want, _ = oracle.conv_direct(to_f64(x), to_f64(w), (1, 2))
    np.testing.assert_array_equal(to_f64(out), want)
