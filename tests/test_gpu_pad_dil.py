"""GPU parity of the calls with zero padding and dilation (the *_ex entry
points, both layouts) against the oracle: the padded window transform bit for
bit, the convolutions (fp32 CUDA cores, fp16/bf16 tensor cores; from the padded
window tensor and fused) within the tolerance of their dtype."""
import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl
from parity import TOL, assert_within, to_f64

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
RAW = {torch.float32: np.uint32, torch.float16: np.uint16, torch.bfloat16: np.uint16}
LAYOUTS = {"nchw": mec.NCHW, "nhwc": mec.NHWC}


def _raw(t: torch.Tensor) -> np.ndarray:
    v = t.detach().cpu().contiguous()
    bits = v.view(torch.int32 if v.element_size() == 4 else torch.int16).numpy()
    return bits.view(RAW[t.dtype])


def _inputs(case, dt, layout, seed):
    N, C_i, H_i, W_i, C_o, H_f, W_f = case[:7]
    layer = wl.Layer("pd", N, C_i, H_i, W_i, C_o, H_f, W_f, 1, 1, seed=seed)
    x, w = wl.make_inputs(layer, dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    return x, w


def _run(x, w, stride, pad, dil, layout, fused):
    lo = LAYOUTS[layout]
    xd, wd = x.cuda(), w.cuda()
    if fused:
        return mec.conv_fused_ex(xd, wd, stride, pad, dil, lo)
    win = mec.transform_ex(xd, w.shape[2], w.shape[3], stride, pad, dil, lo)
    return mec.conv_ex(win, wd, tuple(x.shape), stride, pad, dil, lo)


# N, C_i, H_i, W_i, C_o, H_f, W_f, stride, pad, dil
CASES = [
    (2, 16, 20, 21, 32, 3, 3, (1, 1), (1, 1), (1, 1)),      # "same" 3x3
    (1, 64, 17, 19, 64, 3, 3, (1, 1), (2, 2), (2, 2)),      # dilation 2, C_o <= 64 (no stacking)
    (2, 24, 15, 16, 40, 3, 3, (2, 2), (1, 1), (1, 1)),      # stacked taps with padding
    (1, 3, 30, 31, 8, 7, 7, (2, 2), (3, 3), (1, 1)),        # a first layer: 3 channels, 7x7 s2 p3
    (2, 96, 12, 12, 130, 5, 5, (1, 1), (2, 2), (1, 1)),     # two channel tiles, ragged C_o
    (1, 32, 16, 24, 128, 3, 3, (1, 1), (0, 0), (2, 2)),     # dilation only, rows of 24 (16-byte loads)
    (1, 12, 9, 10, 20, 2, 3, (1, 1), (1, 2), (2, 1)),       # channels not a multiple of 8
    (2, 5, 11, 13, 7, 3, 2, (2, 1), (0, 1), (1, 2)),        # mixed strides, one-sided options
    (1, 8, 6, 7, 16, 3, 3, (1, 1), (4, 4), (1, 1)),         # padding wider than the filter: all-zero rows
    # rows of whole 16-byte vectors: the staged (ring) slab fill with shifted columns
    (1, 40, 14, 32, 64, 5, 5, (1, 1), (2, 2), (1, 1)),      # stacked taps
    (2, 16, 13, 24, 136, 3, 5, (2, 1), (1, 2), (1, 1)),     # two channel tiles, row stride 2
    (1, 24, 12, 16, 96, 3, 3, (1, 2), (3, 1), (2, 3)),      # padding and dilation together
]


@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("dt", ["f32", "f16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:7])) + f"_s{c[7]}_p{c[8]}_d{c[9]}")
def test_transform_ex_bit_exact(case, dt, layout):
    st, pd, dl = case[7:]
    x, w = _inputs(case, dt, layout, seed=sum(case[:7]))
    win = mec.transform_ex(x.cuda(), w.shape[2], w.shape[3], st, pd, dl, LAYOUTS[layout])
    torch.cuda.synchronize()
    want = oracle.im2win_pd(_raw(x), w.shape, st, pd, dl, layout)
    got = _raw(win)
    assert got.shape == want.shape
    assert got.tobytes() == want.tobytes()


def test_transform_ex_rows_too_long_to_stage():
    x = torch.randn(1, 3, 9, 9000, dtype=torch.float32)
    win = mec.transform_ex(x.cuda(), 3, 3, (2, 1), (1, 2), (2, 1), mec.NCHW)
    torch.cuda.synchronize()
    want = oracle.im2win_pd(_raw(x), (1, 3, 3, 3), (2, 1), (1, 2), (2, 1))
    assert _raw(win).tobytes() == want.tobytes()


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:7])) + f"_s{c[7]}_p{c[8]}_d{c[9]}")
def test_conv_ex_small(case, dt, layout, fused):
    st, pd, dl = case[7:]
    x, w = _inputs(case, dt, layout, seed=sum(case[:7]) + 3)
    out = _run(x, w, st, pd, dl, layout, fused)
    torch.cuda.synchronize()
    want, scale = oracle.conv_direct_pd(to_f64(x), to_f64(w), st, pd, dl, layout)
    assert tuple(out.shape) == want.shape
    assert_within(to_f64(out), want, scale, TOL[out.dtype], f"{dt} {layout} {case} fused={fused}")


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[2], CASES[5]],
                         ids=lambda c: "x".join(map(str, c[:7])) + f"_p{c[8]}_d{c[9]}")
def test_conv_ex_exact_on_sparse_integers(case, layout, fused):
    N, C_i, H_i, W_i, C_o, H_f, W_f, st, pd, dl = case
    layer = wl.Layer("int", N, C_i, H_i, W_i, C_o, H_f, W_f, 1, 1, seed=6)
    x, w = wl.make_int_inputs(layer, "f16", seed=33, x_range=1, w_range=1, density=0.5)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    out = _run(x, w, st, pd, dl, layout, fused)
    want, _ = oracle.conv_direct_pd(to_f64(x), to_f64(w), st, pd, dl, layout)
    assert np.abs(want).max() <= 2048
    np.testing.assert_array_equal(to_f64(out), want)


def test_conv_ex_plain_equals_the_valid_calls():
    layer = wl.Layer("eq", 2, 16, 19, 23, 40, 3, 5, 2, 1, seed=12)
    x, w = wl.make_inputs(layer, "bf16")
    xd, wd = x.cuda(), w.cuda()
    a = mec.conv_fused_ex(xd, wd, (2, 1))
    b = mec.conv_fused(xd, wd, (2, 1))
    assert torch.equal(a, b)


def test_conv_ex_rejects_a_filter_wider_than_the_padded_input():
    x = torch.zeros(1, 2, 4, 4, dtype=torch.float16, device="cuda")
    w = torch.zeros(1, 2, 3, 3, dtype=torch.float16, device="cuda")
    with pytest.raises(mec.Im2winError):
        mec.conv_fused_ex(x, w, (1, 1), (1, 1), (3, 3))


@pytest.mark.parametrize("layer,dt", [(wl.SAME_3x3, "bf16"), (wl.SAME_3x3, "f32"), (wl.DIL_3x3, "bf16")],
                         ids=lambda v: getattr(v, "name", v))
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
def test_conv_ex_full_size_sampled(layer, dt, layout):
    x, w = wl.make_inputs(layer, dt)
    xin = x.permute(0, 2, 3, 1).contiguous() if layout == "nhwc" else x
    st = (layer.s_h, layer.s_w)
    rng = np.random.default_rng(7)
    w64 = to_f64(w)
    for fused in (False, True):
        out = _run(xin, w, st, layer.pad, layer.dil, layout, fused)
        torch.cuda.synchronize()
        o = out.permute(0, 3, 1, 2) if layout == "nhwc" else out  # NCHW view
        tol = TOL[out.dtype]
        for n in (0, layer.N - 1):
            want, scale = oracle.conv_direct_pd(to_f64(x[n:n + 1]), w64, st, layer.pad, layer.dil)
            assert_within(to_f64(o[n:n + 1]), want, scale, tol, f"{layer.name} {layout} image {n}")
        idx = np.stack([rng.integers(0, s, 2048) for s in o.shape], axis=1)
        got = to_f64(o[tuple(torch.from_numpy(idx.T.copy()).to(o.device))])
        for n in np.unique(idx[:, 0]):
            sel = idx[:, 0] == n
            loc = idx[sel].copy()
            loc[:, 0] = 0
            vals, scale = oracle.conv_points_pd(to_f64(x[n:n + 1]), w64, loc, st, layer.pad, layer.dil)
            assert_within(got[sel], vals, scale, tol, f"{layer.name} {layout} sampled image {n}")
        del out, o
        torch.cuda.empty_cache()
