"""Pins for the CPU oracle (no GPU needed).

The oracle is checked against things other than itself: the hand-derived
values of the worked example sized like Fig. 1 of "Enabling Memory-efficient
Im2win Convolution with Multi-precision Support on GPU CUDA and Tensor Cores",
closed forms (summed-area box sums, one-hot crops, the 1x1 identity), a library
routine (torch's fp64 conv2d), exact agreement of its three independent
formulations on integer inputs, linearity, and the element-count ratios the
Abstract of "Im2win: Memory Efficient Convolution On SIMD Architectures" argues
from.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "fig1_worked_example.json")


def _fig1_x():
    c, h, w = np.meshgrid(np.arange(3), np.arange(3), np.arange(3), indexing="ij")
    return (9 * c + 3 * h + w).astype(np.float64)[None]


def _fig1_filter(rule):
    if rule == "ones":
        return np.ones((2, 3, 2, 2))
    return (np.arange(24, dtype=np.float64) - 11).reshape(2, 3, 2, 2)


@pytest.mark.parametrize("rule", ["ones", "ramp"])
def test_fig1_worked_example_outputs(rule):
    gold = json.load(open(GOLD))
    x, w = _fig1_x(), _fig1_filter(rule)
    want = np.array(gold["filters"][rule]["out"], dtype=np.float64)[None]
    out, scale = oracle.conv_direct(x, w, (1, 1))
    assert out.shape == (1, 2, 2, 2)
    np.testing.assert_array_equal(out, want)
    np.testing.assert_array_equal(oracle.conv_im2col(x, w), want)
    np.testing.assert_array_equal(oracle.conv_im2win(x, w), want)
    assert np.all(scale >= np.abs(out))


def test_fig1_window_rows_and_counts():
    gold = json.load(open(GOLD))
    x = _fig1_x()
    win = oracle.im2win(x, 2, 1)
    assert win.shape == (1, 3, 2, 6)
    np.testing.assert_array_equal(win[0, 0, 0], gold["window_rows_channel0"]["ho0"])
    np.testing.assert_array_equal(win[0, 0, 1], gold["window_rows_channel0"]["ho1"])
    # other channels are the same rows shifted by 9 per channel (x = 9c + ...)
    np.testing.assert_array_equal(win[0, 1], win[0, 0] + 9)
    np.testing.assert_array_equal(win[0, 2], win[0, 0] + 18)
    n_in, n_win, n_col = oracle.workspace_elems(x.shape, (2, 3, 2, 2), (1, 1))
    cnt = gold["element_counts"]
    assert (n_in, n_win, n_col) == (cnt["input"], cnt["im2win"], cnt["im2col"])


def _box_sums(img, hf, wf, sh, sw):
    """Sliding-window sums of a 2-D array through a summed-area table."""
    sat = np.zeros((img.shape[0] + 1, img.shape[1] + 1))
    sat[1:, 1:] = img.cumsum(0).cumsum(1)
    ho = (img.shape[0] - hf) // sh + 1
    wo = (img.shape[1] - wf) // sw + 1
    r = np.arange(ho)[:, None] * sh
    c = np.arange(wo)[None, :] * sw
    return sat[r + hf, c + wf] - sat[r, c + wf] - sat[r + hf, c] + sat[r, c]


@pytest.mark.parametrize("hf,wf,sh,sw", [(3, 3, 1, 1), (5, 2, 2, 3), (1, 4, 3, 1), (7, 7, 2, 2)])
def test_all_ones_filter_is_box_sum(hf, wf, sh, sw):
    rng = np.random.default_rng(11)
    x = rng.integers(-9, 10, size=(2, 3, 17, 19)).astype(np.float64)
    w = np.ones((2, 3, hf, wf))
    out, _ = oracle.conv_direct(x, w, (sh, sw))
    for n in range(2):
        want = sum(_box_sums(x[n, c], hf, wf, sh, sw) for c in range(3))
        np.testing.assert_array_equal(out[n, 0], want)
        np.testing.assert_array_equal(out[n, 1], want)


@pytest.mark.parametrize("ci0,r0,j0", [(0, 0, 0), (2, 3, 1), (1, 4, 4)])
def test_one_hot_filter_is_strided_crop(ci0, r0, j0):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 3, 23, 21))
    w = np.zeros((4, 3, 5, 5))
    w[2, ci0, r0, j0] = 1.0
    sh, sw = 2, 3
    out, _ = oracle.conv_direct(x, w, (sh, sw))
    ho, wo = out.shape[2:]
    crop = x[:, ci0, r0:r0 + (ho - 1) * sh + 1:sh, j0:j0 + (wo - 1) * sw + 1:sw]
    np.testing.assert_array_equal(out[:, 2], crop)
    assert not out[:, [0, 1, 3]].any()
    np.testing.assert_array_equal(oracle.conv_im2win(x, w, (sh, sw))[:, 2], crop)


def test_1x1_window_is_identity_and_stride_hf_is_permutation():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 4, 9, 7)).astype(np.float32)
    win = oracle.im2win(x, 1, 1)
    assert win.tobytes() == x.tobytes()
    # s_h == H_f with H_i divisible: every input element appears exactly once
    win3 = oracle.im2win(x, 3, 3)
    assert win3.size == x.size
    np.testing.assert_array_equal(np.sort(win3.ravel()), np.sort(x.ravel()))


def test_im2win_is_a_byte_copy_for_every_element_size():
    rng = np.random.default_rng(14)
    for dt in (np.uint8, np.uint16, np.float32, np.float64):
        x = rng.integers(0, 250, size=(2, 3, 10, 11)).astype(dt)
        win = oracle.im2win(x, 4, 3)
        ho = (10 - 4) // 3 + 1
        assert win.shape == (2, 3, ho, 11 * 4)
        for h in range(ho):
            for r in range(4):
                np.testing.assert_array_equal(win[:, :, h, r::4], x[:, :, 3 * h + r, :])


def _random_case(rng):
    hf, wf = rng.integers(1, 5, size=2)
    sh, sw = rng.integers(1, 4, size=2)
    hi = int(rng.integers(hf, 10))
    wi = int(rng.integers(wf, 10))
    ci = int(rng.choice([1, 2, 3, 17]))
    co = int(rng.choice([1, 5]))
    n = int(rng.choice([1, 2]))
    return n, ci, hi, wi, co, int(hf), int(wf), int(sh), int(sw)


def test_three_formulations_agree_exactly_on_integers():
    """direct == im2col+GEMM == im2win+dot, bit for bit (all sums are exact integers)."""
    rng = np.random.default_rng(15)
    for _ in range(300):
        n, ci, hi, wi, co, hf, wf, sh, sw = _random_case(rng)
        x = rng.integers(-3, 4, size=(n, ci, hi, wi)).astype(np.float64)
        w = rng.integers(-3, 4, size=(co, ci, hf, wf)).astype(np.float64)
        d, s = oracle.conv_direct(x, w, (sh, sw))
        np.testing.assert_array_equal(oracle.conv_im2col(x, w, (sh, sw)), d)
        np.testing.assert_array_equal(oracle.conv_im2win(x, w, (sh, sw)), d)
        np.testing.assert_array_equal(s, oracle.conv_direct(np.abs(x), np.abs(w), (sh, sw))[0])


def test_matches_torch_conv2d_fp64():
    rng = np.random.default_rng(16)
    for _ in range(60):
        n, ci, hi, wi, co, hf, wf, sh, sw = _random_case(rng)
        x = rng.uniform(-1, 1, size=(n, ci, hi, wi))
        w = rng.standard_normal((co, ci, hf, wf))
        d, s = oracle.conv_direct(x, w, (sh, sw))
        t = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                                       stride=(sh, sw)).numpy()
        assert np.all(np.abs(d - t) <= 1e-12 * s + 1e-300)


def test_linearity_in_x_and_w():
    rng = np.random.default_rng(17)
    x1, x2 = rng.standard_normal((2, 2, 3, 12, 13))
    w1, w2 = rng.standard_normal((2, 4, 3, 3, 5))
    a, b = 0.75, -1.5
    f = lambda x, w: oracle.conv_direct(x, w, (2, 1))[0]
    np.testing.assert_allclose(f(a * x1 + b * x2, w1), a * f(x1, w1) + b * f(x2, w1), atol=1e-12)
    np.testing.assert_allclose(f(x1, a * w1 + b * w2), a * f(x1, w1) + b * f(x1, w2), atol=1e-12)


def test_points_match_full_output():
    rng = np.random.default_rng(18)
    x = rng.uniform(-1, 1, size=(3, 5, 20, 18))
    w = rng.standard_normal((7, 5, 4, 3))
    full, sfull = oracle.conv_direct(x, w, (2, 3))
    idx = np.stack([rng.integers(0, s, 50) for s in full.shape], axis=1)
    v, s = oracle.conv_points(x, w, idx, (2, 3))
    np.testing.assert_array_equal(v, full[tuple(idx.T)])
    np.testing.assert_array_equal(s, sfull[tuple(idx.T)])


def test_workspace_ratio_window_vs_im2col():
    """Window : im2col element counts are W_i : W_f*W_o (per channel and output row)."""
    for (hi, wi, hf, wf, sh, sw) in [(227, 227, 11, 11, 4, 4), (224, 224, 7, 7, 2, 2),
                                     (24, 24, 5, 5, 1, 1), (56, 56, 3, 7, 1, 1)]:
        x_shape, w_shape = (2, 3, hi, wi), (4, 3, hf, wf)
        _, n_win, n_col = oracle.workspace_elems(x_shape, w_shape, (sh, sw))
        wo = (wi - wf) // sw + 1
        assert n_win * wf * wo == n_col * wi


def test_bad_shapes_are_rejected():
    x = np.zeros((1, 2, 4, 4))
    with pytest.raises(ValueError):
        oracle.conv_direct(x, np.zeros((1, 2, 5, 1)))
    with pytest.raises(ValueError):
        oracle.conv_points(x, np.zeros((1, 2, 2, 2)), [[0, 1, 0, 0]])


# ---- channels-last (NHWC) layouts: the same worked example and identities,
# with channels innermost

@pytest.mark.parametrize("rule", ["ones", "ramp"])
def test_fig1_worked_example_nhwc(rule):
    gold = json.load(open(GOLD))
    x = np.transpose(_fig1_x(), (0, 2, 3, 1))           # x[0][h][w][c] = 9c + 3h + w
    w = _fig1_filter(rule)
    want = np.transpose(np.array(gold["filters"][rule]["out"], dtype=np.float64)[None], (0, 2, 3, 1))
    out, scale = oracle.conv_direct_nhwc(x, w)
    assert out.shape == (1, 2, 2, 2)
    np.testing.assert_array_equal(out, want)
    np.testing.assert_array_equal(oracle.conv_im2win_nhwc(x, w), want)
    assert np.all(scale >= np.abs(out))
    win = oracle.im2win_nhwc(x, 2, 1)
    assert win.shape == (1, 2, 6, 3)
    for c in range(3):
        np.testing.assert_array_equal(win[0, 0, :, c], np.array(gold["window_rows_channel0"]["ho0"]) + 9 * c)
        np.testing.assert_array_equal(win[0, 1, :, c], np.array(gold["window_rows_channel0"]["ho1"]) + 9 * c)


def test_im2win_nhwc_is_a_byte_copy_for_every_element_size():
    rng = np.random.default_rng(24)
    for dt in (np.uint8, np.uint16, np.float32, np.float64):
        x = rng.integers(0, 250, size=(2, 10, 11, 5)).astype(dt)
        win = oracle.im2win_nhwc(x, 4, 3)
        ho = (10 - 4) // 3 + 1
        assert win.shape == (2, ho, 11 * 4, 5)
        for h in range(ho):
            for r in range(4):
                np.testing.assert_array_equal(win[:, h, r::4, :], x[:, 3 * h + r, :, :])


def test_nhwc_window_is_the_nchw_window_with_channels_innermost():
    rng = np.random.default_rng(25)
    x = rng.integers(-100, 100, size=(2, 6, 13, 9)).astype(np.int16)
    for hf, sh in [(1, 1), (3, 1), (4, 3), (13, 2)]:
        win_nchw = oracle.im2win(x, hf, sh)
        win_nhwc = oracle.im2win_nhwc(np.transpose(x, (0, 2, 3, 1)), hf, sh)
        np.testing.assert_array_equal(win_nhwc, np.transpose(win_nchw, (0, 2, 3, 1)))


def test_nhwc_formulations_agree_exactly_on_integers():
    """direct (NHWC) == im2win over the channels-last window, bit for bit."""
    rng = np.random.default_rng(26)
    for _ in range(200):
        n, ci, hi, wi, co, hf, wf, sh, sw = _random_case(rng)
        x = rng.integers(-3, 4, size=(n, hi, wi, ci)).astype(np.float64)
        w = rng.integers(-3, 4, size=(co, ci, hf, wf)).astype(np.float64)
        d, _ = oracle.conv_direct_nhwc(x, w, (sh, sw))
        np.testing.assert_array_equal(oracle.conv_im2win_nhwc(x, w, (sh, sw)), d)
        ref, _ = oracle.conv_direct(np.transpose(x, (0, 3, 1, 2)), w, (sh, sw))
        np.testing.assert_array_equal(d, np.transpose(ref, (0, 2, 3, 1)))
        idx = np.stack([rng.integers(0, s, 8) for s in d.shape], axis=1)
        v, _ = oracle.conv_points_nhwc(x, w, idx, (sh, sw))
        np.testing.assert_array_equal(v, d[tuple(idx.T)])


def test_nhwc_one_hot_filter_is_strided_crop():
    rng = np.random.default_rng(27)
    x = rng.standard_normal((2, 23, 21, 6))
    w = np.zeros((5, 6, 5, 4))
    w[3, 4, 2, 3] = 1.0
    sh, sw = 3, 2
    out = oracle.conv_im2win_nhwc(x, w, (sh, sw))
    ho, wo = out.shape[1:3]
    crop = x[:, 2:2 + (ho - 1) * sh + 1:sh, 3:3 + (wo - 1) * sw + 1:sw, 4]
    np.testing.assert_array_equal(out[..., 3], crop)
    assert not out[..., [0, 1, 2, 4]].any()


# ---- zero padding and dilation (the pages' layers use neither; these pin the
# usual definitions against independent formulations)

def _random_pd_case(rng):
    hf, wf = (int(v) for v in rng.integers(1, 4, size=2))
    sh, sw = (int(v) for v in rng.integers(1, 3, size=2))
    ph, pw = (int(v) for v in rng.integers(0, 3, size=2))
    dh, dw = (int(v) for v in rng.integers(1, 3, size=2))
    hi = int(rng.integers(max(1, dh * (hf - 1) + 1 - 2 * ph), 9))
    wi = int(rng.integers(max(1, dw * (wf - 1) + 1 - 2 * pw), 9))
    ci = int(rng.choice([1, 2, 3, 5]))
    co = int(rng.choice([1, 4]))
    n = int(rng.choice([1, 2]))
    return (n, ci, hi, wi, co, hf, wf), (sh, sw), (ph, pw), (dh, dw)


def _dilate(w, dh, dw):
    co, ci, hf, wf = w.shape
    out = np.zeros((co, ci, dh * (hf - 1) + 1, dw * (wf - 1) + 1), dtype=w.dtype)
    out[:, :, ::dh, ::dw] = w
    return out


def test_pd_matches_torch_conv2d_fp64():
    rng = np.random.default_rng(40)
    for _ in range(80):
        (n, ci, hi, wi, co, hf, wf), st, pd, dl = _random_pd_case(rng)
        x = rng.uniform(-1, 1, size=(n, ci, hi, wi))
        w = rng.standard_normal((co, ci, hf, wf))
        d, s = oracle.conv_direct_pd(x, w, st, pd, dl)
        t = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w), stride=st,
                                       padding=pd, dilation=dl).numpy()
        assert d.shape == t.shape
        assert np.all(np.abs(d - t) <= 1e-12 * s + 1e-300)


def test_pd_is_explicit_padding_and_dilated_filter_exactly():
    """Padding = np.pad of x; dilation = the filter with zeros inserted; both through
    the unpadded direct routine, bit for bit on integers."""
    rng = np.random.default_rng(41)
    for _ in range(150):
        (n, ci, hi, wi, co, hf, wf), st, pd, dl = _random_pd_case(rng)
        x = rng.integers(-3, 4, size=(n, ci, hi, wi)).astype(np.float64)
        w = rng.integers(-3, 4, size=(co, ci, hf, wf)).astype(np.float64)
        d, _ = oracle.conv_direct_pd(x, w, st, pd, dl)
        xp = np.pad(x, ((0, 0), (0, 0), (pd[0], pd[0]), (pd[1], pd[1])))
        want, _ = oracle.conv_direct(xp, _dilate(w, *dl), st)
        np.testing.assert_array_equal(d, want)


def test_pd_reduces_to_the_unpadded_routines():
    rng = np.random.default_rng(42)
    x = rng.integers(-9, 10, size=(2, 3, 11, 13)).astype(np.float64)
    w = rng.integers(-3, 4, size=(4, 3, 3, 2)).astype(np.float64)
    d, s = oracle.conv_direct_pd(x, w, (2, 1))
    d0, s0 = oracle.conv_direct(x, w, (2, 1))
    np.testing.assert_array_equal(d, d0)
    np.testing.assert_array_equal(s, s0)
    xi = x.astype(np.int16)
    assert oracle.im2win_pd(xi, w.shape, (2, 1)).tobytes() == oracle.im2win(xi, 3, 2).tobytes()
    xc = np.ascontiguousarray(np.transpose(xi, (0, 2, 3, 1)))
    assert (oracle.im2win_pd(xc, w.shape, (2, 1), layout="nhwc").tobytes()
            == oracle.im2win_nhwc(xc, 3, 2).tobytes())


def test_pd_window_rows_of_a_hand_example():
    """x[0][0] = 3h + w (3x3), H_f = 2, padding 1: the first window row covers the
    zero row above x and x's row 0, column by column over 5 padded columns:
    (0,0) (0,0) (0,1) (0,2) (0,0); the second covers rows 0 and 1 of x."""
    x = (3 * np.arange(3)[:, None] + np.arange(3)[None, :]).astype(np.float64)[None, None]
    win = oracle.im2win_pd(x, (1, 1, 2, 2), (1, 1), (1, 1))
    assert win.shape == (1, 1, 4, 10)
    np.testing.assert_array_equal(win[0, 0, 0], [0, 0, 0, 0, 0, 1, 0, 2, 0, 0])
    np.testing.assert_array_equal(win[0, 0, 1], [0, 0, 0, 3, 1, 4, 2, 5, 0, 0])
    # dilation 2 along H: rows r*2 under ho: ho = 0 pairs the zero row with x row 1
    wind = oracle.im2win_pd(x, (1, 1, 2, 2), (1, 1), (1, 1), (2, 1))
    assert wind.shape == (1, 1, 3, 10)
    np.testing.assert_array_equal(wind[0, 0, 0], [0, 0, 0, 3, 0, 4, 0, 5, 0, 0])


@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
def test_pd_window_formulation_agrees_exactly_on_integers(layout):
    rng = np.random.default_rng(43)
    for _ in range(150):
        (n, ci, hi, wi, co, hf, wf), st, pd, dl = _random_pd_case(rng)
        shape = (n, hi, wi, ci) if layout == "nhwc" else (n, ci, hi, wi)
        x = rng.integers(-3, 4, size=shape).astype(np.float64)
        w = rng.integers(-3, 4, size=(co, ci, hf, wf)).astype(np.float64)
        d, _ = oracle.conv_direct_pd(x, w, st, pd, dl, layout)
        np.testing.assert_array_equal(oracle.conv_im2win_pd(x, w, st, pd, dl, layout), d)
        if layout == "nhwc":
            ref, _ = oracle.conv_direct_pd(np.transpose(x, (0, 3, 1, 2)), w, st, pd, dl)
            np.testing.assert_array_equal(d, np.transpose(ref, (0, 2, 3, 1)))
        nchw = d if layout == "nchw" else np.transpose(d, (0, 3, 1, 2))
        idx = np.stack([rng.integers(0, s, 6) for s in nchw.shape], axis=1)
        v, _ = oracle.conv_points_pd(x, w, idx, st, pd, dl, layout)
        np.testing.assert_array_equal(v, nchw[tuple(idx.T)])


def test_pd_bad_shapes_are_rejected():
    x = np.zeros((1, 2, 4, 4))
    with pytest.raises(ValueError):   # dilated extent 7 > 4 + 2
        oracle.conv_direct_pd(x, np.zeros((1, 2, 3, 3)), (1, 1), (1, 1), (3, 3))
    with pytest.raises(ValueError):
        oracle.conv_direct_pd(x, np.zeros((1, 2, 3, 3)), (1, 1), (-1, 0))
