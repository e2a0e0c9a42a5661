"""Host-side checks of the convolution planner through the plan query (no GPU
needed): for every layer of the parity set, both layouts and both convolution
calls, and for random shapes with padding and dilation, the tensor-core tap
kernel's tiling fits the SM (shared memory, TMEM columns, one CTA per SM),
covers the output exactly, and agrees with the workspace query on which shapes
are supported."""
import math

import numpy as np
import pytest

import memory_efficient_cnn_gb300 as mec
from memory_efficient_cnn_gb300 import build as mbuild
from memory_efficient_cnn_gb300 import workloads as wl

SMEM_PER_CTA = 227 * 1024      # opt-in shared memory per CTA
SMEM_PER_SM = 228 * 1024       # shared memory of one SM
TMEM_COLUMNS = 512             # the accumulator allocation of a CTA
SMS = 152
OPS = {"window": mec.OP_CONV, "fused": mec.OP_CONV_FUSED}
LAYOUTS = {"nchw": mec.NCHW, "nhwc": mec.NHWC}


@pytest.fixture(scope="module", autouse=True)
def lib():
    mbuild.build()
    return mec.lib()


def _out_hw(H_i, W_i, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w):
    return ((H_i + 2 * p_h - d_h * (H_f - 1) - 1) // s_h + 1,
            (W_i + 2 * p_w - d_w * (W_f - 1) - 1) // s_w + 1)


def check_plan(info, shape, pad=(0, 0), dil=(1, 1), layout=mec.NCHW, dtype=mec.F16, sms=SMS, fused=True):
    """The invariants every plan keeps."""
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = shape
    H_o, _ = _out_hw(H_i, W_i, H_f, W_f, s_h, s_w, *pad, *dil)
    if dtype == mec.F32:
        assert info["kernel"] == mec.KERNEL_F32
        return
    assert info["kernel"] in (mec.KERNEL_TAP, mec.KERNEL_EXPAND)
    if info["kernel"] == mec.KERNEL_EXPAND:
        # the fallback exists for plain NCHW only
        assert layout == mec.NCHW and pad == (0, 0) and dil == (1, 1)
        assert info["tap_mode"] == -1
        return
    assert 0 < info["smem_bytes"] <= SMEM_PER_CTA
    assert 2 * info["smem_bytes"] > SMEM_PER_SM  # one CTA per SM: its 512 TMEM columns are the SM's
    assert info["rows_per_tile"] >= 1 and info["pitch"] >= 1
    if info["stacked"] == 2:
        # transposed stacking: the tile's positions (plus the shifted one) in M blocks
        # of 128 TMEM lanes, two buffers of 256 columns (128 per M block)
        nmb = math.ceil((info["rows_per_tile"] * info["pitch"] + 1) / 128)
        assert nmb <= 2
        assert info["tmem_columns"] == info["tmem_read_end"] == 256 + 128 * nmb <= TMEM_COLUMNS
    else:
        # the MMAs write, and the epilogue reads, every column of the widest tile (plus
        # the shifted one when stacked), all inside the CTA's allocation
        need = info["rows_per_tile"] * info["pitch"] + info["stacked"]
        assert need <= info["tmem_columns"] <= TMEM_COLUMNS
        assert need <= info["tmem_read_end"] <= TMEM_COLUMNS
    assert info["tiles"] == N * math.ceil(C_o / 128) * math.ceil(H_o / info["rows_per_tile"])
    assert info["grid"] == min(sms, info["tiles"])
    assert info["filter_stage_taps"] >= 1 and info["filter_stages"] >= 2 and info["slab_stages"] >= 2
    if info["stacked"]:
        # two taps of one filter row share an MMA: no column dilation; row dilation
        # only from the window tensor, whose rows are already the dilated ones
        assert C_o <= 64 and dil[1] == 1 and (dil[0] == 1 or not fused)
    if layout == mec.NCHW:
        assert info["tap_mode"] in (0, 1, 2)
    else:
        assert info["tap_mode"] in (1, 2, 3)


@pytest.mark.parametrize("op", OPS, ids=str)
@pytest.mark.parametrize("layout", LAYOUTS, ids=str)
@pytest.mark.parametrize("layer", wl.ALL + wl.PADDED, ids=lambda l: l.name)
def test_parity_layers_plan_within_the_sm(layer, layout, op):
    for dt in (mec.F32, mec.F16, mec.BF16):
        info = mec.im2win_plan(OPS[op], *layer.shape_args, *layer.pad, *layer.dil,
                               layout=LAYOUTS[layout], dtype=dt, sms=SMS)
        check_plan(info, layer.shape_args, tuple(layer.pad), tuple(layer.dil), LAYOUTS[layout], dt,
                   fused=op == "fused")


@pytest.mark.parametrize("layer", [wl.CV4, wl.CV5] + [l for l in wl.SWEEP if l.H_f >= 3],
                         ids=lambda l: l.name)
def test_large_channel_layers_run_the_tap_kernel(layer):
    for layout in LAYOUTS.values():
        for op in OPS.values():
            info = mec.im2win_plan(op, *layer.shape_args, layout=layout, dtype=mec.BF16, sms=SMS)
            assert info["kernel"] == mec.KERNEL_TAP
            assert info["grid"] == SMS
            assert (info["stacked"] > 0) == (layer.C_o <= 64)


def test_default_sm_count_without_a_device_is_a_full_grid():
    info = mec.im2win_plan(mec.OP_CONV_FUSED, *wl.CV5.shape_args, dtype=mec.BF16)
    assert info["kernel"] == mec.KERNEL_TAP and info["grid"] >= 1


def test_plan_argument_errors():
    args = wl.CV5.shape_args
    with pytest.raises(mec.Im2winError) as e:
        mec.im2win_plan(mec.OP_TRANSFORM, *args)
    assert e.value.status == mec._binding.ERR_INVALID_ARG
    with pytest.raises(mec.Im2winError):
        mec.im2win_plan(mec.OP_CONV, *args, layout=7)
    with pytest.raises(mec.Im2winError):
        mec.im2win_plan(mec.OP_CONV, *args, dtype=9)
    with pytest.raises(mec.Im2winError):
        mec.im2win_plan(mec.OP_CONV, 1, 4, 5, 5, 8, 7, 3, 1, 1)  # filter taller than the input


def test_random_shapes_plan_within_the_sm_and_agree_with_the_workspace_query():
    rng = np.random.default_rng(2024)
    planned = 0
    for _ in range(250):
        H_f, W_f = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        s_h, s_w = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        p_h, p_w = (int(rng.integers(0, 4)), int(rng.integers(0, 4))) if rng.random() < 0.4 else (0, 0)
        d_h, d_w = (int(rng.integers(1, 4)), int(rng.integers(1, 4))) if rng.random() < 0.3 else (1, 1)
        H_i = int(rng.integers(d_h * (H_f - 1) + 1, 80))
        W_i = int(rng.integers(d_w * (W_f - 1) + 1, 300))
        C_i = int(rng.choice([1, 3, 8, 16, 24, 64, 96, 130]))
        C_o = int(rng.choice([1, 8, 32, 64, 96, 128, 200, 256]))
        shape = (int(rng.integers(1, 5)), C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w)
        for layout in LAYOUTS.values():
            for op in OPS.values():
                dt = mec.BF16 if rng.random() < 0.5 else mec.F16
                try:
                    info = mec.im2win_plan(op, *shape, p_h, p_w, d_h, d_w, layout=layout, dtype=dt, sms=SMS)
                except mec.Im2winError as err:
                    assert err.status == mec._binding.ERR_UNSUPPORTED
                    continue
                planned += 1
                check_plan(info, shape, (p_h, p_w), (d_h, d_w), layout, dt, fused=op == mec.OP_CONV_FUSED)
                ws = mec.im2win_workspace_size_ex(op, *shape, p_h, p_w, d_h, d_w, layout, dt)
                assert ws > 256  # status block + re-laid filter
    assert planned > 500
