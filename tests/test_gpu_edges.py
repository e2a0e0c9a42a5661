"""Edge cases of every call, both layouts, against the oracle: empty batches,
degenerate extents (one output row or column, one channel), strides that skip
input rows and columns, the widest row a tensor-core tile holds, many output
channel tiles and long reductions."""
import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl
from parity import TOL, assert_within, to_f64

pytestmark = pytest.mark.gpu
LAYOUTS = {"nchw": mec.NCHW, "nhwc": mec.NHWC}


def _run(x, w, stride, layout, fused):
    lo = LAYOUTS[layout]
    xd, wd = x.cuda(), w.cuda()
    if fused:
        return mec.conv_fused_ex(xd, wd, stride, layout=lo)
    win = mec.transform_ex(xd, w.shape[2], w.shape[3], stride, layout=lo)
    return mec.conv_ex(win, wd, tuple(x.shape), stride, layout=lo)


def _check(case, dt, layout, fused, seed=0):
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = case
    layer = wl.Layer("edge", N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, seed=seed + sum(case))
    x, w = wl.make_inputs(layer, dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    out = _run(x, w, (s_h, s_w), layout, fused)
    torch.cuda.synchronize()
    want, scale = oracle.conv_direct_pd(to_f64(x), to_f64(w), (s_h, s_w), layout=layout)
    assert tuple(out.shape) == want.shape
    assert_within(to_f64(out), want, scale, TOL[out.dtype], f"{dt} {layout} {case} fused={fused}")


EDGE = [  # N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w
    (2, 8, 7, 9, 16, 7, 9, 1, 1),        # the filter covers the input: one output pixel
    (1, 16, 5, 40, 24, 5, 3, 2, 1),      # one output row
    (1, 16, 40, 5, 24, 3, 5, 1, 2),      # one output column
    (2, 8, 17, 23, 8, 2, 3, 3, 4),       # strides larger than the filter: rows and columns skipped
    (1, 1, 12, 13, 1, 3, 3, 1, 1),       # one input and one output channel
    (1, 16, 3, 512, 32, 3, 3, 1, 1),     # a 512-position row: the widest tile row
    (1, 16, 6, 20, 300, 3, 3, 1, 1),     # three output-channel tiles, the last ragged
    (1, 512, 6, 10, 64, 3, 3, 1, 1),     # a long reduction: 32 sixteen-channel chunks
]


@pytest.mark.parametrize("fused", [False, True], ids=["window", "fused"])
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: "x".join(map(str, c)))
def test_edge_shapes(case, dt, layout, fused):
    _check(case, dt, layout, fused)


@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("dt", ["f32", "f16"])
def test_empty_batch_writes_nothing(dt, layout):
    """N = 0: every call returns without reading or writing (the output buffer is
    a sentinel-filled tensor of one element)."""
    tdt = wl.DTYPES[dt]
    lo = LAYOUTS[layout]
    x = torch.zeros((0, 4, 9, 9) if layout == "nchw" else (0, 9, 9, 4), dtype=tdt, device="cuda")
    w = torch.zeros((8, 4, 3, 3), dtype=tdt, device="cuda")
    sentinel = torch.full((8,), 3.0, dtype=tdt, device="cuda")
    args = (0, 4, 9, 9, 8, 3, 3, 1, 1, 0, 0, 1, 1)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    mec.im2win_transform_ex(x, sentinel, *args, lo)
    mec.im2win_conv_ex(sentinel, w, sentinel, ws, *args, lo)
    mec.im2win_conv_fused_ex(x, w, sentinel, ws, *args, lo)
    torch.cuda.synchronize()
    assert torch.all(sentinel == 3.0)
    assert mec.im2win_workspace_size_ex(mec.OP_TRANSFORM, *args, lo, mec._binding._DTYPE[tdt]) == 0


def test_rows_wider_than_a_tile():
    """Rows of more than 512 positions: NCHW falls back to the expand kernel; the
    channels-last tensor-core calls refuse with IM2WIN_ERR_UNSUPPORTED (fp32 runs)."""
    case = (1, 16, 4, 600, 16, 3, 3, 1, 1)
    _check(case, "f16", "nchw", True)
    _check(case, "f32", "nhwc", True)
    layer = wl.Layer("wide", *case, seed=1)
    x, w = wl.make_inputs(layer, "f16")
    xc = x.permute(0, 2, 3, 1).contiguous().cuda()
    with pytest.raises(mec.Im2winError) as err:
        mec.conv_fused_ex(xc, w.cuda(), (1, 1), layout=mec.NHWC)
    assert err.value.status == mec._binding.ERR_UNSUPPORTED
