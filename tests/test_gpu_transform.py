"""GPU parity of the im2win transform: bit-exact against the oracle's byte copy."""
import numpy as np
import pytest
import torch

import memory_efficient_cnn_gb300 as mec
import oracle
from memory_efficient_cnn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
RAW = {torch.float32: np.uint32, torch.float16: np.uint16, torch.bfloat16: np.uint16}


def _raw(t: torch.Tensor) -> np.ndarray:
    v = t.detach().cpu().contiguous()
    bits = v.view(torch.int32 if v.element_size() == 4 else torch.int16).numpy()
    return bits.view(RAW[t.dtype])


def _check(x_cpu, H_f, s_h):
    win = mec.transform(x_cpu.cuda(), H_f, s_h)
    torch.cuda.synchronize()
    want = oracle.im2win(_raw(x_cpu), H_f, s_h)
    got = _raw(win)
    assert got.shape == want.shape
    assert got.tobytes() == want.tobytes()


CASES = [  # N, C_i, H_i, W_i, H_f, s_h
    (2, 3, 32, 32, 3, 1), (3, 5, 37, 227, 11, 4), (1, 7, 29, 231, 7, 2), (2, 2, 9, 13, 9, 1),
    (1, 3, 40, 5, 1, 1), (2, 4, 50, 17, 3, 5), (1, 1, 300, 3, 2, 1), (5, 3, 24, 24, 5, 1),
    (1, 2, 6, 12000, 3, 2),  # one output row of input exceeds the default band budget
    # many small planes: several whole planes per CTA, the last group ragged
    (64, 64, 11, 13, 3, 2), (27, 113, 7, 9, 2, 1),
    # rows of whole 16-byte vectors (16-bit: staged as vertical pairs): bands of a tall
    # plane, H_f >= 8, H_f = 1, many planes per CTA, stride = H_f, one output row
    (1, 3, 200, 64, 7, 1), (2, 4, 30, 16, 11, 3), (3, 5, 10, 8, 1, 1), (64, 32, 12, 8, 2, 2),
    (1, 2, 50, 96, 4, 4), (2, 3, 9, 40, 9, 1),
    # 16-bit rows of whole 16-byte vectors, H_f up to 12, item counts not a multiple of 32
    (2, 3, 20, 24, 12, 2), (1, 2, 14, 16, 6, 1), (1, 3, 12, 8, 8, 2), (2, 2, 15, 32, 10, 5),
    (1, 1, 5, 8, 3, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_transform_small_bit_exact(case, dt):
    N, C_i, H_i, W_i, H_f, s_h = case
    g = torch.Generator().manual_seed(hash(case) & 0xFFFF)
    x = (torch.rand((N, C_i, H_i, W_i), generator=g) * 2 - 1).to(DT[dt])
    _check(x, H_f, s_h)


def test_transform_empty_batch_is_a_noop():
    x = torch.zeros((0, 3, 8, 8), device="cuda")
    win = mec.transform(x, 3, 1)
    assert win.shape == (0, 3, 6, 24)


@pytest.mark.parametrize("W_i", [227, 64])
def test_transform_does_not_write_past_the_window(W_i):
    x = torch.randn(2, 3, 31, W_i, dtype=torch.float16)
    H_f, s_h = 11, 4
    H_o = (31 - H_f) // s_h + 1
    n = 2 * 3 * H_o * W_i * H_f
    buf = torch.full((n + 64,), 7, dtype=torch.float16, device="cuda")
    mec.im2win_transform(x.cuda(), buf, 1, H_f, 1, s_h, 1)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7)
    assert _raw(buf[:n]).tobytes() == oracle.im2win(_raw(x), H_f, s_h).tobytes()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_transform_window_not_16_byte_aligned_is_refused(dt):
    # the entry points take 16-byte aligned buffers; one element past a boundary is
    # refused before any launch, and the buffer is left as it was
    x = torch.zeros((2, 3, 20, 32), dtype=DT[dt], device="cuda")
    H_f, s_h = 5, 2
    H_o = (20 - H_f) // s_h + 1
    n = 2 * 3 * H_o * 32 * H_f
    buf = torch.full((n + 16,), 3, dtype=DT[dt], device="cuda")
    with pytest.raises(mec.Im2winError, match="aligned"):
        mec.im2win_transform(x, buf[1:n + 1], 1, H_f, 1, s_h, 1)
    torch.cuda.synchronize()
    assert torch.all(buf == 3)


@pytest.mark.parametrize("layer,dt", [(wl.CV1, "f16"), (wl.CV1, "f32"), (wl.CV2, "f16"), (wl.CV3, "f32"),
                                      (wl.CV5, "bf16")]
                         + [(l, "bf16") for l in wl.SWEEP] + [(wl.SWEEP[1], "f32"), (wl.SWEEP[4], "f32")],
                         ids=lambda v: getattr(v, "name", v))
def test_transform_full_size_bit_exact(layer, dt):
    x, _ = wl.make_inputs(layer, dt)
    _check(x, layer.H_f, layer.s_h)


def test_transform_cv4_full_size_sampled_images():
    layer = wl.CV4
    x, _ = wl.make_inputs(layer, "f16")
    win = mec.transform(x.cuda(), layer.H_f, layer.s_h)
    torch.cuda.synchronize()
    for n in (0, 1, 63, 127):
        want = oracle.im2win(_raw(x[n:n + 1]), layer.H_f, layer.s_h)
        assert _raw(win[n:n + 1]).tobytes() == want.tobytes(), n
