"""The seeded input recipe is deterministic and prefix-consistent."""
import torch

from memory_efficient_cnn_gb300 import workloads as wl


def test_same_seed_same_tensors_and_prefix():
    layer = wl.TINY.with_batch(4)
    x1, w1 = wl.make_inputs(layer, "f32")
    x2, w2 = wl.make_inputs(layer, "f32", n_images=2)
    assert torch.equal(x1[:2], x2) and torch.equal(w1, w2)
    assert x1.abs().max() <= 1.0
    # the fp16 draw is the RNE rounding of the fp32 draw
    xh, wh = wl.make_inputs(layer, "f16")
    assert torch.equal(xh, x1.to(torch.float16)) and torch.equal(wh, w1.to(torch.float16))


def test_weight_scale_follows_fan_in():
    layer = wl.Layer("t", 1, 16, 8, 8, 256, 3, 3, 1, 1, seed=9)
    _, w = wl.make_inputs(layer, "f32")
    std = w.double().std().item()
    assert abs(std - (16 * 9) ** -0.5) < 0.1 * (16 * 9) ** -0.5


def test_int_inputs_are_small_integers():
    x, w = wl.make_int_inputs(wl.TINY, "bf16", seed=3)
    assert torch.equal(x.float(), x.float().round()) and x.abs().max() <= 2
    assert torch.equal(w.float(), w.float().round()) and w.abs().max() <= 2
