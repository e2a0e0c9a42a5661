"""Seeded synthetic workloads: the convolution layers and their input recipe.

This module holds shapes, seeds and random draws only -- none of the method's
arithmetic -- so that the CUDA path's tests and the oracle can be fed the very
same tensors.

Recipe (one reading, stated once): ``numpy.random.default_rng(seed)`` (PCG64);
x ~ U[-1, 1] is drawn first, image by image, then w ~ N(0, 1/fan_in) with
fan_in = C_i*H_f*W_f (std = 1/sqrt(fan_in)); both are drawn in float64, cast to
float32 and then to the dtype under test with round-to-nearest-even. The
rounded tensor *is* the input: the oracle widens exactly those values.

The layer shapes cv1, cv4 and cv5 are rows of Table I of "Enabling
Memory-efficient Im2win Convolution with Multi-precision Support on GPU CUDA and
Tensor Cores"; the batch sizes, the kernel-size sweep and the tiny correctness
case are the benchmark's own choices (the page prints no batch size).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    C_i: int
    H_i: int
    W_i: int
    C_o: int
    H_f: int
    W_f: int
    s_h: int
    s_w: int
    seed: int
    dtypes: tuple = field(default=("f32",))
    pad: tuple = (0, 0)   # zero padding (p_h, p_w)
    dil: tuple = (1, 1)   # dilation (d_h, d_w)

    @property
    def shape_args(self):
        return (self.N, self.C_i, self.H_i, self.W_i, self.C_o, self.H_f, self.W_f,
                self.s_h, self.s_w)

    @property
    def plain(self) -> bool:
        return tuple(self.pad) == (0, 0) and tuple(self.dil) == (1, 1)

    @property
    def out_hw(self):
        return ((self.H_i + 2 * self.pad[0] - self.dil[0] * (self.H_f - 1) - 1) // self.s_h + 1,
                (self.W_i + 2 * self.pad[1] - self.dil[1] * (self.W_f - 1) - 1) // self.s_w + 1)

    def with_batch(self, n: int) -> "Layer":
        return Layer(self.name, n, self.C_i, self.H_i, self.W_i, self.C_o, self.H_f,
                     self.W_f, self.s_h, self.s_w, self.seed, self.dtypes, self.pad, self.dil)


TINY = Layer("tiny_3x32x32_8x3x3", 1, 3, 32, 32, 8, 3, 3, 1, 1, seed=0, dtypes=("f32",))
CV1 = Layer("cv1", 128, 3, 227, 227, 96, 11, 11, 4, 4, seed=1, dtypes=("f16", "f32"))
CV4 = Layer("cv4", 128, 64, 224, 224, 64, 7, 7, 2, 2, seed=2, dtypes=("f16",))
CV5 = Layer("cv5", 128, 96, 24, 24, 256, 5, 5, 1, 1, seed=3, dtypes=("bf16",))
SWEEP = tuple(
    Layer(f"sweep_{hf}x{wf}", 64, 128, 56, 56, 128, hf, wf, 1, 1, seed=400 + i,
          dtypes=("f32", "bf16"))
    for i, (hf, wf) in enumerate([(1, 1), (3, 3), (5, 5), (7, 7), (11, 11), (3, 7)]))
# Table I layers with no config of their own (same kernels, odd input pitches).
CV2 = Layer("cv2", 128, 3, 231, 231, 96, 11, 11, 4, 4, seed=5, dtypes=("f16", "f32"))
CV3 = Layer("cv3", 128, 3, 227, 227, 64, 7, 7, 2, 2, seed=6, dtypes=("f16", "f32"))

ALL = (TINY, CV1, CV4, CV5) + SWEEP + (CV2, CV3)

# Zero padding and dilation (not on the pages; the usual CNN options): the 3x3
# sweep layer as a "same" convolution, and with dilation 2.
SAME_3x3 = Layer("sweep_3x3_pad1", 64, 128, 56, 56, 128, 3, 3, 1, 1, seed=500, dtypes=("f32", "bf16"),
                 pad=(1, 1))
DIL_3x3 = Layer("sweep_3x3_pad2_dil2", 64, 128, 56, 56, 128, 3, 3, 1, 1, seed=501, dtypes=("f32", "bf16"),
                pad=(2, 2), dil=(2, 2))
PADDED = (SAME_3x3, DIL_3x3)


def make_inputs(layer: Layer, dtype: str, seed: int | None = None, n_images: int | None = None):
    """Return CPU tensors (x, w) of `dtype` for `layer`, drawn per the recipe.

    `n_images` draws only the first images of the batch (the stream is consumed
    image by image, so they equal the leading images of the full draw; w is then
    drawn from a fresh generator state advanced past all N images).
    """
    rng = np.random.default_rng(layer.seed if seed is None else seed)
    tdt = DTYPES[dtype]
    per_img = layer.C_i * layer.H_i * layer.W_i
    keep = layer.N if n_images is None else min(n_images, layer.N)
    x = torch.empty((keep, layer.C_i, layer.H_i, layer.W_i), dtype=tdt)
    for n in range(layer.N):
        if n < keep:
            a = rng.uniform(-1.0, 1.0, size=per_img)
            x[n] = torch.from_numpy(a.astype(np.float32)).reshape(x.shape[1:]).to(tdt)
        else:
            rng.uniform(-1.0, 1.0, size=per_img)
    fan_in = layer.C_i * layer.H_f * layer.W_f
    w64 = rng.normal(0.0, 1.0 / np.sqrt(fan_in), size=(layer.C_o, layer.C_i, layer.H_f, layer.W_f))
    w = torch.from_numpy(w64.astype(np.float32)).to(tdt)
    return x, w


def make_int_inputs(layer: Layer, dtype: str, seed: int, x_range=2, w_range=2, density=1.0):
    """Integer-valued inputs in [-range, range] (optionally sparse).

    Every product and partial sum of such inputs is a small integer, exactly
    representable in fp32, so an fp32 accumulation is exact in any order.
    """
    rng = np.random.default_rng(seed)
    x = rng.integers(-x_range, x_range + 1, size=(layer.N, layer.C_i, layer.H_i, layer.W_i))
    w = rng.integers(-w_range, w_range + 1, size=(layer.C_o, layer.C_i, layer.H_f, layer.W_f))
    if density < 1.0:
        x = x * (rng.random(x.shape) < density)
        w = w * (rng.random(w.shape) < density)
    tdt = DTYPES[dtype]
    return (torch.from_numpy(x.astype(np.float32)).to(tdt),
            torch.from_numpy(w.astype(np.float32)).to(tdt))
