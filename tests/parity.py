"""Shared helpers for the GPU parity tests (compare the CUDA path with the oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the parity bar, per output: |gpu - oracle| <= TOL * S with
# S = sum |x||w| over the output's terms. fp32: products are exact in fp64 and an
# fp32 accumulation of K terms of random sign errs by ~sqrt(K) * 2^-24 * S; 1e-5
# leaves a wide margin (the worst case K * 2^-24 is not reached by random data).
# fp16/bf16: inputs are exact, accumulation is fp32, and the final rounding to
# the input dtype costs at most 2^-11 (fp16) or 2^-8 (bf16) of |out| <= S.
TOL = {torch.float32: 1e-5, torch.float16: 4e-3, torch.bfloat16: 4e-3}


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_within(got: np.ndarray, want: np.ndarray, scale: np.ndarray, tol: float, what=""):
    err = np.abs(got - want)
    bound = tol * scale
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; worst at flat "
            f"{i}: got {got.ravel()[i]!r} want {want.ravel()[i]!r} err {err.ravel()[i]:.3e} "
            f"bound {bound.ravel()[i]:.3e}")


def check_full(out_gpu: torch.Tensor, x: torch.Tensor, w: torch.Tensor, stride, what=""):
    want, scale = oracle.conv_direct(to_f64(x), to_f64(w), stride)
    assert tuple(out_gpu.shape) == want.shape, (tuple(out_gpu.shape), want.shape)
    assert_within(to_f64(out_gpu), want, scale, TOL[out_gpu.dtype], what)


def check_sampled(out_gpu: torch.Tensor, x_cpu: torch.Tensor, w_cpu: torch.Tensor, stride,
                  images=(0, -1), n_points=4096, seed=0, what=""):
    """Full outputs of a few images plus random points across the batch."""
    N = out_gpu.shape[0]
    tol = TOL[out_gpu.dtype]
    w64 = to_f64(w_cpu)
    for n in sorted({i % N for i in images}):
        want, scale = oracle.conv_direct(to_f64(x_cpu[n:n + 1]), w64, stride)
        assert_within(to_f64(out_gpu[n:n + 1]), want, scale, tol, f"{what} image {n}")
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.integers(0, s, n_points) for s in out_gpu.shape], axis=1)
    got = out_gpu[tuple(torch.from_numpy(idx.T.copy()).to(out_gpu.device))]
    got = to_f64(got)
    for n in np.unique(idx[:, 0]):
        sel = idx[:, 0] == n
        loc = idx[sel].copy()
        loc[:, 0] = 0
        vals, scale = oracle.conv_points(to_f64(x_cpu[n:n + 1]), w64, loc, stride)
        assert_within(got[sel], vals, scale, tol, f"{what} sampled image {n}")
