"""Tolerances of the parity tests (GPU path vs the float64 oracle).

fp32 outputs: per output tensor, max_i |x_i - r_i| / max(|r_i|, rms(r)) <= 1e-5
    (relative error, with the tensor's RMS as the floor of the denominator so
    that entries near zero are judged against the tensor's scale).
bf16-input paths with fp32 accumulation: per output tensor, e_i =
    |x_i - r_i| / rms(r); max_i e_i <= 2e-2 and mean_i e_i <= 5e-3.
"""
import numpy as np
import torch

FP32_REL = 1e-5
BF16_MAX = 2e-2
BF16_MEAN = 5e-3


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(x, r):
    x, r = _np(x), _np(r)
    assert x.shape == r.shape, (x.shape, r.shape)
    if r.size == 0:
        return 0.0
    assert np.all(np.isfinite(x)), "non-finite values in GPU output"
    rms = float(np.sqrt(np.mean(r * r)))
    floor = rms if rms > 0 else 1.0
    return float(np.max(np.abs(x - r) / np.maximum(np.abs(r), floor)))


def rms_err(x, r):
    x, r = _np(x), _np(r)
    assert x.shape == r.shape, (x.shape, r.shape)
    if r.size == 0:
        return 0.0, 0.0
    assert np.all(np.isfinite(x)), "non-finite values in GPU output"
    rms = float(np.sqrt(np.mean(r * r)))
    e = np.abs(x - r) / (rms if rms > 0 else 1.0)
    return float(e.max()), float(e.mean())


def assert_fp32(name, x, r, tol=FP32_REL):
    e = rel_err(x, r)
    assert e <= tol, f"{name}: relative error {e:.3e} > {tol:.1e}"
    return e


def assert_bf16(name, x, r, tol_max=BF16_MAX, tol_mean=BF16_MEAN):
    mx, mean = rms_err(x, r)
    assert mx <= tol_max and mean <= tol_mean, f"{name}: max {mx:.3e} (<= {tol_max}), mean {mean:.3e} (<= {tol_mean})"
    return mx, mean
