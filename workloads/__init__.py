"""Seeded synthetic inputs for the five workloads, shared by tests and bench.

This module holds input recipes only -- shapes, distributions and seeds -- and
none of the method's arithmetic.  Values are drawn on the CPU with NumPy's
PCG64, rounded once to the dtype the library consumes (float32 or bfloat16),
and returned as CPU torch tensors; the GPU path copies those exact values to
the device and the oracle widens the same values to float64.

Workloads (each runnable at any smaller shape with the same distributions):

* ``scan_small``  diagonal scan forward, fp32: B=1, T=1024, D=64;
  a ~ U(0.8, 0.999), b ~ N(0, 1), h0 = 0.
* ``scan``        diagonal scan forward+backward, fp32: B=8, T=4096, D=1024;
  a = exp(-0.05 softplus(z)), z ~ N(0, 1); b ~ N(0, 1); h0 ~ N(0, 1);
  upstream dL/dh ~ N(0, 1).
* ``selective``   selective scan forward+backward: B=4, T=8192, D=2048, N=16;
  x, B_t, C_t bf16 ~ N(0, 1); Delta = softplus(N(-2, 0.5)) fp32 per (t, d);
  A[d, n] = -(n + 1); h0 = 0; dL/dy ~ N(0, 1) fp32.
* ``la_const``    chunkwise linear attention, per-head constant decay:
  B=4, H=16, T=8192, d_k=d_v=64; q, k, v bf16 ~ N(0, 1)/8;
  lambda_h = 1 - 2^-(5 + 8h/H); chunk 64; S0 = 0; dL/do ~ N(0, 1) bf16.
* ``la_long``     long-context linear attention, data-dependent scalar decay:
  B=1, H=32, T=65536, d_k=d_v=128; q, k, v bf16 ~ N(0, 1)/sqrt(128);
  log a = -softplus(N(0, 1))/16 per (head, token); S0 ~ N(0, 0.01^2) fp32;
  chunk 128; dL/do ~ N(0, 1) bf16.

* ``gla``         gated linear attention, one decay per key dimension (the next
  row after the five above): B=2, H=16, T=16384, d_k=d_v=128; q, k, v bf16
  ~ N(0, 1)/sqrt(128); log a = -softplus(N(0, 1))/16 per (head, token, key
  dimension); S0 ~ N(0, 0.01^2) fp32; chunk 64; dL/do ~ N(0, 1) bf16.

* ``delta``       delta rule with a decay per head (Gated DeltaNet): B=4, H=32,
  T=4096, d_k=d_v=128; q, v bf16 ~ N(0, 1)/sqrt(128); k ~ N(0, 1) per
  element, L2-normalised per token, then bf16; log a = -softplus(N(0, 1))/16
  and beta = sigmoid(N(0, 1)) per (head, token); S0 ~ N(0, 0.01^2) fp32;
  upstream dL/do ~ N(0, 1) bf16; chunk 64.

The second parameter of N(mu, s) is read as a standard deviation.
"""
from __future__ import annotations

import math

import numpy as np
import torch

WORKLOADS = {
    "scan_small": dict(kind="scan_diag", B=1, T=1024, D=64, seed=1, backward=False),
    "scan": dict(kind="scan_diag", B=8, T=4096, D=1024, seed=2, backward=True),
    "selective": dict(kind="selective", B=4, T=8192, D=2048, N=16, seed=3, backward=True),
    "la_const": dict(kind="chunk_la", B=4, H=16, T=8192, dk=64, dv=64, chunk=64, seed=4, backward=True),
    "la_long": dict(kind="chunk_la", B=1, H=32, T=65536, dk=128, dv=128, chunk=128, seed=5, backward=True),
    "gla": dict(kind="gla", B=2, H=16, T=16384, dk=128, dv=128, chunk=64, seed=6, backward=True),
    "delta": dict(kind="delta", B=4, H=32, T=4096, dk=128, dv=128, chunk=64, seed=7, backward=True),
}


def _rng(seed: int, offset: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(offset)]))


def _normal(seed, offset, shape, mean=0.0, std=1.0) -> np.ndarray:
    z = _rng(seed, offset).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    if mean != 0.0:
        z += np.float32(mean)
    return z


def _softplus(z: np.ndarray) -> np.ndarray:
    z64 = z.astype(np.float64)
    return np.where(z64 > 20.0, z64, np.log1p(np.exp(np.minimum(z64, 20.0))))


def _f32(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))


def _bf16(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


# ---------------------------------------------------------------- diagonal scan
def scan_small_inputs(B=1, T=1024, D=64, seed=1):
    """a ~ U(0.8, 0.999), b ~ N(0,1), h0 = 0 (fp32)."""
    a = _rng(seed, 0).uniform(0.8, 0.999, size=(B, T, D)).astype(np.float32)
    b = _normal(seed, 1, (B, T, D))
    return dict(a=_f32(a), b=_f32(b), h0=None)


def scan_inputs(B=8, T=4096, D=1024, seed=2):
    """a = exp(-0.05 softplus(z)), b, h0, dh ~ N(0,1) (fp32)."""
    z = _normal(seed, 0, (B, T, D))
    a = np.exp(-0.05 * _softplus(z)).astype(np.float32)
    b = _normal(seed, 1, (B, T, D))
    h0 = _normal(seed, 2, (B, D))
    dh = _normal(seed, 3, (B, T, D))
    return dict(a=_f32(a), b=_f32(b), h0=_f32(h0), dh=_f32(dh))


# ---------------------------------------------------------------- selective scan
def selective_inputs(B=4, T=8192, D=2048, N=16, seed=3):
    x = _bf16(_normal(seed, 0, (B, T, D)))
    Bm = _bf16(_normal(seed, 1, (B, T, N)))
    Cm = _bf16(_normal(seed, 2, (B, T, N)))
    delta = _f32(_softplus(_normal(seed, 3, (B, T, D), mean=-2.0, std=0.5)))
    A = _f32(-np.broadcast_to(np.arange(1, N + 1, dtype=np.float32), (D, N)))
    dy = _f32(_normal(seed, 4, (B, T, D)))
    return dict(x=x, delta=delta, A=A, Bm=Bm, Cm=Cm, h0=None, dy=dy)


# ---------------------------------------------------------------- linear attention
def la_const_inputs(B=4, H=16, T=8192, dk=64, dv=64, seed=4):
    q = _bf16(_normal(seed, 0, (B, H, T, dk), std=1.0 / 8.0))
    k = _bf16(_normal(seed, 1, (B, H, T, dk), std=1.0 / 8.0))
    v = _bf16(_normal(seed, 2, (B, H, T, dv), std=1.0 / 8.0))
    lam = 1.0 - 2.0 ** (-(5.0 + 8.0 * np.arange(H, dtype=np.float64) / H))
    log_a = np.broadcast_to(np.log(lam)[None, :, None], (B, H, T)).astype(np.float32)
    dO = _bf16(_normal(seed, 3, (B, H, T, dv)))
    return dict(q=q, k=k, v=v, log_a=_f32(log_a), S0=None, dO=dO)


def la_long_inputs(B=1, H=32, T=65536, dk=128, dv=128, seed=5):
    s = 1.0 / math.sqrt(dk)
    q = _bf16(_normal(seed, 0, (B, H, T, dk), std=s))
    k = _bf16(_normal(seed, 1, (B, H, T, dk), std=s))
    v = _bf16(_normal(seed, 2, (B, H, T, dv), std=s))
    log_a = (-_softplus(_normal(seed, 3, (B, H, T))) / 16.0).astype(np.float32)
    S0 = _normal(seed, 4, (B, H, dk, dv), std=0.01)
    dO = _bf16(_normal(seed, 5, (B, H, T, dv)))
    return dict(q=q, k=k, v=v, log_a=_f32(log_a), S0=_f32(S0), dO=dO)


def gla_inputs(B=2, H=16, T=16384, dk=128, dv=128, seed=6):
    s = 1.0 / math.sqrt(dk)
    q = _bf16(_normal(seed, 0, (B, H, T, dk), std=s))
    k = _bf16(_normal(seed, 1, (B, H, T, dk), std=s))
    v = _bf16(_normal(seed, 2, (B, H, T, dv), std=s))
    log_a = (-_softplus(_normal(seed, 3, (B, H, T, dk))) / 16.0).astype(np.float32)
    S0 = _normal(seed, 4, (B, H, dk, dv), std=0.01)
    dO = _bf16(_normal(seed, 5, (B, H, T, dv)))
    return dict(q=q, k=k, v=v, log_a=_f32(log_a), S0=_f32(S0), dO=dO)


def delta_inputs(B=4, H=32, T=4096, dk=128, dv=128, seed=7):
    s = 1.0 / math.sqrt(dk)
    q = _bf16(_normal(seed, 0, (B, H, T, dk), std=s))
    kr = _normal(seed, 1, (B, H, T, dk)).astype(np.float64)
    k = _bf16((kr / np.linalg.norm(kr, axis=-1, keepdims=True)).astype(np.float32))
    v = _bf16(_normal(seed, 2, (B, H, T, dv), std=s))
    log_a = (-_softplus(_normal(seed, 3, (B, H, T))) / 16.0).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-_normal(seed, 4, (B, H, T)).astype(np.float64)))).astype(np.float32)
    S0 = _normal(seed, 5, (B, H, dk, dv), std=0.01)
    dO = _bf16(_normal(seed, 6, (B, H, T, dv)))
    return dict(q=q, k=k, v=v, log_a=_f32(log_a), beta=_f32(beta), S0=_f32(S0), dO=dO)


GENERATORS = {
    "scan_small": scan_small_inputs,
    "scan": scan_inputs,
    "selective": selective_inputs,
    "la_const": la_const_inputs,
    "la_long": la_long_inputs,
    "gla": gla_inputs,
    "delta": delta_inputs,
}


def make(name: str, **shape_overrides):
    """Inputs of workload ``name``; keyword overrides shrink the shape."""
    spec = WORKLOADS[name]
    gen = GENERATORS[name]
    import inspect

    params = inspect.signature(gen).parameters
    kw = {k: spec[k] for k in params if k in spec}
    kw.update(shape_overrides)
    return gen(**kw)


# ---------------------------------------------------------------- device-side draws for very large shapes
# The same distributions drawn on a CUDA device with torch's Philox generator (seeded), for
# shapes beyond what the host draws in reasonable time (the maximum-size tests: more than
# 2^31 elements per tensor).  The oracle then reads back the slices it checks.
def _dev_gen(seed: int, offset: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(offset))
    return g


def _dev_normal(seed, offset, shape, device, std=1.0, dtype=torch.float32) -> torch.Tensor:
    z = torch.empty(shape, dtype=torch.float32, device=device)
    z.normal_(0.0, float(std), generator=_dev_gen(seed, offset, device))
    return z if dtype == torch.float32 else z.to(dtype)


def scan_inputs_device(B, T, D, seed, device):
    """The ``scan`` recipe drawn on the device: a = exp(-0.05 softplus(z)), b, h0, dh ~ N(0, 1)."""
    z = _dev_normal(seed, 0, (B, T, D), device)
    a = torch.exp(-0.05 * torch.nn.functional.softplus(z))
    del z
    return dict(a=a, b=_dev_normal(seed, 1, (B, T, D), device), h0=_dev_normal(seed, 2, (B, D), device),
                dh=_dev_normal(seed, 3, (B, T, D), device))


def la_long_inputs_device(B, H, T, dk, dv, seed, device):
    """The ``la_long`` recipe drawn on the device (S0 = 0)."""
    s = 1.0 / math.sqrt(dk)
    bf = torch.bfloat16
    log_a = -torch.nn.functional.softplus(_dev_normal(seed, 3, (B, H, T), device)) / 16.0
    return dict(q=_dev_normal(seed, 0, (B, H, T, dk), device, s, bf), k=_dev_normal(seed, 1, (B, H, T, dk), device, s, bf),
                v=_dev_normal(seed, 2, (B, H, T, dv), device, s, bf), log_a=log_a, S0=None,
                dO=_dev_normal(seed, 5, (B, H, T, dv), device, 1.0, bf))


def gla_inputs_device(B, H, T, dk, dv, seed, device):
    """The ``gla`` recipe drawn on the device (S0 = 0)."""
    s = 1.0 / math.sqrt(dk)
    bf = torch.bfloat16
    log_a = -torch.nn.functional.softplus(_dev_normal(seed, 3, (B, H, T, dk), device)) / 16.0
    return dict(q=_dev_normal(seed, 0, (B, H, T, dk), device, s, bf), k=_dev_normal(seed, 1, (B, H, T, dk), device, s, bf),
                v=_dev_normal(seed, 2, (B, H, T, dv), device, s, bf), log_a=log_a, S0=None,
                dO=_dev_normal(seed, 5, (B, H, T, dv), device, 1.0, bf))


def delta_inputs_device(B, H, T, dk, dv, seed, device):
    """The ``delta`` recipe drawn on the device (S0 = 0): unit-norm keys, beta = sigmoid(N(0, 1))."""
    s = 1.0 / math.sqrt(dk)
    bf = torch.bfloat16
    kr = _dev_normal(seed, 1, (B, H, T, dk), device)
    k = (kr / torch.linalg.vector_norm(kr, dim=-1, keepdim=True)).to(bf)
    del kr
    log_a = -torch.nn.functional.softplus(_dev_normal(seed, 3, (B, H, T), device)) / 16.0
    beta = torch.sigmoid(_dev_normal(seed, 4, (B, H, T), device))
    return dict(q=_dev_normal(seed, 0, (B, H, T, dk), device, s, bf), k=k,
                v=_dev_normal(seed, 2, (B, H, T, dv), device, s, bf), log_a=log_a, beta=beta, S0=None,
                dO=_dev_normal(seed, 6, (B, H, T, dv), device, 1.0, bf))


def selective_inputs_device(B, T, D, N, seed, device):
    """The ``selective`` recipe drawn on the device."""
    bf = torch.bfloat16
    delta = torch.nn.functional.softplus(_dev_normal(seed, 3, (B, T, D), device, 0.5) - 2.0)
    A = -torch.arange(1, N + 1, dtype=torch.float32, device=device).expand(D, N).contiguous()
    return dict(x=_dev_normal(seed, 0, (B, T, D), device, 1.0, bf), delta=delta, A=A,
                Bm=_dev_normal(seed, 1, (B, T, N), device, 1.0, bf), Cm=_dev_normal(seed, 2, (B, T, N), device, 1.0, bf),
                h0=None, dy=_dev_normal(seed, 4, (B, T, D), device))
