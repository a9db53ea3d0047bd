"""The seeded input recipes (``workloads``): deterministic, the stated shapes and dtypes, and
the stated distributions -- checked on cut shapes, on the CPU."""
import math

import numpy as np
import pytest
import torch

import workloads

CUT = {
    "scan_small": dict(T=256, D=16),
    "scan": dict(B=2, T=512, D=64),
    "selective": dict(B=2, T=256, D=64, N=16),
    "la_const": dict(B=2, H=4, T=256),
    "la_long": dict(B=1, H=2, T=512),
    "gla": dict(B=1, H=2, T=256),
    "delta": dict(B=1, H=2, T=256),
}


def _same(x, y):
    if x is None or y is None:
        return x is None and y is None
    return x.dtype == y.dtype and x.shape == y.shape and torch.equal(x, y)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_recipes_are_deterministic(name):
    a, b = workloads.make(name, **CUT[name]), workloads.make(name, **CUT[name])
    assert a.keys() == b.keys()
    for k in a:
        assert _same(a[k], b[k]), (name, k)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_every_cut_is_in_the_workload_table(name):
    """Every override names a size of the workload, and the full table names every generator."""
    spec = workloads.WORKLOADS[name]
    assert set(CUT[name]) <= set(spec)
    assert name in workloads.GENERATORS


def test_scan_recipes():
    s = workloads.make("scan_small", **CUT["scan_small"])
    assert s["a"].dtype == torch.float32 and tuple(s["a"].shape) == (1, 256, 16) and s["h0"] is None
    assert float(s["a"].min()) >= 0.8 and float(s["a"].max()) <= 0.999
    t = workloads.make("scan", **CUT["scan"])
    assert tuple(t["a"].shape) == (2, 512, 64) and tuple(t["h0"].shape) == (2, 64)
    a = t["a"].double()
    # a = exp(-0.05 softplus(z)): in (0, 1), and -20 log(a) = softplus(z) > 0 with mean E softplus(N(0,1))
    assert float(a.max()) < 1.0 and float(a.min()) > 0.0
    sp = -20.0 * torch.log(a)
    assert abs(float(sp.mean()) - 0.8061) < 0.02  # E[softplus(z)], z ~ N(0, 1)
    for k in ("b", "h0", "dh"):
        x = t[k].double()
        assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05, k
    assert not torch.equal(t["b"], t["dh"])  # independent streams


def test_selective_recipe():
    s = workloads.make("selective", **CUT["selective"])
    assert s["x"].dtype == torch.bfloat16 and s["Bm"].dtype == torch.bfloat16 and s["Cm"].dtype == torch.bfloat16
    assert s["delta"].dtype == torch.float32 and tuple(s["delta"].shape) == (2, 256, 64)
    assert tuple(s["Bm"].shape) == (2, 256, 16) and s["h0"] is None
    A = s["A"]
    assert tuple(A.shape) == (64, 16)
    assert torch.equal(A, -torch.arange(1, 17, dtype=torch.float32).expand(64, 16))
    d = s["delta"].double()
    # Delta = softplus(N(-2, 0.5)): positive, median softplus(-2) = 0.1269
    assert float(d.min()) > 0.0 and abs(float(d.median()) - math.log1p(math.exp(-2.0))) < 0.01


def test_la_const_recipe():
    t = workloads.make("la_const", **CUT["la_const"])
    B, H, T = 2, 4, 256
    assert tuple(t["q"].shape) == (B, H, T, 64) and t["q"].dtype == torch.bfloat16 and t["S0"] is None
    lam = 1.0 - 2.0 ** (-(5.0 + 8.0 * np.arange(H) / H))
    la = t["log_a"]
    for h in range(H):
        assert torch.all(la[:, h, :] == la[0, h, 0])  # constant per head
        assert abs(float(la[0, h, 0]) - math.log(lam[h])) < 1e-7
    assert abs(float(t["q"].double().std()) - 1.0 / 8.0) < 0.01


@pytest.mark.parametrize("name", ["la_long", "gla", "delta"])
def test_data_dependent_decay_recipes(name):
    t = workloads.make(name, **CUT[name])
    q, la, S0 = t["q"], t["log_a"].double(), t["S0"]
    dk = q.shape[-1]
    assert q.dtype == torch.bfloat16 and dk == 128
    assert abs(float(q.double().std()) - 1.0 / math.sqrt(dk)) < 0.005
    # log a = -softplus(N(0, 1)) / 16: negative, mean -E[softplus(z)] / 16
    assert float(la.max()) < 0.0 and abs(float(la.mean()) + 0.8061 / 16.0) < 0.005
    assert tuple(la.shape) == (tuple(q.shape) if name == "gla" else tuple(q.shape[:3]))
    assert S0.dtype == torch.float32 and abs(float(S0.double().std()) - 0.01) < 0.001


def test_delta_keys_and_strengths():
    t = workloads.make("delta", **CUT["delta"])
    norms = t["k"].double().norm(dim=-1)
    assert float((norms - 1.0).abs().max()) < 1e-2  # unit rows, then one bf16 rounding
    beta = t["beta"].double()
    assert float(beta.min()) > 0.0 and float(beta.max()) < 1.0
    assert abs(float(beta.mean()) - 0.5) < 0.03  # sigmoid(N(0, 1)) is symmetric about 1/2
