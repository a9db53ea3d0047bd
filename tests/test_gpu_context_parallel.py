"""Context parallelism by state passing on one GPU: the library's state-passing
kernels (cla_decay_total, cla_state_compose) against the oracle, and the
context-parallel schedule stepped through for P = 2 to 4 slices of one
sequence in one process (each slice's local pair, the exchange as a stack of
the pairs, the composition, the rerun; the adjoint from the right) with the
library's chunkwise kernels, against the oracle on the whole sequence.  No
kernel waits on another: the slices run one after the other."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_bf16, assert_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import chunkwise_linear_attention_gb300 as m

    m.lib()
    return m


@pytest.mark.parametrize("shape", [(2, 3, 1000), (1, 4, 77, 64), (3, 2, 0), (1, 1, 5000, 128)])
def test_decay_total_kernel(cla, shape):
    rng = np.random.default_rng(len(shape) + shape[2])
    ld = torch.from_numpy((-rng.uniform(0, 0.02, shape)).astype(np.float32))
    got = cla.decay_total(ld.cuda())
    torch.cuda.synchronize()
    B, H, T = shape[:3]
    A = 1 if len(shape) == 3 else shape[3]
    ref = oracle.decay_total(ld.reshape(B * H, T, A)).reshape(got.shape)
    assert_fp32("alpha", got, ref)


@pytest.mark.parametrize("A", [1, 64])
@pytest.mark.parametrize("first,count,step", [(0, 0, 1), (0, 3, 1), (1, 2, 1), (4, 5, -1), (3, 2, -1)])
def test_state_compose_kernel(cla, A, first, count, step):
    rng = np.random.default_rng(first * 10 + count + A)
    P, B, H, dk, dv = 5, 2, 3, 64, 128
    alphas = rng.uniform(0.2, 1.0, (P, B, H) if A == 1 else (P, B, H, A)).astype(np.float32)
    dSs = rng.normal(size=(P, B, H, dk, dv)).astype(np.float32)
    edge = rng.normal(size=(B, H, dk, dv)).astype(np.float32)
    got = cla.state_compose(torch.from_numpy(alphas).cuda(), torch.from_numpy(dSs).cuda(),
                            torch.from_numpy(edge).cuda(), first, count, step)
    torch.cuda.synchronize()
    ref = oracle.state_compose(alphas.reshape(P, B * H, A), dSs.reshape(P, B * H, dk * dv),
                               edge.reshape(B * H, dk * dv), first, count, step).reshape(B, H, dk, dv)
    assert_fp32("state", got, ref)


def _schedule(cla, kind, inp, bounds, chunk):
    """The schedule of context_parallel.forward / backward, stepped through for every slice."""
    from chunkwise_linear_attention_gb300 import context_parallel as cp

    ops = cp.cuda_ops(kind, chunk)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    P = len(bounds) - 1
    sl = [{k: d[k][:, :, lo:hi].contiguous() for k in ("q", "k", "v", "log_a", "dO")}
          for lo, hi in zip(bounds[:-1], bounds[1:])]
    pairs = [cp.local_pair_fwd(ops, s["q"], s["k"], s["v"], s["log_a"]) for s in sl]
    alphas = torch.stack([a for a, _ in pairs])
    dSs = torch.stack([x for _, x in pairs])
    S_in = [cp.incoming_state(ops, alphas, dSs, p, d["S0"]) for p in range(P)]
    outs = [ops.fwd(s["q"], s["k"], s["v"], s["log_a"], S_in[p]) for p, s in enumerate(sl)]
    dDs = torch.stack([cp.local_pair_bwd(ops, s["q"], s["k"], s["v"], s["log_a"], S_in[p], s["dO"])
                       for p, s in enumerate(sl)])
    dST = d.get("dST")
    grads = [ops.bwd(s["q"], s["k"], s["v"], s["log_a"], S_in[p], s["dO"],
                     cp.upstream_state(ops, alphas, dDs, p, P, dST)) for p, s in enumerate(sl)]
    torch.cuda.synchronize()
    o = torch.cat([x[0] for x in outs], dim=2)
    g = [torch.cat([x[i] for x in grads], dim=2) for i in range(4)]
    return o, outs[-1][1], g, grads[0][4]


@pytest.mark.parametrize("kind,bounds,chunk", [
    ("la", (0, 700, 1500), 64), ("la", (0, 64, 65, 900, 2000), 128), ("gla", (0, 333, 1000), 64),
    ("gla", (0, 500, 501, 1200), 64),
])
def test_context_parallel_schedule_matches_whole_sequence(cla, kind, bounds, chunk):
    T = bounds[-1]
    inp = workloads.make("la_long" if kind == "la" else "gla", B=1, H=2, T=T, dk=64, dv=64)
    inp["dST"] = torch.from_numpy(np.random.default_rng(3).normal(0, 0.1, (1, 2, 64, 64)).astype(np.float32))
    o, ST, g, dS0 = _schedule(cla, kind, inp, bounds, chunk)
    fwd = oracle.la_fwd if kind == "la" else oracle.gla_fwd
    bwd = oracle.la_bwd if kind == "la" else oracle.gla_bwd
    ro, rST = fwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"])
    rg = bwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"], inp["dO"], inp["dST"])
    assert_bf16("o", o, ro)
    assert_bf16("S_T", ST, rST)
    for name, x, r in zip(("dq", "dk", "dv", "dlog_a"), g, rg[:4]):
        assert_bf16(name, x, r)
    assert_bf16("dS0", dS0, rg[4])
