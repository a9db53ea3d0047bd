"""Delta rule with a decay per head (Gated DeltaNet), forward and backward:
GPU (through the C ABI) vs the oracle's per-token recurrence and its adjoint,
with the bf16 tolerance (per output tensor, |x - r| / rms(r): max <= 2e-2,
mean <= 5e-3), and the range check on non-finite decays."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import chunkwise_linear_attention_gb300 as m

    m.lib()
    return m


def _run(cla, inp, heads=None):
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    B, H, T, dk = t["q"].shape
    ws = torch.empty(max(cla.delta_workspace_size(B, H, T, dk, t["v"].shape[-1], 64), 256), dtype=torch.uint8,
                     device="cuda")
    o, ST = cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], workspace=ws)
    cla.check_status(ws)
    sel = (lambda x: x) if heads is None else (lambda x: None if x is None else x[:, heads])
    ci = {k: sel(v) for k, v in inp.items()}
    ro, rST = oracle.delta_fwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["beta"], ci["S0"])
    assert_bf16("o", sel(o), ro)
    assert_bf16("S_T", sel(ST), rST)


@pytest.mark.parametrize("B,H,T,dk,dv", [
    (1, 2, 64, 64, 64), (1, 2, 300, 64, 64), (2, 1, 1, 64, 64), (1, 1, 1000, 128, 128),
    (1, 2, 700, 128, 64), (1, 1, 129, 64, 192), (2, 2, 1500, 128, 128),
])
@pytest.mark.parametrize("with_state", [False, True])
def test_delta_small(cla, B, H, T, dk, dv, with_state):
    inp = workloads.make("delta", B=B, H=H, T=T, dk=dk, dv=dv)
    if not with_state:
        inp["S0"] = None
    _run(cla, inp)


def test_delta_full_writes_and_strong_decay(cla):
    """beta = 1 (every write overwrites what its key stored) in one head, strong decays
    (e^-3 per token) in the other."""
    inp = workloads.make("delta", B=1, H=2, T=900, dk=64, dv=64)
    inp["beta"][:, 0] = 1.0
    inp["log_a"][:, 1] = -3.0
    _run(cla, inp)


# a header-only workspace: (I + A)^-1 formed inside the chunk loop; the size query's: formed
# for all chunks beforehand
@pytest.mark.parametrize("full_ws", [False, True])
def test_delta_nonfinite_decay_is_reported(cla, full_ws):
    inp = workloads.make("delta", B=1, H=1, T=200, dk=64, dv=64)
    inp["log_a"][0, 0, 77] = -float("inf")
    t = {k: v.cuda() for k, v in inp.items()}
    n = cla.delta_workspace_size(1, 1, 200, 64, 64, 64) if full_ws else 256
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], workspace=ws)
    with pytest.raises(cla.ClaError, match="outside the kernel's range") as ei:
        cla.check_status(ws)
    assert ei.value.status == 2


@pytest.mark.parametrize("dk,dv,T", [(64, 64, 300), (128, 192, 1000)])
def test_delta_precomputed_inverse_matches_in_loop(cla, dk, dv, T):
    """The chunks' (I + A)^-1 formed beforehand (the size query's workspace) and inside the chunk
    loop (a header-only workspace) are the same computation: bit-identical outputs."""
    inp = workloads.make("delta", B=2, H=2, T=T, dk=dk, dv=dv)
    t = {k: v.cuda() for k, v in inp.items()}
    outs = []
    for n in (256, cla.delta_workspace_size(2, 2, T, dk, dv, 64)):
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        outs.append(cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], workspace=ws))
        cla.check_status(ws)
    assert n > 256
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_delta_workload_full_sampled_heads(cla):
    """The full delta workload (4 x 32 x 4096, d = 128), every output of three heads."""
    inp = workloads.make("delta")
    _run(cla, inp, heads=[0, 17, 31])


# ---------------------------------------------------------------- backward
def _run_bwd(cla, inp, heads=None, dST=None):
    """The backward through the C ABI against the oracle's adjoint: dq, dk, dv, dlog_a, dbeta, dS0."""
    t = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    B, H, T, dk = t["q"].shape
    dv = t["v"].shape[-1]
    ws = torch.empty(max(cla.delta_bwd_workspace_size(B, H, T, dk, dv, 64), 256), dtype=torch.uint8, device="cuda")
    got = cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], t["dO"],
                        None if dST is None else dST.cuda(), workspace=ws)
    cla.check_status(ws)
    sel = (lambda x: x) if heads is None else (lambda x: None if x is None else x[:, heads])
    ci = {k: sel(v) for k, v in inp.items()}
    ref = oracle.delta_bwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["beta"], ci["S0"], ci["dO"], sel(dST))
    for name, g, r in zip(("dq", "dk", "dv", "dlog_a", "dbeta", "dS0"), got, ref):
        assert_bf16(name, sel(g), r)


@pytest.mark.parametrize("B,H,T,dk,dv", [
    (1, 2, 64, 64, 64), (1, 2, 300, 64, 64), (2, 1, 1, 64, 64), (1, 1, 1000, 128, 128),
    (1, 2, 700, 128, 64), (1, 1, 129, 64, 192), (2, 2, 1100, 128, 128),
])
@pytest.mark.parametrize("with_state", [False, True])
def test_delta_bwd_small(cla, B, H, T, dk, dv, with_state):
    """Ragged last chunks, one-token sequences, d_k != d_v and three value-column blocks; with
    S0 and an upstream gradient on S_T, or neither."""
    inp = workloads.make("delta", B=B, H=H, T=T, dk=dk, dv=dv)
    dST = None
    if with_state:
        dST = torch.from_numpy(np.random.default_rng(T).normal(size=(B, H, dk, dv)).astype(np.float32))
    else:
        inp["S0"] = None
    _run_bwd(cla, inp, dST=dST)


def test_delta_bwd_full_writes_and_strong_decay(cla):
    """beta = 1 in one head, e^-3 per token in the other."""
    inp = workloads.make("delta", B=1, H=2, T=900, dk=64, dv=64)
    inp["beta"][:, 0] = 1.0
    inp["log_a"][:, 1] = -3.0
    _run_bwd(cla, inp)


def test_delta_bwd_zero_length_passes_the_state_gradient(cla):
    inp = workloads.make("delta", B=1, H=2, T=0, dk=64, dv=128)
    dST = torch.randn(1, 2, 64, 128)
    t = {k: v.cuda() for k, v in inp.items()}
    g = cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], t["dO"], dST.cuda())
    assert torch.equal(g[5].cpu(), dST)


def test_delta_bwd_workload_full_sampled_heads(cla):
    """The full delta workload (4 x 32 x 4096, d = 128), every gradient of two heads."""
    inp = workloads.make("delta")
    _run_bwd(cla, inp, heads=[5, 26])


@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 2, 700, 128, 64), (1, 1, 129, 64, 192), (2, 2, 1100, 128, 128)])
def test_delta_checkpoint_gives_the_same_gradients(cla, B, H, T, dk, dv):
    """A forward that saves the state entering every chunk, then the backward from it (no states
    pass): the same output and, bit for bit, the same gradients as the plain calls, which match
    the oracle; the backward's workspace then needs no room for the states."""
    inp = workloads.make("delta", B=B, H=H, T=T, dk=dk, dv=dv)
    t = {k: v.cuda() for k, v in inp.items()}
    dST = torch.from_numpy(np.random.default_rng(5).normal(size=(B, H, dk, dv)).astype(np.float32)).cuda()
    ck = cla.delta_ckpt(t["q"], t["v"])
    o1, ST1 = cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"])
    o2, ST2 = cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], ckpt=ck)
    assert torch.equal(o1, o2) and torch.equal(ST1, ST2)
    g1 = cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], t["dO"], dST)
    full = cla.delta_bwd_workspace_size(B, H, T, dk, dv, 64)
    small = full - cla.delta_ckpt_size(B, H, T, dk, dv, 64)
    ws = torch.empty(max(small, 256) + 16, dtype=torch.uint8, device="cuda")
    g2 = cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], t["dO"], dST, ckpt=ck,
                       workspace=ws[: max(small, 256)])
    cla.check_status(ws)
    for name, a, b in zip(("dq", "dk", "dv", "dlog_a", "dbeta", "dS0"), g1, g2):
        assert torch.equal(a, b), name
    ref = oracle.delta_bwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["beta"], inp["S0"], inp["dO"], dST.cpu())
    for name, g, r in zip(("dq", "dk", "dv", "dlog_a", "dbeta", "dS0"), g2, ref):
        assert_bf16(name, g, r)
