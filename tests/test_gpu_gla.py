"""Gated linear attention forward and backward (one decay per key dimension):
GPU (through the C ABI) vs the oracle's per-token recurrence and its adjoint,
with the bf16 tolerance (per output tensor, |x - r| / rms(r): max <= 2e-2,
mean <= 5e-3), and the kernels' range check on decays they cannot factor."""
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


def _dev(x):
    return None if x is None else x.cuda()


def _run(cla, inp, heads=None, bwd=False, dST=None):
    t = {k: _dev(v) for k, v in inp.items()}
    ws = torch.empty(max(cla.gla_workspace_size(*t["q"].shape, t["v"].shape[-1], 64), 256), dtype=torch.uint8,
                     device="cuda")
    o, ST = cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], workspace=ws)
    cla.check_status(ws)
    sel = (lambda x: x) if heads is None else (lambda x: None if x is None else x[:, heads])
    ci = {k: sel(v) for k, v in inp.items()}
    ro, rST = oracle.gla_fwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["S0"])
    assert_bf16("o", sel(o), ro)
    assert_bf16("S_T", sel(ST), rST)
    if not bwd:
        return
    wb = torch.empty(max(cla.gla_bwd_workspace_size(*t["q"].shape, t["v"].shape[-1], 64), 256), dtype=torch.uint8,
                     device="cuda")
    g = cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], _dev(dST), workspace=wb)
    cla.check_status(wb)
    ref = oracle.gla_bwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["S0"], ci["dO"], sel(dST))
    for name, x, r in zip(("dq", "dk", "dv", "dlog_a", "dS0"), map(sel, g), ref):
        assert_bf16(name, x, r)


@pytest.mark.parametrize("B,H,T,dk,dv", [
    (1, 2, 64, 64, 64), (1, 2, 300, 64, 64), (2, 1, 1, 64, 64), (1, 1, 1000, 128, 128),
    (1, 2, 700, 128, 64), (1, 1, 129, 64, 192), (2, 2, 2000, 128, 128), (1, 1, 4097, 64, 128),
])
@pytest.mark.parametrize("with_state", [False, True])
def test_gla_small(cla, B, H, T, dk, dv, with_state):
    inp = workloads.make("gla", B=B, H=H, T=T, dk=dk, dv=dv)
    if not with_state:
        inp["S0"] = None
    _run(cla, inp)


def test_gla_strong_decay_within_range(cla):
    """Gates down to e^-2.5 per token in some dimensions (a 32-token product near 2^-115, inside
    the kernel's 2^-120 range), others near 1: the factored scores stay finite and exact."""
    inp = workloads.make("gla", B=1, H=2, T=900, dk=64, dv=64)
    la = inp["log_a"].clone()
    la[:, :, :, ::3] = -2.5
    la[:, :, :, 1::7] = -1e-4
    inp["log_a"] = la
    _run(cla, inp)


def test_gla_decay_out_of_range_is_reported(cla):
    """A zero gate (log a = -inf) or a 32-token product below 2^-120 cannot be factored:
    cla_check_status reports CLA_ERR_UNSUPPORTED instead of returning overflowed results."""
    for bad in (-float("inf"), -6.0):
        inp = workloads.make("gla", B=1, H=1, T=200, dk=64, dv=64)
        la = inp["log_a"].clone()
        la[0, 0, 100:140, 5] = bad
        t = {k: _dev(v) for k, v in inp.items()}
        ws = torch.empty(cla.gla_workspace_size(1, 1, 200, 64, 64, 64), dtype=torch.uint8, device="cuda")
        cla.gla_fwd(t["q"], t["k"], t["v"], la.cuda(), t["S0"], workspace=ws)
        with pytest.raises(cla.ClaError, match="outside the kernel's range") as ei:
            cla.check_status(ws)
        assert ei.value.status == 2
        # the context stays usable: a valid call right after passes
        ws2 = torch.empty(cla.gla_workspace_size(1, 1, 200, 64, 64, 64), dtype=torch.uint8, device="cuda")
        cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], workspace=ws2)
        cla.check_status(ws2)


def test_gla_empty(cla):
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    S0 = torch.randn(1, 2, 64, 64, device="cuda")
    o, ST = cla.gla_fwd(q, q, q, torch.empty(1, 2, 0, 64, device="cuda"), S0)
    torch.cuda.synchronize()
    assert torch.equal(ST, S0)


def test_gla_workload_full_sampled_heads(cla):
    """The full gla workload (2 x 16 x 16384, d = 128), every output of three heads spread over
    the batch (the heads are independent problems)."""
    inp = workloads.make("gla")
    _run(cla, inp, heads=[0, 7, 15])


@pytest.mark.parametrize("B,H,T,dk,dv", [
    (1, 2, 64, 64, 64), (1, 2, 300, 64, 64), (2, 1, 1, 64, 64), (1, 1, 1000, 128, 128),
    (1, 2, 700, 128, 64), (1, 1, 777, 64, 128), (2, 2, 2000, 128, 128),
])
@pytest.mark.parametrize("with_state", [False, True])
def test_gla_bwd_small(cla, B, H, T, dk, dv, with_state):
    inp = workloads.make("gla", B=B, H=H, T=T, dk=dk, dv=dv)
    dST = None
    if not with_state:
        inp["S0"] = None
    else:
        rng = np.random.default_rng(T + dk + dv)
        dST = torch.from_numpy(rng.normal(0, 0.1, (B, H, dk, dv)).astype(np.float32))
    _run(cla, inp, bwd=True, dST=dST)


def test_gla_bwd_strong_decay_within_range(cla):
    """Backward with gates down to e^-2.5 per token in some dimensions (the decay gradient's
    suffix sums then cancel strongly) and near 1 in others."""
    inp = workloads.make("gla", B=1, H=2, T=900, dk=64, dv=64)
    la = inp["log_a"].clone()
    la[:, :, :, ::3] = -2.5
    la[:, :, :, 1::7] = -1e-4
    inp["log_a"] = la
    dST = torch.from_numpy(np.random.default_rng(1).normal(0, 0.1, (1, 2, 64, 64)).astype(np.float32))
    _run(cla, inp, bwd=True, dST=dST)


def test_gla_bwd_unequal_segments_sampled_heads(cla):
    """d_k = 128, d_v = 64 on 32 heads of 16384 tokens: the dV traversal (one column block) and
    the dK traversal (two key blocks) pick different segment lengths, so dK runs its own phase 1
    and look-back instead of starting from dV's segment states; two heads checked."""
    inp = workloads.make("gla", B=2, H=16, T=16384, dk=128, dv=64)
    _run(cla, inp, heads=[0, 13], bwd=True)


def test_gla_bwd_workload_full_sampled_heads(cla):
    """The full gla workload, backward, every output of two heads."""
    inp = workloads.make("gla")
    _run(cla, inp, heads=[3, 12], bwd=True)


# ---------------------------------------------------------------- checkpoint
def _gla_seg_chunks(n_chunks, n_seg):
    """The segment length of a checkpoint with n_seg segments (the largest of 64, 32, 16, 8 that
    gives that count)."""
    for c in (64, 32, 16, 8):
        if -(-n_chunks // c) == n_seg:
            return c
    raise AssertionError((n_chunks, n_seg))


@pytest.mark.parametrize("B,H,T,dk,dv", [(1, 2, 1000, 64, 64), (1, 1, 2500, 128, 64), (2, 2, 3000, 128, 128)])
def test_gla_checkpoint(cla, B, H, T, dk, dv):
    """The forward saving the state entering every segment: the same o and S_T bit for bit; each
    saved state equals the oracle's state after the tokens before its segment; the backward
    from the checkpoint (no state rebuilding in its dq traversal) matches the oracle."""
    inp = workloads.make("gla", B=B, H=H, T=T, dk=dk, dv=dv)
    t = {k: _dev(v) for k, v in inp.items()}
    dST = torch.from_numpy(np.random.default_rng(T).normal(0, 0.1, (B, H, dk, dv)).astype(np.float32))
    ck = cla.gla_ckpt(t["q"], t["v"])
    o1, ST1 = cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"])
    o2, ST2 = cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], ckpt=ck)
    assert torch.equal(o1, o2) and torch.equal(ST1, ST2)
    n_chunks = -(-T // 64)
    n_seg = ck.numel() // (B * H * dk * dv)
    assert n_seg >= 2
    seg_chunks = _gla_seg_chunks(n_chunks, n_seg)
    ckv = ck[: n_seg * B * H * dk * dv].view(n_seg, B, H, dk, dv)
    for sg in (0, 1, n_seg - 1):
        t0 = sg * seg_chunks * 64
        if t0 == 0:
            ref = inp["S0"] if inp["S0"] is not None else torch.zeros(B, H, dk, dv)
        else:
            _, ref = oracle.gla_fwd(inp["q"][:, :, :t0], inp["k"][:, :, :t0], inp["v"][:, :, :t0],
                                    inp["log_a"][:, :, :t0], inp["S0"])
        assert_bf16(f"ckpt[{sg}]", ckv[sg], ref)
    g = cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], dST.cuda(), ckpt=ck)
    ref = oracle.gla_bwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"], inp["dO"], dST)
    for name, x, r in zip(("dq", "dk", "dv", "dlog_a", "dS0"), g, ref):
        assert_bf16(name, x, r)


def test_gla_bwd_decay_gradient_unaligned_output(cla):
    """A dlog_decay buffer only 4-byte aligned takes the scalar decay-gradient kernels (the
    aligned one the 8-dimension ones): both match the oracle and each other."""
    B, H, T, dk, dv = 1, 2, 700, 128, 64
    inp = workloads.make("gla", B=B, H=H, T=T, dk=dk, dv=dv)
    t = {k: _dev(v) for k, v in inp.items()}
    buf = torch.empty(B * H * T * dk + 1, device="cuda")
    odd = buf[1:].view(B, H, T, dk)
    assert odd.data_ptr() % 16 != 0
    g_al = cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"])
    g_un = cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], dlog_decay=odd)
    ref = oracle.gla_bwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"], inp["dO"])
    assert_bf16("dlog_a (8 dimensions a thread)", g_al[3], ref[3])
    assert_bf16("dlog_a (scalar)", g_un[3], ref[3])
    assert_bf16("dlog_a (two paths)", g_un[3], g_al[3], tol_max=1e-5, tol_mean=1e-6)
