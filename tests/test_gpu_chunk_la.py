"""Chunkwise decayed linear attention, forward and backward: GPU (through the
C ABI) vs the oracle's per-token recurrence, with the bf16 tolerance
(per output tensor, |x - r| / rms(r): max <= 2e-2, mean <= 5e-3)."""
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


def _check(cla, inp, chunk, dST=None, heads=None, check_bwd=True, ckpt=False):
    """ckpt: the forward saves its segment states and the backward starts from them (the
    training-step path the benchmark times)."""
    t = {k: _dev(v) for k, v in inp.items()}
    cp = cla.chunk_la_ckpt(t["q"], t["v"], chunk=chunk) if ckpt else None
    o, ST = cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=chunk, ckpt=cp)
    if check_bwd:
        g = cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], _dev(dST), chunk=chunk,
                             ckpt=cp)
    torch.cuda.synchronize()
    sel = (lambda x: x) if heads is None else (lambda x: None if x is None else x[:, heads])
    ci = {k: sel(v) for k, v in inp.items()}
    ro, rST = oracle.la_fwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["S0"])
    assert_bf16("o", sel(o), ro)
    assert_bf16("S_T", sel(ST), rST)
    if not check_bwd:
        return
    rdq, rdk, rdv, rdl, rdS0 = oracle.la_bwd(ci["q"], ci["k"], ci["v"], ci["log_a"], ci["S0"], ci["dO"], sel(dST))
    for name, x, r in zip(("dq", "dk", "dv", "dlog_a", "dS0"), map(sel, g), (rdq, rdk, rdv, rdl, rdS0)):
        assert_bf16(name, x, r)


@pytest.mark.parametrize("B,H,T,d,chunk", [
    (1, 2, 64, 64, 64), (1, 2, 300, 64, 64), (2, 1, 1, 64, 64), (1, 1, 1000, 64, 64),
    (1, 1, 3000, 64, 64), (1, 2, 700, 64, 128), (1, 1, 2000, 128, 128), (1, 1, 500, 128, 64),
    (2, 1, 129, 128, 128),
])
@pytest.mark.parametrize("with_state", [False, True])
def test_chunk_la_small(cla, B, H, T, d, chunk, with_state):
    inp = workloads.make("la_long", B=B, H=H, T=T, dk=d, dv=d)
    dST = None
    if not with_state:
        inp["S0"] = None
    else:
        rng = np.random.default_rng(T + d)
        dST = torch.from_numpy(rng.normal(0, 0.1, (B, H, d, d)).astype(np.float32))
    _check(cla, inp, chunk, dST)


def test_chunk_la_constant_decay_small(cla):
    inp = workloads.make("la_const", B=1, H=16, T=777, dk=64, dv=64)
    _check(cla, inp, 64)


def test_chunk_la_resets(cla):
    """log a = -inf (a reset) inside and at the start of chunks: products that
    span it are 0, never NaN."""
    inp = workloads.make("la_long", B=1, H=2, T=400, dk=64, dv=64)
    la = inp["log_a"].clone()
    for t in (0, 5, 64, 100, 255, 399):
        la[0, 0, t] = -float("inf")
    la[0, 1, 130] = -float("inf")
    inp["log_a"] = la
    t = {k: _dev(v) for k, v in inp.items()}
    o, ST = cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=64)
    dq, dk, dv, dl, dS0 = cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], chunk=64)
    torch.cuda.synchronize()
    ro, rST = oracle.la_fwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"])
    assert_bf16("o", o, ro)
    assert_bf16("S_T", ST, rST)
    rdq, rdk, rdv, rdl, rdS0 = oracle.la_bwd(inp["q"], inp["k"], inp["v"], inp["log_a"], inp["S0"], inp["dO"])
    for name, x, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv), ("dS0", dS0, rdS0)):
        assert_bf16(name, x, r)
    # dlog_a at a reset: the definition gives a_t <.,.> = 0 there
    dl = dl.cpu().numpy()
    assert np.all(np.isfinite(dl))
    assert_bf16("dlog_a", dl, rdl)


def test_chunk_la_empty(cla):
    dev = torch.device("cuda")
    z = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device=dev)
    S0 = torch.randn(1, 2, 64, 64, device=dev)
    o, ST = cla.chunk_la_fwd(z, z, z, torch.empty(1, 2, 0, device=dev), S0)
    torch.cuda.synchronize()
    assert torch.equal(ST, S0)


def test_chunk_la_constant_decay_workload_full(cla):
    """4 x 16 x 8192, d = 64, chunk 64, every output element (forward saving its
    segment states, backward starting from them, as the benchmark runs it)."""
    inp = workloads.make("la_const")
    _check(cla, inp, 64, ckpt=True)


def test_chunk_la_long_workload_sampled_heads(cla):
    """1 x 32 x 65536, d = 128, chunk 128 on the GPU; heads 0, 31 and two seeded
    middle heads against the oracle (heads are independent problems); the
    benchmark's path, with the forward's segment states."""
    inp = workloads.make("la_long")
    # the first and last heads and two seeded middle ones
    mid = sorted(np.random.default_rng(128).choice(np.arange(1, 31), 2, replace=False).tolist())
    _check(cla, inp, 128, heads=[0] + mid + [31], ckpt=True)


@pytest.mark.parametrize("B,H,T,d,chunk", [
    (1, 2, 40, 64, 64), (1, 1, 3000, 64, 64), (1, 2, 700, 64, 128), (1, 1, 2000, 128, 128),
    (1, 1, 500, 128, 64), (2, 1, 129, 128, 128),
])
def test_chunk_la_ckpt(cla, B, H, T, d, chunk):
    """The backward started from the forward's saved segment states: against the
    oracle, and against the backward that rebuilds the states (equal up to fp32
    rounding: the two build the same states with the operands' roles swapped).
    T = 40 is shorter than a chunk: nothing is saved and the backward rebuilds."""
    inp = workloads.make("la_long", B=B, H=H, T=T, dk=d, dv=d)
    rng = np.random.default_rng(T * 7 + d)
    dST = torch.from_numpy(rng.normal(0, 0.1, (B, H, d, d)).astype(np.float32))
    _check(cla, inp, chunk, dST, ckpt=True)
    t = {k: _dev(v) for k, v in inp.items()}
    cp = cla.chunk_la_ckpt(t["q"], t["v"], chunk=chunk)
    cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=chunk, ckpt=cp)
    with_ck = cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], _dev(dST), chunk=chunk,
                               ckpt=cp)
    rebuilt = cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], _dev(dST), chunk=chunk)
    torch.cuda.synchronize()
    for name, x, r in zip(("dq", "dk", "dv", "dlog_a", "dS0"), with_ck, rebuilt):
        rms = float(torch.sqrt(torch.mean(r.double() ** 2)))
        err = float(torch.max(torch.abs(x.double() - r.double()))) / max(rms, 1e-30)
        assert err <= 1e-4, f"{name}: checkpointed backward differs from the rebuilding one by {err:.2e} rms"


def test_chunk_la_ckpt_rejects_short_buffer(cla):
    inp = workloads.make("la_long", B=1, H=1, T=300, dk=64, dv=64)
    t = {k: _dev(v) for k, v in inp.items()}
    with pytest.raises(ValueError):
        cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=64,
                         ckpt=torch.empty(4, dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("d,chunk", [(128, 128), (64, 128), (128, 64)])
def test_chunk_la_resets_across_pieces(cla, d, chunk):
    """Resets at and next to the 32-token piece boundaries inside a chunk (the
    off-diagonal pieces' decays are formed as row x column factors, which a
    reset between piece and row must zero), in both traversal directions."""
    inp = workloads.make("la_long", B=1, H=2, T=700, dk=d, dv=d)
    la = inp["log_a"].clone()
    for t in (31, 32, 33, 63, 95, 96, 127, 128, 200, 330, 511, 512, 699):
        la[0, 0, t] = -float("inf")
    for t in (17, 150, 401):
        la[0, 1, t] = -float("inf")
    inp["log_a"] = la
    _check(cla, inp, chunk, dST=torch.from_numpy(np.random.default_rng(5).normal(0, 0.1, (1, 2, d, d)).astype(np.float32)))


@pytest.mark.parametrize("d,chunk", [(128, 128), (64, 64)])
def test_chunk_la_strong_decay(cla, d, chunk):
    """Decays far from 1 (log a in [-8, -2]): products over a chunk underflow to
    0 in fp32; every term must stay finite and match the recurrence."""
    inp = workloads.make("la_long", B=1, H=2, T=600, dk=d, dv=d)
    rng = np.random.default_rng(11)
    inp["log_a"] = torch.from_numpy(-rng.uniform(2.0, 8.0, (1, 2, 600)).astype(np.float32))
    _check(cla, inp, chunk)


def test_chunk_la_long_workload_chunk64_sampled_heads(cla):
    """1 x 32 x 65536, d = 128, chunk 64 (segments of 64 chunks) on the GPU;
    heads 5 and 20 against the oracle (with the forward's segment states, as
    the benchmark runs it)."""
    inp = workloads.make("la_long")
    _check(cla, inp, 64, heads=[5, 20], ckpt=True)


@pytest.mark.parametrize("dk,dv,chunk", [(64, 128, 128), (128, 64, 64), (128, 64, 128)])
@pytest.mark.parametrize("ckpt", [False, True])
def test_chunk_la_unequal_head_dims(cla, dk, dv, chunk, ckpt):
    """dim_k != dim_v: the forward's state is dim_k x dim_v, the dQ traversal's
    its transpose (dim_v rows), the dK traversal's the adjoint's transpose."""
    inp = workloads.make("la_long", B=1, H=2, T=700, dk=dk, dv=dv)
    rng = np.random.default_rng(dk * 3 + dv)
    dST = torch.from_numpy(rng.normal(0, 0.1, (1, 2, dk, dv)).astype(np.float32))
    _check(cla, inp, chunk, dST, ckpt=ckpt)


@pytest.mark.parametrize("d,chunk", [(64, 64), (128, 128)])
def test_chunk_la_ckpt_holds_segment_states(cla, d, chunk):
    """The checkpoint is the state entering each segment: entry s equals the oracle's state
    after the first s * seg_chunks * chunk tokens (S0 and the decays included).  One head, so
    segments are 8 chunks long (the smallest choice when blocks are few)."""
    T = 3000 if chunk == 64 else 5000
    inp = workloads.make("la_long", B=1, H=1, T=T, dk=d, dv=d)
    t = {k: _dev(v) for k, v in inp.items()}
    cp = cla.chunk_la_ckpt(t["q"], t["v"], chunk=chunk)
    cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=chunk, ckpt=cp)
    torch.cuda.synchronize()
    seg_tokens = 8 * chunk
    n_seg = (T + seg_tokens - 1) // seg_tokens
    assert cp.numel() * 4 == cla.chunk_la_ckpt_size(1, 1, T, d, d, chunk) == n_seg * d * d * 4
    states = cp.view(n_seg, d, d).cpu()
    for s in range(n_seg):
        t0 = s * seg_tokens
        if t0 == 0:
            ref = inp["S0"][0, 0].double().numpy()
        else:
            _, rST = oracle.la_fwd(inp["q"][:, :, :t0], inp["k"][:, :, :t0], inp["v"][:, :, :t0],
                                   inp["log_a"][:, :, :t0], inp["S0"])
            ref = rST[0, 0]
        assert_bf16(f"segment {s} state", states[s].numpy(), ref)
