"""Maximum sizes: tensors of more than 2^31 elements (64-bit index arithmetic in every
kernel, look-back unit and tensor-map coordinate), checked against the oracle on slices.

Inputs are drawn on the device (same distributions as the workloads, seeded) since the
host would take minutes; the oracle reads the slices it checks back from the device."""
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


def test_scan_diag_beyond_int32_elements(cla):
    """B=1, T = 2^21 + 71 (a ragged last chunk), D = 1024: 2^31 + 72704 elements per tensor.
    Channels are independent, so three whole channels (every step) are checked."""
    dev = torch.device("cuda")
    B, T, D = 1, (1 << 21) + 71, 1024
    inp = workloads.scan_inputs_device(B, T, D, seed=21, device=dev)
    a, b, h0, dh = inp["a"], inp["b"], inp["h0"], inp["dh"]
    h, hT = cla.scan_diag_fwd(a, b, h0)
    da, db, dh0 = cla.scan_diag_bwd(a, None, h0, h, dh)
    torch.cuda.synchronize()
    ch = [0, 517, 1023]
    sub = lambda x: x[..., ch].contiguous().cpu()
    ra, rb, rh0, rdh = sub(a), sub(b), sub(h0), sub(dh)
    rh, rhT = oracle.scan_diag_fwd(ra, rb, rh0)
    rda, rdb, rdh0 = oracle.scan_diag_bwd(ra, rb, rh0, rdh)
    assert_fp32("h", sub(h), rh)
    assert_fp32("hT", sub(hT), rhT)
    assert_fp32("da", sub(da), rda)
    assert_fp32("db", sub(db), rdb)
    assert_fp32("dh0", sub(dh0), rdh0)


def test_chunk_la_beyond_int32_elements(cla):
    """B=1, H=16, T = 2^20 + 100, d = 128, chunk 128: 2^31 + 204800 elements per q/k/v/dO
    tensor (and twice that many bytes in o, dq, dk, dv).  A reset (a = 0) 2500 tokens before
    the end makes everything after it independent of the earlier tokens, so the oracle runs
    on that tail alone: the tokens with the highest indices, of the first and last head,
    forward and backward (the forward saving its checkpoint, the backward using it)."""
    dev = torch.device("cuda")
    B, H, T, d, chunk = 1, 16, (1 << 20) + 100, 128, 128
    inp = workloads.la_long_inputs_device(B, H, T, d, d, seed=22, device=dev)
    t_r = T - 2500
    inp["log_a"][:, :, t_r] = -float("inf")
    t = inp
    cp = cla.chunk_la_ckpt(t["q"], t["v"], chunk=chunk)
    o, ST = cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], None, chunk=chunk, ckpt=cp)
    dq, dk, dv, dl, dS0 = cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], None, t["dO"], chunk=chunk, ckpt=cp)
    torch.cuda.synchronize()
    for hd in (0, H - 1):
        tail = lambda x: x[:, hd:hd + 1, t_r:].contiguous().cpu()
        q, k, v, la, dO = (tail(t[n]) for n in ("q", "k", "v", "log_a", "dO"))
        ro, rST = oracle.la_fwd(q, k, v, la, None)
        assert_bf16(f"o[head {hd}]", tail(o), ro)
        assert_bf16(f"S_T[head {hd}]", ST[:, hd:hd + 1].cpu(), rST)
        rdq, rdk, rdv, rdl, _ = oracle.la_bwd(q, k, v, la, None, dO)
        for name, x, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
            assert_bf16(f"{name}[head {hd}]", tail(x), r)
        # the decay gradient from the token after the reset on (at the reset it is 0 by
        # definition, a sum of terms that cancel in the closed form)
        assert_bf16(f"dlog_a[head {hd}]", tail(dl)[..., 1:], rdl[..., 1:])


# Gated linear attention and the delta rule take no zero gates, so a tail independent of the earlier
# tokens is made by strong decay instead of a reset: log a = -2 for the tail's first 192 tokens
# scales whatever the state held before the tail by at most e^-384 (0 in fp32, far below the
# tolerance in fp64), so from token 192 of the tail on the outputs, and everywhere in the tail the
# gradients that look only forward in time, equal the oracle's on the tail from a zero state.
_TAIL, _WARM = 2500, 192


def _tail_check(inp, heads, fwd_out, bwd_out, oracle_fwd, oracle_bwd, names_bwd, t_r, extra=(), look_back=()):
    for hd in heads:
        tail = lambda x: x[:, hd:hd + 1, t_r:].contiguous().cpu()
        args = [tail(inp[n]) for n in ("q", "k", "v", "log_a") + extra]
        dO = tail(inp["dO"])
        ro, _ = oracle_fwd(*args, None)
        assert_bf16(f"o[head {hd}]", tail(fwd_out)[:, :, _WARM:], ro[:, :, _WARM:])
        ref = oracle_bwd(*args, None, dO)
        for name, x, r in zip(names_bwd, bwd_out, ref):
            # the gradients that read the state entering a step (look back): from token _WARM on
            lo = _WARM if name in look_back else 0
            assert_bf16(f"{name}[head {hd}]", tail(x)[:, :, lo:], r[:, :, lo:])


def test_gla_beyond_int32_elements(cla):
    """B=1, H=64, T = 262,200, d = 128: 2^31 + 6.6 M elements per q/k/dq/dk/log-decay tensor;
    forward saving its checkpoint and the backward from it, checked on the tail of the first and
    last head (the highest element indices)."""
    dev = torch.device("cuda")
    B, H, T, d = 1, 64, 262200, 128
    assert B * H * T * d > (1 << 31)
    t = workloads.gla_inputs_device(B, H, T, d, d, seed=24, device=dev)
    t_r = T - _TAIL
    t["log_a"][:, :, t_r:t_r + _WARM] = -2.0
    ck = cla.gla_ckpt(t["q"], t["v"])
    o, ST = cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], None, ckpt=ck)
    g = cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], None, t["dO"], ckpt=ck)
    torch.cuda.synchronize()
    _tail_check(t, (0, H - 1), o, g[:4], oracle.gla_fwd, oracle.gla_bwd, ("dq", "dk", "dv", "dlog_a"), t_r,
                look_back=("dq", "dlog_a"))


def test_delta_beyond_int32_elements(cla):
    """B=1, H=64, T = 262,200, d = 128: 2^31 + 6.6 M elements per q/k/v/dO tensor; forward
    saving its checkpoint and the backward from it, checked on the tail of the first and last
    head."""
    dev = torch.device("cuda")
    B, H, T, d = 1, 64, 262200, 128
    assert B * H * T * d > (1 << 31)
    t = workloads.delta_inputs_device(B, H, T, d, d, seed=25, device=dev)
    t_r = T - _TAIL
    t["log_a"][:, :, t_r:t_r + _WARM] = -2.0
    ck = cla.delta_ckpt(t["q"], t["v"])
    o, ST = cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], None, ckpt=ck)
    g = cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], None, t["dO"], ckpt=ck)
    torch.cuda.synchronize()
    # the key, its gate strength and the decay enter the transition applied to the incoming state
    _tail_check(t, (0, H - 1), o, g[:5], oracle.delta_fwd, oracle.delta_bwd, ("dq", "dk", "dv", "dlog_a", "dbeta"),
                t_r, extra=("beta",), look_back=("dq", "dk", "dlog_a", "dbeta"))


# B = 1: the chunk look-back forward; B = 3 (6144 channels): the forward walking each
# channel's whole sequence once
@pytest.mark.parametrize("B,T", [(1, (1 << 20) + 37), (3, 350021)])
def test_selective_beyond_int32_elements(cla, B, T):
    """D = 2048, N = 16: B T D above 2^31 (t, d) elements (and 16 times as many state
    entries).  Channels are independent in y, dx, dDelta and dA, so three whole channels
    are checked; dB and dC sum over every channel and are left to the full-workload test."""
    dev = torch.device("cuda")
    D, N = 2048, 16
    assert B * T * D > (1 << 31)
    t = workloads.selective_inputs_device(B, T, D, N, seed=23, device=dev)
    y, hT, ck = cla.selective_scan_fwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], None)
    dx, dd, dA, dB, dC, dh0 = cla.selective_scan_bwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], None, ck, t["dy"])
    torch.cuda.synchronize()
    ch = [0, 1029, 2047]
    sub = lambda x: x[..., ch].contiguous().cpu()
    x, delta, dy = sub(t["x"]), sub(t["delta"]), sub(t["dy"])
    A = t["A"][ch].cpu()
    Bm, Cm = t["Bm"].cpu(), t["Cm"].cpu()
    ry, rhT = oracle.selective_fwd(x, delta, A, Bm, Cm, None)
    assert_fp32("y", sub(y), ry)
    assert_fp32("hT", hT[:, ch].cpu(), rhT)
    rdx, rdd, rdA, _, _, _ = oracle.selective_bwd(x, delta, A, Bm, Cm, None, dy)
    assert_fp32("dx", sub(dx), rdx)
    assert_fp32("ddelta", sub(dd), rdd)
    assert_fp32("dA", dA[ch].cpu(), rdA)
