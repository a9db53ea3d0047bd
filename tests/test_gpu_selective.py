"""Selective (Mamba-1 style) scan, forward and backward: GPU (through the C
ABI) vs the float64 oracle, fp32 tolerance (per output tensor,
max |x - r| / max(|r|, rms(r)) <= 1e-5)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import chunkwise_linear_attention_gb300 as m

    m.lib()
    return m


def _run_gpu(cla, inp, h0=None, dhT=None):
    t = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    h0d = h0.cuda() if h0 is not None else None
    y, hT, ck = cla.selective_scan_fwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], h0d)
    g = cla.selective_scan_bwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], h0d, ck, t["dy"],
                               dhT.cuda() if dhT is not None else None)
    torch.cuda.synchronize()
    return y, hT, g


@pytest.mark.parametrize("B,T,D", [(1, 64, 128), (2, 150, 130), (1, 1, 16), (1, 1000, 64), (2, 300, 256),
                                   (1, 129, 7)])
@pytest.mark.parametrize("with_state", [False, True])
def test_selective_small(cla, B, T, D, with_state):
    inp = workloads.make("selective", B=B, T=T, D=D)
    N = inp["A"].shape[1]
    rng = np.random.default_rng(B * T + D)
    h0 = torch.from_numpy(rng.standard_normal((B, D, N)).astype(np.float32)) if with_state else None
    dhT = torch.from_numpy(rng.standard_normal((B, D, N)).astype(np.float32)) if with_state else None
    y, hT, (dx, dd, dA, dB, dC, dh0) = _run_gpu(cla, inp, h0, dhT)
    ry, rhT = oracle.selective_fwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], h0)
    rdx, rdd, rdA, rdB, rdC, rdh0 = oracle.selective_bwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"],
                                                         h0, inp["dy"], dhT)
    for name, x, r in (("y", y, ry), ("hT", hT, rhT), ("dx", dx, rdx), ("ddelta", dd, rdd), ("dA", dA, rdA),
                       ("dB", dB, rdB), ("dC", dC, rdC), ("dh0", dh0, rdh0)):
        assert_fp32(name, x, r)


# B * D >= 16 * (SM count) channels (3 x 2048 on 152 SMs; 1 x 2048 stays below) take
# the forward that walks each channel's whole sequence once instead of the chunk look-back
@pytest.mark.parametrize("T", [1, 64, 150, 333])
@pytest.mark.parametrize("with_state", [False, True])
def test_selective_many_channels(cla, T, with_state):
    B, D = 3, 2048
    inp = workloads.make("selective", B=B, T=T, D=D)
    N = inp["A"].shape[1]
    rng = np.random.default_rng(T + 7)
    h0 = torch.from_numpy(rng.standard_normal((B, D, N)).astype(np.float32)) if with_state else None
    dhT = torch.from_numpy(rng.standard_normal((B, D, N)).astype(np.float32)) if with_state else None
    y, hT, (dx, dd, dA, dB, dC, dh0) = _run_gpu(cla, inp, h0, dhT)
    ry, rhT = oracle.selective_fwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], h0)
    rdx, rdd, rdA, rdB, rdC, rdh0 = oracle.selective_bwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"],
                                                         h0, inp["dy"], dhT)
    for name, x, r in (("y", y, ry), ("hT", hT, rhT), ("dx", dx, rdx), ("ddelta", dd, rdd), ("dA", dA, rdA),
                       ("dB", dB, rdB), ("dC", dC, rdC), ("dh0", dh0, rdh0)):
        assert_fp32(name, x, r)


def test_selective_many_channels_ckpt(cla):
    """The saved states: entry i is the state entering step 16 i (oracle run to that step)."""
    B, T, D = 3, 150, 2048
    inp = workloads.make("selective", B=B, T=T, D=D)
    t = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    _, _, ck = cla.selective_scan_fwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], None)
    torch.cuda.synchronize()
    n_ck = (T + cla.SELECTIVE_CKPT_CHUNK - 1) // cla.SELECTIVE_CKPT_CHUNK
    ck = ck.view(B, n_ck, D, 16)
    assert_fp32("ckpt[0]", ck[:, 0], torch.zeros(B, D, 16))
    for i in (1, 5, n_ck - 1):
        s = i * cla.SELECTIVE_CKPT_CHUNK
        _, rh = oracle.selective_fwd(inp["x"][:, :s], inp["delta"][:, :s], inp["A"], inp["Bm"][:, :s],
                                     inp["Cm"][:, :s])
        assert_fp32(f"ckpt[{i}]", ck[:, i], rh)


def test_selective_general_A(cla):
    """A not of the -(n+1) form (positive and negative rates per channel)."""
    for B, D in ((1, 64), (3, 2048)):  # the chunk look-back and the per-channel walk
        _general_A_case(cla, B, D)


def _general_A_case(cla, B, D):
    inp = workloads.make("selective", B=B, T=200, D=D)
    rng = np.random.default_rng(9)
    inp["A"] = torch.from_numpy(-rng.uniform(0.05, 4.0, (D, 16)).astype(np.float32))
    y, hT, (dx, dd, dA, dB, dC, dh0) = _run_gpu(cla, inp)
    ry, rhT = oracle.selective_fwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"])
    rg = oracle.selective_bwd(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], None, inp["dy"])
    assert_fp32("y", y, ry)
    for name, x, r in zip(("dx", "ddelta", "dA", "dB", "dC"), (dx, dd, dA, dB, dC), rg[:5]):
        assert_fp32(name, x, r)


def test_selective_workload_full(cla):
    """4 x 8192 x 2048 x 16 on the GPU.  Per-channel outputs (y, hT, dx,
    ddelta, dA) are checked on 96 channels (first, last and seeded middle ones)
    over every batch row and step; the channel sums dB, dC on batch row 0 and a
    seeded other row over all channels."""
    inp = workloads.make("selective")
    y, hT, (dx, dd, dA, dB, dC, dh0) = _run_gpu(cla, inp)
    # the first and last 32 channels, and 32 seeded ones from the middle
    mid = np.random.default_rng(2048).choice(np.arange(32, 2016), 32, replace=False)
    chans = list(range(32)) + sorted(mid.tolist()) + list(range(2016, 2048))
    sub = {k: (v[:, :, chans] if k in ("x", "delta", "dy") else v) for k, v in inp.items() if v is not None}
    sub["A"] = inp["A"][chans]
    ry, rhT = oracle.selective_fwd(sub["x"], sub["delta"], sub["A"], sub["Bm"], sub["Cm"])
    rdx, rdd, rdA, _, _, _ = oracle.selective_bwd(sub["x"], sub["delta"], sub["A"], sub["Bm"], sub["Cm"], None,
                                                  sub["dy"])
    assert_fp32("y", y[:, :, chans], ry)
    assert_fp32("hT", hT[:, chans], rhT)
    assert_fp32("dx", dx[:, :, chans], rdx)
    assert_fp32("ddelta", dd[:, :, chans], rdd)
    assert_fp32("dA", dA[chans], rdA)
    # channel sums over all channels: batch row 0 and a seeded middle row
    for row in (0, int(np.random.default_rng(4).integers(1, 4))):
        b0 = {k: (v[row:row + 1] if k not in ("A",) else v) for k, v in inp.items() if v is not None}
        _, _, _, rdB, rdC, _ = oracle.selective_bwd(b0["x"], b0["delta"], b0["A"], b0["Bm"], b0["Cm"], None,
                                                    b0["dy"])
        assert_fp32("dB", dB[row:row + 1], rdB)
        assert_fp32("dC", dC[row:row + 1], rdC)


@pytest.mark.parametrize("B", [1, 3])  # B = 3: the per-channel walk
def test_selective_decay_accuracy(cla, B):
    """One step from h0 = 1 with x = 0 leaves h_T = exp(delta A).  Against the
    float64 value: within 2 ulp plus the rounding of the argument
    delta * A * log2(e) (relative |arg| * 2^-23), and unbiased where the
    decays are near 1 (where long products of them build up)."""
    D, N = 2048, 16
    rng = np.random.default_rng(17)
    delta = rng.uniform(0.0, 3.0, (B, 1, D)).astype(np.float32)
    A = -rng.uniform(0.0, 20.0, (D, N)).astype(np.float32)
    z = torch.zeros(B, 1, D, dtype=torch.bfloat16, device="cuda")
    Bm = torch.zeros(B, 1, N, dtype=torch.bfloat16, device="cuda")
    h0 = torch.ones(B, D, N, device="cuda")
    _, hT, _ = cla.selective_scan_fwd(z, torch.from_numpy(delta).cuda(), torch.from_numpy(A).cuda(), Bm, Bm, h0)
    torch.cuda.synchronize()
    ref = np.exp(delta[:, 0][:, :, None].astype(np.float64) * A.astype(np.float64))
    got = hT.cpu().double().numpy()
    arg = np.abs(delta[:, 0][:, :, None].astype(np.float64) * A.astype(np.float64)) * np.log2(np.e)
    ok = ref > 2.0 ** -120  # normal range
    rel = (got[ok] - ref[ok]) / ref[ok]
    bound = 2.5e-7 + arg[ok] * 2.0 ** -23
    assert np.all(np.abs(rel) <= bound), float(np.max(np.abs(rel) / bound))
    near1 = arg[ok] <= 1.0
    assert near1.sum() > 500
    assert abs(np.mean(rel[near1])) <= 2e-8, np.mean(rel[near1])
