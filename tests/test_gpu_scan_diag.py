"""Diagonal scan, forward and backward: GPU (through the C ABI) vs oracle."""
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


def _run(cla, inp, with_h0=True, with_dhT=False, seed=0, recompute=False):
    """recompute: the backward gets b instead of the forward's h and rebuilds the states."""
    dev = torch.device("cuda")
    a, b = inp["a"].to(dev), inp["b"].to(dev)
    h0 = inp["h0"].to(dev) if (with_h0 and inp.get("h0") is not None) else None
    B, T, D = a.shape
    dh = inp.get("dh")
    if dh is None:
        dh = torch.from_numpy(np.random.default_rng(seed).standard_normal((B, T, D)).astype(np.float32))
    dhT = torch.from_numpy(np.random.default_rng(seed + 1).standard_normal((B, D)).astype(np.float32)) if with_dhT else None
    h, hT = cla.scan_diag_fwd(a, b, h0)
    if recompute:
        da, db, dh0 = cla.scan_diag_bwd(a, b, h0, None, dh.to(dev), dhT.to(dev) if dhT is not None else None)
    else:
        da, db, dh0 = cla.scan_diag_bwd(a, None, h0, h, dh.to(dev), dhT.to(dev) if dhT is not None else None)
    torch.cuda.synchronize()
    h0c = h0.cpu() if h0 is not None else None
    rh, rhT = oracle.scan_diag_fwd(inp["a"], inp["b"], h0c)
    rda, rdb, rdh0 = oracle.scan_diag_bwd(inp["a"], inp["b"], h0c, dh, dhT)
    assert_fp32("h", h, rh)
    assert_fp32("hT", hT, rhT)
    assert_fp32("db", db, rdb)
    assert_fp32("da", da, rda)
    assert_fp32("dh0", dh0, rdh0)


@pytest.mark.parametrize("B,T,D", [(1, 1, 4), (2, 63, 16), (2, 64, 16), (2, 65, 20), (3, 200, 96),
                                   (1, 1000, 7), (2, 513, 130), (1, 4097, 8), (2, 130, 3), (2, 2500, 12),
                                   (1, 4096, 64)])
@pytest.mark.parametrize("with_h0", [False, True])
def test_scan_diag_small(cla, B, T, D, with_h0):
    inp = workloads.make("scan", B=B, T=T, D=D)
    _run(cla, inp, with_h0=with_h0, with_dhT=True)


@pytest.mark.parametrize("B,T,D", [(1, 1, 4), (2, 63, 16), (2, 64, 16), (2, 65, 20), (3, 200, 96),
                                   (1, 1000, 7), (2, 513, 130), (1, 4097, 8), (2, 130, 3)])
@pytest.mark.parametrize("with_h0", [False, True])
def test_scan_diag_bwd_recompute_small(cla, B, T, D, with_h0):
    """Backward without the forward's states: rebuilt from (a, b, h0) chunk by chunk."""
    inp = workloads.make("scan", B=B, T=T, D=D)
    _run(cla, inp, with_h0=with_h0, with_dhT=True, recompute=True)


def test_scan_diag_bwd_recompute_workload_full(cla):
    """8 x 4096 x 1024 backward with recomputed states, every output element."""
    inp = workloads.make("scan")
    _run(cla, inp, with_h0=True, with_dhT=True, recompute=True)


def test_scan_diag_small_workload_full(cla):
    """1 x 1024 x 64, a ~ U(0.8, 0.999) (long memory), forward."""
    inp = workloads.make("scan_small")
    dev = torch.device("cuda")
    h, hT = cla.scan_diag_fwd(inp["a"].to(dev), inp["b"].to(dev))
    torch.cuda.synchronize()
    rh, rhT = oracle.scan_diag_fwd(inp["a"], inp["b"])
    assert_fp32("h", h, rh)
    assert_fp32("hT", hT, rhT)


def test_scan_diag_workload_full(cla):
    """8 x 4096 x 1024, forward and backward, every output element."""
    inp = workloads.make("scan")
    _run(cla, inp, with_h0=True)


def test_scan_diag_empty(cla):
    dev = torch.device("cuda")
    h0 = torch.randn(2, 8, device=dev)
    a = torch.empty(2, 0, 8, device=dev)
    h, hT = cla.scan_diag_fwd(a, a, h0)
    da, db, dh0 = cla.scan_diag_bwd(a, None, h0, h, a, hT * 0 + 3.0)
    torch.cuda.synchronize()
    assert torch.equal(hT, h0)
    assert torch.all(dh0 == 3.0)
    a = torch.empty(0, 5, 8, device=dev)
    cla.scan_diag_fwd(a, a)


def test_scan_diag_canaries_untouched(cla):
    """Guard regions around every output stay as written."""
    dev = torch.device("cuda")
    inp = workloads.make("scan", B=2, T=77, D=36)
    B, T, D = inp["a"].shape
    pad = 1024

    def guarded(n):
        buf = torch.full((n + 2 * pad,), 12345.0, device=dev)
        return buf, buf[pad:pad + n]

    hb, h = guarded(B * T * D)
    tb, hT = guarded(B * D)
    cla.scan_diag_fwd(inp["a"].to(dev), inp["b"].to(dev), inp["h0"].to(dev), h=h.view(B, T, D), hT=hT.view(B, D))
    dab, da = guarded(B * T * D)
    dbb, db = guarded(B * T * D)
    d0b, dh0 = guarded(B * D)
    cla.scan_diag_bwd(inp["a"].to(dev), None, inp["h0"].to(dev), h.view(B, T, D), inp["dh"].to(dev),
                      da=da.view(B, T, D), db=db.view(B, T, D), dh0=dh0.view(B, D))
    torch.cuda.synchronize()
    for buf in (hb, tb, dab, dbb, d0b):
        assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[-pad:] == 12345.0)


def test_scan_diag_reused_workspace_and_status(cla):
    """The same workspace serves repeated calls; no wait gave up.  Look-back
    may compose predecessors in a different grouping from run to run, so two
    runs agree to rounding, not bit for bit."""
    dev = torch.device("cuda")
    inp = workloads.make("scan", B=2, T=1000, D=256)
    a, b, h0 = inp["a"].to(dev), inp["b"].to(dev), inp["h0"].to(dev)
    ws = torch.empty(cla.scan_diag_workspace_size(2, 1000, 256), dtype=torch.uint8, device=dev)
    h1, _ = cla.scan_diag_fwd(a, b, h0, workspace=ws)
    h2, _ = cla.scan_diag_fwd(a, b, h0, workspace=ws)
    cla.check_status(ws)
    assert float(((h1 - h2).abs() / h2.abs().clamp_min(1.0)).max()) <= 1e-6


@pytest.mark.parametrize("B,T,D", [(1, 1, 4), (2, 63, 16), (2, 65, 20), (3, 200, 96), (1, 1000, 7), (2, 513, 130),
                                   (1, 4097, 8)])
@pytest.mark.parametrize("with_h0", [False, True])
def test_scan_diag_blelloch_small(cla, B, T, D, with_h0):
    """The Blelloch composition of a chunk's runs gives the recurrence's states."""
    inp = workloads.make("scan", B=B, T=T, D=D)
    dev = torch.device("cuda")
    h0 = inp["h0"].to(dev) if with_h0 else None
    h, hT = cla.scan_diag_fwd_blelloch(inp["a"].to(dev), inp["b"].to(dev), h0)
    torch.cuda.synchronize()
    rh, rhT = oracle.scan_diag_fwd(inp["a"], inp["b"], inp["h0"] if with_h0 else None)
    assert_fp32("h", h, rh)
    assert_fp32("hT", hT, rhT)


def test_scan_diag_blelloch_workload_full(cla):
    """8 x 4096 x 1024 forward with the Blelloch composition, every element."""
    inp = workloads.make("scan")
    dev = torch.device("cuda")
    h, hT = cla.scan_diag_fwd_blelloch(inp["a"].to(dev), inp["b"].to(dev), inp["h0"].to(dev))
    torch.cuda.synchronize()
    rh, rhT = oracle.scan_diag_fwd(inp["a"], inp["b"], inp["h0"])
    assert_fp32("h", h, rh)
    assert_fp32("hT", hT, rhT)
