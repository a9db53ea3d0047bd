"""Delta rule with a decay per head (Gated DeltaNet), forward: GPU (through the
C ABI) vs the oracle's per-token recurrence, with the bf16 tolerance (per
output tensor, |x - r| / rms(r): max <= 2e-2, mean <= 5e-3), and the range
check on non-finite decays."""
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


def test_delta_nonfinite_decay_is_reported(cla):
    inp = workloads.make("delta", B=1, H=1, T=200, dk=64, dv=64)
    inp["log_a"][0, 0, 77] = -float("inf")
    t = {k: v.cuda() for k, v in inp.items()}
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], workspace=ws)
    with pytest.raises(cla.ClaError, match="outside the kernel's range") as ei:
        cla.check_status(ws)
    assert ei.value.status == 2


def test_delta_workload_full_sampled_heads(cla):
    """The full delta workload (4 x 32 x 4096, d = 128), every output of three heads."""
    inp = workloads.make("delta")
    _run(cla, inp, heads=[0, 17, 31])
