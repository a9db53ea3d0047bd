"""A cross-block wait that runs out reports an error status; the context
stays usable (no trap, no fault, no hang)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import chunkwise_linear_attention_gb300 as cla

    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    cla.selftest_wait_timeout(ws)
    with pytest.raises(cla.ClaError) as ei:
        cla.check_status(ws)
    assert ei.value.status == 4  # CLA_ERR_TIMEOUT
    # the context still works afterwards
    x = torch.ones(1000, device="cuda")
    assert float(x.sum()) == 1000.0
    a = torch.full((1, 10, 4), 0.5, device="cuda")
    # reusing the workspace that timed out: the new call's status replaces the old one
    h, hT = cla.scan_diag_fwd(a, torch.ones_like(a), workspace=ws)
    cla.check_status(ws)
    ws2 = torch.empty(cla.scan_diag_workspace_size(8, 4096, 64), dtype=torch.uint8, device="cuda")
    a2 = torch.full((8, 4096, 64), 0.5, device="cuda")
    cla.scan_diag_fwd(a2, torch.ones_like(a2), workspace=ws2)  # the multi-block path
    cla.check_status(ws2)
    assert abs(float(hT[0, 0]) - 2.0 * (1 - 0.5 ** 10)) < 1e-6
