"""The no-allocation forward diagonal scan (cla_scan_diag_fwd_noalloc).

It serves callers that cannot give the library a workspace (a framework
plugin with no scratch buffer, a fixed device-memory footprint, a path where
allocation calls are not allowed).  Called through the C ABI, it must agree
with cla_scan_diag_fwd within the fp32 tolerance of the scan tests, on two
calls in a row (the static scratch keeps the previous call's contents), and
refuse sizes whose scratch exceeds its fixed array without launching.  On a
small case it is also checked against the float64 oracle directly, so that a
fault shared by both library paths cannot pass unseen, and its status query
reports a clean run.

This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import oracle
import workloads
from tests._parity import assert_fp32

pytestmark = pytest.mark.gpu


def _fn():
    import chunkwise_linear_attention_gb300 as cla

    f = cla.lib().cla_scan_diag_fwd_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [P, P, P, P, P, I64, I64, I64, P]
    f.restype = ctypes.c_int
    return cla, f


def f_status(stream):
    import chunkwise_linear_attention_gb300 as cla

    g = cla.lib().cla_scan_diag_noalloc_check_status
    g.argtypes = [ctypes.c_void_p]
    g.restype = ctypes.c_int
    return g(stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("B,T,D,with_h0", [(2, 1000, 256, True), (8, 4096, 1024, True), (3, 77, 6, False)])
def test_noalloc_matches_workspace_path_twice(B, T, D, with_h0):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cla, f = _fn()
    inp = workloads.make("scan", B=B, T=T, D=D)
    a, b = inp["a"].cuda(), inp["b"].cuda()
    h0 = inp["h0"].cuda() if with_h0 else None
    ref_h, ref_hT = cla.scan_diag_fwd(a, b, h0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        h = torch.full((B, T, D), float("nan"), device="cuda")
        hT = torch.full((B, D), float("nan"), device="cuda")
        st = f(_p(a), _p(b), _p(h0), _p(h), _p(hT), B, T, D, stream)
        assert st == 0, cla.last_error_message()
        torch.cuda.synchronize()
        assert_fp32("h", h, ref_h)
        assert_fp32("hT", hT, ref_hT)
        assert f_status(stream) == 0, cla.last_error_message()


def test_noalloc_matches_oracle_twice():
    """Small ragged case against the float64 oracle on the same seeded inputs."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cla, f = _fn()
    B, T, D = 3, 77, 6
    inp = workloads.make("scan", B=B, T=T, D=D)
    ro_h, ro_hT = oracle.scan_diag_fwd(inp["a"], inp["b"], inp["h0"])
    a, b, h0 = inp["a"].cuda(), inp["b"].cuda(), inp["h0"].cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        h = torch.full((B, T, D), float("nan"), device="cuda")
        hT = torch.full((B, D), float("nan"), device="cuda")
        assert f(_p(a), _p(b), _p(h0), _p(h), _p(hT), B, T, D, stream) == 0, cla.last_error_message()
        assert f_status(stream) == 0, cla.last_error_message()
        assert_fp32("h", h, ro_h)
        assert_fp32("hT", hT, ro_hT)


def test_noalloc_rejects_oversize():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cla, f = _fn()
    x = torch.empty(4, device="cuda")
    # 16 x 8192 x 1024 needs about 25 MB of look-back scratch
    st = f(_p(x), _p(x), None, _p(x), None, 16, 8192, 1024, None)
    assert st == 2  # CLA_ERR_UNSUPPORTED, nothing launched
    assert "static array" in cla.last_error_message()
