"""The C ABI library builds, loads, exports every symbol its header declares,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cla.h")


@pytest.fixture(scope="module")
def lib():
    from chunkwise_linear_attention_gb300 import build

    build.build()
    import chunkwise_linear_attention_gb300 as cla

    return cla.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cla_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = _declared()
    for want in ("cla_scan_diag_fwd", "cla_scan_diag_bwd", "cla_selective_scan_fwd", "cla_selective_scan_bwd",
                 "cla_chunk_la_fwd", "cla_chunk_la_bwd", "cla_check_status"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in cla.h but not exported"


def test_status_strings(lib):
    import chunkwise_linear_attention_gb300 as cla

    assert cla.status_string(0) == "CLA_OK"
    assert cla.status_string(4) == "CLA_ERR_TIMEOUT"
    assert cla.status_string(99) == "CLA_ERR_UNKNOWN"


def test_host_validation_without_gpu(lib):
    """Negative sizes and missing pointers are rejected before any CUDA call."""
    P = ctypes.c_void_p
    st = lib.cla_scan_diag_fwd(None, None, None, None, None, -1, 4, 4, None, 0, None)
    assert st == 1  # CLA_ERR_INVALID_ARG
    assert b"negative" in lib.cla_last_error_message()
    dummy = P(256)
    st = lib.cla_scan_diag_fwd(None, None, None, None, None, 2, 4, 4, dummy, 1 << 20, None)
    assert st == 1
    st = lib.cla_scan_diag_fwd(dummy, dummy, None, dummy, None, 2, 4, 4, None, 0, None)
    assert st == 5  # CLA_ERR_WORKSPACE
    st = lib.cla_scan_diag_fwd(dummy, dummy, None, dummy, None, 2, 100, 64, dummy, 16, None)
    assert st == 5
    assert lib.cla_scan_diag_workspace_size(8, 4096, 1024) > 0
    assert lib.cla_scan_diag_workspace_size(-1, 1, 1) == 0
