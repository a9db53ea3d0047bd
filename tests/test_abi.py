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


def test_plan_named_aliases(lib):
    """The boundary plan's names for the workspace queries and the status call are the same
    functions as the library's own."""
    lib.cla_scan_diag_workspace.restype = ctypes.c_size_t
    lib.cla_scan_diag_workspace.argtypes = [ctypes.c_int64] * 3
    lib.cla_chunk_la_workspace.restype = ctypes.c_size_t
    lib.cla_chunk_la_workspace.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_int]
    for shape in ((8, 4096, 1024), (1, 1024, 64), (3, 77, 6), (-1, 1, 1)):
        assert lib.cla_scan_diag_workspace(*shape) == lib.cla_scan_diag_workspace_size(*shape)
    for shape in ((4, 16, 8192, 64, 64, 64), (1, 32, 65536, 128, 128, 128), (1, 2, 1000, 96, 64, 64)):
        assert lib.cla_chunk_la_workspace(*shape) == lib.cla_chunk_la_workspace_size(*shape)
    assert hasattr(lib, "cla_check_device_status")


def test_chunk_la_ckpt_size_follows_the_segment_rule(lib):
    """The checkpoint holds one d_k x d_v fp32 state per segment and head; segments are the
    largest of 64/32/16/8 chunks that still leave at least 1024 blocks (heads x 64-column
    blocks x segments; 256 in the compact layout, d_k = d_v = chunk = 64).  Long-context workload, chunk 128: 512 chunks per head, 32 heads,
    2 column blocks -> segments of 32 chunks, 16 of them."""
    f = lib.cla_chunk_la_ckpt_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_int]
    assert f(1, 32, 65536, 128, 128, 128) == 16 * 32 * 128 * 128 * 4
    # chunk 64: 1024 chunks, segments of 64 chunks (16 x 32 x 2 = 1024 blocks)
    assert f(1, 32, 65536, 128, 128, 64) == 16 * 32 * 128 * 128 * 4
    # constant-decay workload (the compact layout, d = chunk = 64: at least 256 blocks): 128
    # chunks per head, 64 heads, one column block -> segments of 32, 4 of them
    assert f(4, 16, 8192, 64, 64, 64) == 4 * 64 * 64 * 64 * 4
    # compact layout, one head of 1024 chunks: no choice reaches 256 blocks -> the smallest
    # (8 chunks), 128 segments
    assert f(1, 1, 65536, 64, 64, 64) == 128 * 1 * 64 * 64 * 4
    # compact layout, 256 heads: 64-chunk segments already give 512 blocks
    assert f(8, 32, 8192, 64, 64, 64) == 2 * 256 * 64 * 64 * 4
    # d = 64 at chunk 128 is not the compact layout: the 1024-block rule, 64 chunks per head and
    # 64 heads -> even 8-chunk segments give 512 blocks, so the smallest choice, 8 segments
    assert f(4, 16, 8192, 64, 64, 128) == 8 * 64 * 64 * 64 * 4
    assert f(-1, 1, 1, 64, 64, 64) == 0 and f(1, 1, 1, 64, 64, 0) == 0


def test_gla_and_delta_ckpt_sizes(lib):
    """GLA: one d_k x d_v fp32 state per segment and head, segments the largest of 64/32/16/8
    chunks that leave at least 1024 blocks (heads x max(d_k, d_v)/64 column blocks x segments).
    The workload (2 x 16 heads, 16384 tokens = 256 chunks, d = 128): 16-chunk segments, 16 of
    them.  Delta rule: per 64-token chunk the state (d_k x d_v fp32), the (I + A)^-1 parts
    (16 KB) and E (16 KB).  Both 0 for what the calls refuse."""
    for n in ("cla_gla_ckpt_size", "cla_delta_ckpt_size"):
        f = getattr(lib, n)
        f.restype = ctypes.c_size_t
        f.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_int]
    g, d = lib.cla_gla_ckpt_size, lib.cla_delta_ckpt_size
    assert g(2, 16, 16384, 128, 128, 64) == 16 * 32 * 128 * 128 * 4
    assert g(2, 16, 16384, 64, 128, 64) == 16 * 32 * 64 * 128 * 4  # column blocks from max(d_k, d_v)
    assert g(1, 1, 1000, 96, 128, 64) == 0 and g(1, 1, 1000, 128, 128, 128) == 0
    assert d(4, 32, 4096, 128, 128, 64) == 4 * 32 * 64 * (128 * 128 * 4 + 16384 + 16384)
    assert d(1, 1, 100, 64, 192, 64) == 2 * (64 * 192 * 4 + 16384 + 16384)  # ragged: 2 chunks
    assert d(1, 1, 100, 64, 64, 128) == 0


def test_chunk_la_size_queries_refuse_what_the_calls_refuse(lib):
    """The workspace and checkpoint size queries return 0 for head dims or chunks the fwd / bwd
    calls reject (CLA_ERR_UNSUPPORTED), so no caller sizes a buffer for a call that cannot run."""
    i64, ci = ctypes.c_int64, ctypes.c_int
    for f in (lib.cla_chunk_la_workspace_size, lib.cla_chunk_la_ckpt_size):
        f.restype = ctypes.c_size_t
        f.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_int]
    P = ctypes.c_void_p
    d, ws, big = P(256), P(1 << 20), ctypes.c_size_t(1 << 30)
    for dk, dv, chunk in ((32, 64, 64), (64, 96, 64), (256, 256, 128), (64, 64, 32), (128, 128, 256)):
        assert lib.cla_chunk_la_workspace_size(1, 2, 1000, dk, dv, chunk) == 0, (dk, dv, chunk)
        assert lib.cla_chunk_la_ckpt_size(1, 2, 1000, dk, dv, chunk) == 0, (dk, dv, chunk)
        st = lib.cla_chunk_la_fwd(d, d, d, d, None, d, None, i64(1), i64(2), i64(1000), i64(dk), i64(dv), ci(chunk),
                                  ws, big, None)
        assert st == 2, (dk, dv, chunk)
    for dk, dv, chunk in ((64, 64, 64), (64, 128, 128), (128, 64, 64), (128, 128, 128)):
        assert lib.cla_chunk_la_workspace_size(1, 2, 1000, dk, dv, chunk) > 0
        assert lib.cla_chunk_la_ckpt_size(1, 2, 1000, dk, dv, chunk) > 0


def test_chunk_la_ckpt_rejects_unaligned_without_gpu(lib):
    P = ctypes.c_void_p
    d = P(256)
    i64 = ctypes.c_int64
    st = lib.cla_chunk_la_fwd_ckpt(d, d, d, d, None, d, None, P(260), i64(1), i64(1), i64(256), i64(64), i64(64),
                                   ctypes.c_int(64), d, ctypes.c_size_t(1 << 30), None)
    assert st == 1  # CLA_ERR_INVALID_ARG
    assert b"ckpt" in lib.cla_last_error_message()
    st = lib.cla_chunk_la_bwd_ckpt(d, d, d, d, None, d, None, d, d, d, None, None, P(260), i64(1), i64(1),
                                   i64(256), i64(64), i64(64), ctypes.c_int(64), d, ctypes.c_size_t(1 << 30), None)
    assert st == 1


def test_binding_refuses_host_tensors(lib):
    """No CPU fallback: host tensors are rejected before anything reaches the library."""
    import torch

    import chunkwise_linear_attention_gb300 as cla

    a = torch.rand(1, 8, 4)
    with pytest.raises(ValueError, match="CUDA"):
        cla.scan_diag_fwd(a, a)
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        cla.chunk_la_fwd(q, q, q, torch.zeros(1, 1, 8))


def test_misaligned_pointers_rejected_without_gpu(lib):
    """A pointer misaligned for the kernel's loads or stores is refused on the host
    (CLA_ERR_INVALID_ARG) before anything is enqueued, so it never reaches the GPU."""
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    d, ws, big = P(256), P(1 << 20), sz(1 << 30)
    odd2, odd4 = P(258), P(260)  # 2-byte and 4-byte aligned, not 16-byte

    # diagonal scan: fp32 tensors need 4-byte alignment
    st = lib.cla_scan_diag_fwd(odd2, d, None, d, None, i64(2), i64(64), i64(64), ws, big, None)
    assert st == 1 and b"aligned" in lib.cla_last_error_message()
    st = lib.cla_scan_diag_bwd(d, None, None, d, d, None, d, d, odd2, i64(2), i64(64), i64(64), ws, big, None)
    assert st == 1
    st = lib.cla_scan_diag_fwd_noalloc(d, d, odd2, d, None, i64(2), i64(64), i64(64), None)
    assert st == 1

    # selective scan: bf16 inputs need 2 bytes, fp32 tensors 4
    st = lib.cla_selective_scan_fwd(P(257), d, d, d, d, None, d, None, None, i64(1), i64(64), i64(64), i64(16),
                                    ws, big, None)
    assert st == 1
    st = lib.cla_selective_scan_fwd(d, odd2, d, d, d, None, d, None, None, i64(1), i64(64), i64(64), i64(16),
                                    ws, big, None)
    assert st == 1
    st = lib.cla_selective_scan_bwd(d, d, d, d, d, None, d, d, None, d, d, odd2, d, d, None, i64(1), i64(64),
                                    i64(64), i64(16), ws, big, None)
    assert st == 1

    # chunkwise LA: S0 and dST are read in 16-byte rows; the fp32 vectors need 4 bytes
    fwd = lib.cla_chunk_la_fwd
    st = fwd(d, d, d, d, odd4, d, None, i64(1), i64(1), i64(256), i64(64), i64(64), ctypes.c_int(64), ws, big, None)
    assert st == 1 and b"S0" in lib.cla_last_error_message()
    st = fwd(d, d, d, odd2, None, d, None, i64(1), i64(1), i64(256), i64(64), i64(64), ctypes.c_int(64), ws, big,
             None)
    assert st == 1
    bwd = lib.cla_chunk_la_bwd
    st = bwd(d, d, d, d, None, d, odd4, d, d, d, None, None, i64(1), i64(1), i64(256), i64(64), i64(64),
             ctypes.c_int(64), ws, big, None)
    assert st == 1 and b"dST" in lib.cla_last_error_message()
    st = bwd(d, d, d, d, None, d, None, d, d, d, None, odd2, i64(1), i64(1), i64(256), i64(64), i64(64),
             ctypes.c_int(64), ws, big, None)
    assert st == 1
    # the same pointers 16-byte aligned pass validation up to the workspace check
    st = fwd(d, d, d, d, d, d, None, i64(1), i64(1), i64(256), i64(64), i64(64), ctypes.c_int(64), ws, sz(16), None)
    assert st == 5  # CLA_ERR_WORKSPACE: too small


def test_sizes_whose_counts_would_overflow_are_unsupported(lib):
    """Sizes whose grid or workspace arithmetic would overflow a 64-bit product are refused
    (CLA_ERR_UNSUPPORTED) and the size queries return 0, instead of wrapping around."""
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    d, ws, big = P(256), P(1 << 20), sz(1 << 30)
    for f in (lib.cla_scan_diag_workspace_size, lib.cla_selective_scan_workspace_size,
              lib.cla_selective_scan_ckpt_elems, lib.cla_chunk_la_workspace_size, lib.cla_chunk_la_ckpt_size):
        f.restype = ctypes.c_size_t

    B, T, D = 1 << 24, 1 << 40, 1 << 30  # each within its own limit, product far beyond 2^63
    assert lib.cla_scan_diag_workspace_size(i64(B), i64(T), i64(D)) == 0
    st = lib.cla_scan_diag_fwd(d, d, None, d, None, i64(B), i64(T), i64(D), ws, big, None)
    assert st == 2 and b"out of range" in lib.cla_last_error_message()

    B, T, D = 1 << 20, 1 << 36, 1 << 24
    assert lib.cla_selective_scan_workspace_size(i64(B), i64(T), i64(D), i64(16)) == 0
    assert lib.cla_selective_scan_ckpt_elems(i64(B), i64(T), i64(D), i64(16)) == 0
    st = lib.cla_selective_scan_fwd(d, d, d, d, d, None, d, None, None, i64(B), i64(T), i64(D), i64(16), ws, big,
                                    None)
    assert st == 2

    # B * H = 2^64 wraps to 0 in 64-bit arithmetic
    B = H = 1 << 32
    args = (i64(B), i64(H), i64(256), i64(64), i64(64), ctypes.c_int(64))
    assert lib.cla_chunk_la_workspace_size(*args) == 0 and lib.cla_chunk_la_ckpt_size(*args) == 0
    st = lib.cla_chunk_la_fwd(d, d, d, d, None, d, None, *args, ws, big, None)
    assert st == 2
    # B*H within 2^24 but B*H*T beyond 2^40
    args = (i64(1 << 12), i64(1 << 12), i64(1 << 30), i64(64), i64(64), ctypes.c_int(64))
    assert lib.cla_chunk_la_workspace_size(*args) == 0
    st = lib.cla_chunk_la_bwd(d, d, d, d, None, d, None, d, d, d, None, None, *args, ws, big, None)
    assert st == 2
    # the workloads' own sizes are unaffected
    assert lib.cla_chunk_la_workspace_size(i64(1), i64(32), i64(65536), i64(128), i64(128), ctypes.c_int(128)) > 0
    assert lib.cla_selective_scan_workspace_size(i64(4), i64(8192), i64(2048), i64(16)) > 0
    assert lib.cla_scan_diag_workspace_size(i64(8), i64(4096), i64(1024)) > 0


def test_binding_checks_shapes_before_anything_else(lib):
    """The binding checks every tensor's dtype and shape against the sizes it passes (the C ABI
    sees bare pointers and cannot), for all arguments before any device check."""
    import torch

    import chunkwise_linear_attention_gb300 as cla

    f32, bf16 = torch.float32, torch.bfloat16
    a = torch.rand(2, 8, 4)

    def raises(fn, *args, match, **kw):
        with pytest.raises(ValueError, match=match):
            fn(*args, **kw)

    raises(cla.scan_diag_fwd, a, torch.rand(2, 8, 3), match=r"b must have shape \(2, 8, 4\)")
    raises(cla.scan_diag_fwd, a, a, torch.rand(2, 5), match="h0 must have shape")
    raises(cla.scan_diag_fwd, a, a, h=torch.empty(2, 8, 5), match="h must have shape")
    raises(cla.scan_diag_fwd, a, a.double(), match="b must be torch.float32")
    raises(cla.scan_diag_fwd, torch.rand(8, 4), a, match="a must have 3 dimensions")
    raises(cla.scan_diag_fwd_noalloc, a, a, hT=torch.empty(3, 4), match="hT must have shape")
    raises(cla.scan_diag_bwd, a, None, None, a, torch.rand(2, 7, 4), match="dh must have shape")
    raises(cla.scan_diag_bwd, a, torch.rand(2, 8, 5), None, None, a, match="b must have shape")

    x = torch.zeros(1, 64, 32, dtype=bf16)
    A = torch.zeros(32, 16)
    Bm = torch.zeros(1, 64, 16, dtype=bf16)
    raises(cla.selective_scan_fwd, x, torch.zeros(1, 64, 32), A, Bm, torch.zeros(1, 64, 8, dtype=bf16),
           match="Cm must have shape")
    raises(cla.selective_scan_fwd, x, torch.zeros(1, 64, 32), torch.zeros(31, 16), Bm, Bm, match="A must have shape")
    raises(cla.selective_scan_bwd, x, torch.zeros(1, 64, 32), A, Bm, Bm, None, torch.zeros(3), torch.zeros(1, 64, 32),
           match="ckpt: need at least")

    q = torch.zeros(1, 2, 16, 64, dtype=bf16)
    ld = torch.zeros(1, 2, 16)
    raises(cla.chunk_la_fwd, q, q, q, torch.zeros(1, 2, 15), match="log_decay must have shape")
    raises(cla.chunk_la_fwd, q, q, q, ld, torch.zeros(1, 2, 64, 32), match="S0 must have shape")
    raises(cla.chunk_la_fwd, q, q.float(), q, ld, match="k must be torch.bfloat16")
    raises(cla.chunk_la_fwd, q, q, q, ld, ckpt=torch.zeros(1), match="ckpt: need at least")
    raises(cla.chunk_la_bwd, q, q, q, ld, None, torch.zeros(1, 2, 16, 32, dtype=bf16), match="dO must have shape")
    raises(cla.chunk_la_bwd, q, q, q, ld, None, q, dST=torch.zeros(2, 64, 64), match="dST must have shape")
    # with every shape right, the first host tensor stops the call
    raises(cla.chunk_la_bwd, q, q, q, ld, None, q, match="q must be a CUDA tensor")
