"""Python binding of libcla.so (ctypes), with the C entry points' names.

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  If the
shared library has not been built the import of a function fails loudly;
there is no CPU fallback.

All tensors must be CUDA tensors, contiguous, with the dtype the C ABI names
(float32, or bfloat16 passed as its bit pattern).  Outputs and the workspace
are allocated with torch when not supplied.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcla.so")
_lock = threading.Lock()
_lib = None

CLA_OK = 0
SELECTIVE_CKPT_CHUNK = 64


class ClaError(RuntimeError):
    def __init__(self, fn, status, message):
        super().__init__(f"{fn}: {status_string(status)}: {message}")
        self.status = status


def lib():
    """The loaded libcla.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with chunkwise_linear_attention_gb300.build.build() "
                    "(needs nvcc); there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, SZ, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
            sig = {
                "cla_status_string": ([INT], ctypes.c_char_p),
                "cla_last_error_message": ([], ctypes.c_char_p),
                "cla_check_status": ([P, P], INT),
                "cla_selftest_wait_timeout": ([P, SZ, P], INT),
                "cla_scan_diag_workspace_size": ([I64, I64, I64], SZ),
                "cla_scan_diag_fwd": ([P, P, P, P, P, I64, I64, I64, P, SZ, P], INT),
                "cla_scan_diag_fwd_blelloch": ([P, P, P, P, P, I64, I64, I64, P, SZ, P], INT),
                "cla_scan_diag_bwd": ([P, P, P, P, P, P, P, P, I64, I64, I64, P, SZ, P], INT),
                "cla_scan_diag_fwd_noalloc": ([P, P, P, P, P, I64, I64, I64, P], INT),
                "cla_selective_scan_workspace_size": ([I64, I64, I64, I64], SZ),
                "cla_selective_scan_ckpt_elems": ([I64, I64, I64, I64], SZ),
                "cla_selective_scan_fwd": ([P] * 9 + [I64] * 4 + [P, SZ, P], INT),
                "cla_selective_scan_bwd": ([P] * 15 + [I64] * 4 + [P, SZ, P], INT),
                "cla_chunk_la_workspace_size": ([I64] * 5 + [INT], SZ),
                "cla_chunk_la_fwd": ([P] * 7 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_chunk_la_bwd": ([P] * 12 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_chunk_la_ckpt_size": ([I64] * 5 + [INT], SZ),
                "cla_chunk_la_fwd_ckpt": ([P] * 8 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_chunk_la_bwd_ckpt": ([P] * 13 + [I64] * 5 + [INT, P, SZ, P], INT),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().cla_status_string(int(status)).decode()


def last_error_message() -> str:
    return lib().cla_last_error_message().decode()


def _check(fn: str, status: int) -> None:
    if status != CLA_OK:
        raise ClaError(fn, status, last_error_message())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _ws(nbytes, device, workspace):
    if workspace is None:
        workspace = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace of {workspace.numel()} bytes < {nbytes} needed")
    return workspace


def _out(t, shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device) if t is None else t


def check_status(workspace, stream=None) -> None:
    """Synchronise and raise if a kernel of the last call on `workspace` gave up a wait."""
    _check("cla_check_status", lib().cla_check_status(_ptr(workspace), _stream(stream)))


def selftest_wait_timeout(workspace, stream=None) -> None:
    """Launch the bounded-wait self-test on `workspace` (>= 256 bytes)."""
    _check("cla_selftest_wait_timeout",
           lib().cla_selftest_wait_timeout(_ptr(workspace), workspace.numel(), _stream(stream)))


# ---------------------------------------------------------------- diagonal scan
def scan_diag_workspace_size(B, T, D) -> int:
    return int(lib().cla_scan_diag_workspace_size(B, T, D))


def scan_diag_fwd(a, b, h0=None, *, h=None, hT=None, workspace=None, stream=None):
    """h_t = a_t h_{t-1} + b_t over axis 1 of [B, T, D] (fp32); returns (h, hT)."""
    B, T, D = a.shape
    dev = a.device
    f32 = torch.float32
    h = _out(h, (B, T, D), f32, dev)
    hT = _out(hT, (B, D), f32, dev)
    ws = _ws(scan_diag_workspace_size(B, T, D), dev, workspace)
    _check("cla_scan_diag_fwd", lib().cla_scan_diag_fwd(
        _ptr(a, f32, "a"), _ptr(b, f32, "b"), _ptr(h0, f32, "h0"), _ptr(h, f32, "h"), _ptr(hT, f32, "hT"),
        B, T, D, _ptr(ws), ws.numel(), _stream(stream)))
    return h, hT


def scan_diag_fwd_blelloch(a, b, h0=None, *, h=None, hT=None, workspace=None, stream=None):
    """scan_diag_fwd with a Blelloch tree across the runs of a chunk (a measured
    alternative to Hillis-Steele); returns (h, hT)."""
    B, T, D = a.shape
    dev = a.device
    f32 = torch.float32
    h = _out(h, (B, T, D), f32, dev)
    hT = _out(hT, (B, D), f32, dev)
    ws = _ws(scan_diag_workspace_size(B, T, D), dev, workspace)
    _check("cla_scan_diag_fwd_blelloch", lib().cla_scan_diag_fwd_blelloch(
        _ptr(a, f32, "a"), _ptr(b, f32, "b"), _ptr(h0, f32, "h0"), _ptr(h, f32, "h"), _ptr(hT, f32, "hT"),
        B, T, D, _ptr(ws), ws.numel(), _stream(stream)))
    return h, hT


def scan_diag_fwd_noalloc(a, b, h0=None, *, h=None, hT=None, stream=None):
    """scan_diag_fwd without a workspace: the library's static scratch array
    is used (limited size; overlapping calls race).  Returns (h, hT)."""
    B, T, D = a.shape
    dev = a.device
    f32 = torch.float32
    h = _out(h, (B, T, D), f32, dev)
    hT = _out(hT, (B, D), f32, dev)
    _check("cla_scan_diag_fwd_noalloc", lib().cla_scan_diag_fwd_noalloc(
        _ptr(a, f32, "a"), _ptr(b, f32, "b"), _ptr(h0, f32, "h0"), _ptr(h, f32, "h"), _ptr(hT, f32, "hT"),
        B, T, D, _stream(stream)))
    return h, hT


def scan_diag_bwd(a, h0, h, dh, dhT=None, *, da=None, db=None, dh0=None, workspace=None, stream=None):
    """Adjoint of scan_diag_fwd; returns (da, db, dh0)."""
    B, T, D = a.shape
    dev = a.device
    f32 = torch.float32
    da = _out(da, (B, T, D), f32, dev)
    db = _out(db, (B, T, D), f32, dev)
    dh0 = _out(dh0, (B, D), f32, dev)
    ws = _ws(scan_diag_workspace_size(B, T, D), dev, workspace)
    _check("cla_scan_diag_bwd", lib().cla_scan_diag_bwd(
        _ptr(a, f32, "a"), _ptr(h0, f32, "h0"), _ptr(h, f32, "h"), _ptr(dh, f32, "dh"), _ptr(dhT, f32, "dhT"),
        _ptr(da, f32, "da"), _ptr(db, f32, "db"), _ptr(dh0, f32, "dh0"), B, T, D, _ptr(ws), ws.numel(),
        _stream(stream)))
    return da, db, dh0


# ---------------------------------------------------------------- selective scan
def selective_scan_workspace_size(B, T, D, N) -> int:
    return int(lib().cla_selective_scan_workspace_size(B, T, D, N))


def selective_scan_ckpt_elems(B, T, D, N) -> int:
    return int(lib().cla_selective_scan_ckpt_elems(B, T, D, N))


def selective_scan_fwd(x, delta, A, Bm, Cm, h0=None, *, y=None, hT=None, ckpt=None, want_ckpt=True,
                       workspace=None, stream=None):
    """Selective scan forward; returns (y, hT, ckpt)."""
    B, T, D = x.shape
    N = A.shape[1]
    dev = x.device
    f32, bf16 = torch.float32, torch.bfloat16
    y = _out(y, (B, T, D), f32, dev)
    hT = _out(hT, (B, D, N), f32, dev)
    if ckpt is None and want_ckpt:
        ckpt = torch.empty(selective_scan_ckpt_elems(B, T, D, N), dtype=f32, device=dev)
    ws = _ws(selective_scan_workspace_size(B, T, D, N), dev, workspace)
    _check("cla_selective_scan_fwd", lib().cla_selective_scan_fwd(
        _ptr(x, bf16, "x"), _ptr(delta, f32, "delta"), _ptr(A, f32, "A"), _ptr(Bm, bf16, "Bm"),
        _ptr(Cm, bf16, "Cm"), _ptr(h0, f32, "h0"), _ptr(y, f32, "y"), _ptr(hT, f32, "hT"),
        _ptr(ckpt, f32, "ckpt"), B, T, D, N, _ptr(ws), ws.numel(), _stream(stream)))
    return y, hT, ckpt


def selective_scan_bwd(x, delta, A, Bm, Cm, h0, ckpt, dy, dhT=None, *, dx=None, ddelta=None, dA=None,
                       dB=None, dC=None, dh0=None, want_dA=True, want_dh0=True, workspace=None, stream=None):
    """Selective scan backward; returns (dx, ddelta, dA, dB, dC, dh0)."""
    B, T, D = x.shape
    N = A.shape[1]
    dev = x.device
    f32, bf16 = torch.float32, torch.bfloat16
    dx = _out(dx, (B, T, D), f32, dev)
    ddelta = _out(ddelta, (B, T, D), f32, dev)
    dA = _out(dA, (D, N), f32, dev) if (want_dA or dA is not None) else None
    dB = _out(dB, (B, T, N), f32, dev)
    dC = _out(dC, (B, T, N), f32, dev)
    dh0 = _out(dh0, (B, D, N), f32, dev) if (want_dh0 or dh0 is not None) else None
    ws = _ws(selective_scan_workspace_size(B, T, D, N), dev, workspace)
    _check("cla_selective_scan_bwd", lib().cla_selective_scan_bwd(
        _ptr(x, bf16, "x"), _ptr(delta, f32, "delta"), _ptr(A, f32, "A"), _ptr(Bm, bf16, "Bm"),
        _ptr(Cm, bf16, "Cm"), _ptr(h0, f32, "h0"), _ptr(ckpt, f32, "ckpt"), _ptr(dy, f32, "dy"),
        _ptr(dhT, f32, "dhT"), _ptr(dx, f32, "dx"), _ptr(ddelta, f32, "ddelta"), _ptr(dA, f32, "dA"),
        _ptr(dB, f32, "dB"), _ptr(dC, f32, "dC"), _ptr(dh0, f32, "dh0"), B, T, D, N, _ptr(ws), ws.numel(),
        _stream(stream)))
    return dx, ddelta, dA, dB, dC, dh0


# ---------------------------------------------------------------- chunkwise linear attention
def chunk_la_workspace_size(B, H, T, dim_k, dim_v, chunk) -> int:
    return int(lib().cla_chunk_la_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def chunk_la_ckpt_size(B, H, T, dim_k, dim_v, chunk) -> int:
    """Bytes of the segment-state checkpoint the forward can save for the backward."""
    return int(lib().cla_chunk_la_ckpt_size(B, H, T, dim_k, dim_v, int(chunk)))


def chunk_la_ckpt(q, v, *, chunk=64):
    """A device buffer (fp32) for the checkpoint of a forward on q [B, H, T, dk], v [.., dv]."""
    B, H, T, dk = q.shape
    n = chunk_la_ckpt_size(B, H, T, dk, v.shape[-1], chunk) // 4
    return torch.empty(max(n, 1), dtype=torch.float32, device=q.device)


def _ckpt_ptr(ckpt, B, H, T, dk, dv, chunk):
    if ckpt is None:
        return None
    need = chunk_la_ckpt_size(B, H, T, dk, dv, chunk)
    if ckpt.numel() * ckpt.element_size() < need:
        raise ValueError(f"ckpt: need at least {need} bytes, got {ckpt.numel() * ckpt.element_size()}")
    return _ptr(ckpt, torch.float32, "ckpt")


def chunk_la_fwd(q, k, v, log_decay, S0=None, *, chunk=64, o=None, ST=None, ckpt=None, workspace=None,
                 stream=None):
    """Chunkwise decayed linear attention forward; returns (o, ST).  With ckpt (see
    chunk_la_ckpt) it also saves the state entering each segment for chunk_la_bwd."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    o = _out(o, (B, H, T, dv), f32, dev)
    ST = _out(ST, (B, H, dk, dv), f32, dev)
    ws = _ws(chunk_la_workspace_size(B, H, T, dk, dv, chunk), dev, workspace)
    args = (_ptr(q, bf16, "q"), _ptr(k, bf16, "k"), _ptr(v, bf16, "v"), _ptr(log_decay, f32, "log_decay"),
            _ptr(S0, f32, "S0"), _ptr(o, f32, "o"), _ptr(ST, f32, "ST"))
    tail = (B, H, T, dk, dv, int(chunk), _ptr(ws), ws.numel(), _stream(stream))
    if ckpt is None:
        _check("cla_chunk_la_fwd", lib().cla_chunk_la_fwd(*args, *tail))
    else:
        _check("cla_chunk_la_fwd_ckpt", lib().cla_chunk_la_fwd_ckpt(
            *args, _ckpt_ptr(ckpt, B, H, T, dk, dv, chunk), *tail))
    return o, ST


def chunk_la_bwd(q, k, v, log_decay, S0, dO, dST=None, *, chunk=64, dq=None, dk=None, dv=None,
                 dlog_decay=None, dS0=None, ckpt=None, workspace=None, stream=None):
    """Chunkwise decayed linear attention backward; returns (dq, dk, dv, dlog_decay, dS0).  ckpt:
    the checkpoint a chunk_la_fwd on the same inputs saved (its states are then not rebuilt)."""
    B, H, T, dkk = q.shape
    dvv = v.shape[-1]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    dq = _out(dq, (B, H, T, dkk), f32, dev)
    dk = _out(dk, (B, H, T, dkk), f32, dev)
    dv = _out(dv, (B, H, T, dvv), f32, dev)
    dlog_decay = _out(dlog_decay, (B, H, T), f32, dev)
    dS0 = _out(dS0, (B, H, dkk, dvv), f32, dev)
    ws = _ws(chunk_la_workspace_size(B, H, T, dkk, dvv, chunk), dev, workspace)
    args = (_ptr(q, bf16, "q"), _ptr(k, bf16, "k"), _ptr(v, bf16, "v"), _ptr(log_decay, f32, "log_decay"),
            _ptr(S0, f32, "S0"), _ptr(dO, bf16, "dO"), _ptr(dST, f32, "dST"), _ptr(dq, f32, "dq"),
            _ptr(dk, f32, "dk"), _ptr(dv, f32, "dv"), _ptr(dlog_decay, f32, "dlog_decay"), _ptr(dS0, f32, "dS0"))
    tail = (B, H, T, dkk, dvv, int(chunk), _ptr(ws), ws.numel(), _stream(stream))
    if ckpt is None:
        _check("cla_chunk_la_bwd", lib().cla_chunk_la_bwd(*args, *tail))
    else:
        _check("cla_chunk_la_bwd_ckpt", lib().cla_chunk_la_bwd_ckpt(
            *args, _ckpt_ptr(ckpt, B, H, T, dkk, dvv, chunk), *tail))
    return dq, dk, dv, dlog_decay, dS0
