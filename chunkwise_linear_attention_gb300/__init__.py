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
SELECTIVE_CKPT_CHUNK = 16


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
                "cla_scan_diag_bwd": ([P] * 9 + [I64, I64, I64, P, SZ, P], INT),
                "cla_scan_diag_fwd_noalloc": ([P, P, P, P, P, I64, I64, I64, P], INT),
                "cla_scan_diag_noalloc_check_status": ([P], INT),
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
                "cla_gla_workspace_size": ([I64] * 5 + [INT], SZ),
                "cla_gla_fwd": ([P] * 7 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_gla_bwd_workspace_size": ([I64] * 5 + [INT], SZ),
                "cla_gla_bwd": ([P] * 12 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_gla_ckpt_size": ([I64] * 5 + [INT], SZ),
                "cla_gla_fwd_ckpt": ([P] * 8 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_gla_bwd_ckpt": ([P] * 13 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_decay_total": ([P, P, I64, I64, I64, P], INT),
                "cla_delta_workspace_size": ([I64] * 5 + [INT], SZ),
                "cla_delta_fwd": ([P] * 8 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_delta_bwd_workspace_size": ([I64] * 5 + [INT], SZ),
                "cla_delta_bwd": ([P] * 14 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_delta_ckpt_size": ([I64] * 5 + [INT], SZ),
                "cla_delta_fwd_ckpt": ([P] * 9 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_delta_bwd_ckpt": ([P] * 15 + [I64] * 5 + [INT, P, SZ, P], INT),
                "cla_state_compose": ([P] * 4 + [I64] * 7 + [P], INT),
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


def _stream(stream, device=None):
    """The cudaStream_t to launch on: `stream` (a torch.cuda.Stream or a raw handle), else the
    current stream of `device` (else of the current device)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and isinstance(stream, torch.cuda.Stream) and stream.device != device:
        raise ValueError(f"stream belongs to {stream.device}, the tensors to {device}")
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims(t, n, name):
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")
    return tuple(t.shape)


class _T:
    """A tensor argument of an entry point (None stays NULL), checked by _launch for what the
    C ABI cannot check: dtype and shape (the sizes the call passes), then device and layout."""

    __slots__ = ("t", "dtype", "name", "shape")

    def __init__(self, t, dtype, name, shape=None):
        self.t, self.dtype, self.name, self.shape = t, dtype, name, shape

    def check_meta(self):
        t = self.t
        if self.dtype is not None and t.dtype != self.dtype:
            raise ValueError(f"{self.name} must be {self.dtype}, got {t.dtype}")
        if self.shape is not None and tuple(t.shape) != tuple(self.shape):
            raise ValueError(f"{self.name} must have shape {tuple(self.shape)}, got {tuple(t.shape)}")

    def check_place(self, device):
        t = self.t
        if not t.is_cuda:
            raise ValueError(f"{self.name} must be a CUDA tensor")
        if t.device != device:
            raise ValueError(f"{self.name} is on {t.device}, the call's first tensor on {device}")
        if not t.is_contiguous():
            raise ValueError(f"{self.name} must be contiguous")


def _nbytes(t):
    return t.numel() * t.element_size()


def _ws(nbytes, device, workspace, minimum=None):
    """A workspace of nbytes (allocated when not given); a given one needs at least `minimum`
    bytes (default nbytes) -- the entry points that take less than their size query's amount."""
    if workspace is None:
        workspace = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    need = nbytes if minimum is None else minimum
    if _nbytes(workspace) < need:
        raise ValueError(f"workspace of {_nbytes(workspace)} bytes < {need} needed")
    return workspace


def _out(t, shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device) if t is None else t


def _launch(fn, device, args, stream):
    """Calls entry point `fn` with the tensors' device current: `args` are plain values and _T
    tensor arguments, every one of which is checked (dtype and shape of all of them first)
    before its pointer is taken; raises ClaError on a non-OK status."""
    tensors = [a for a in args if isinstance(a, _T) and a.t is not None]
    for a in tensors:
        a.check_meta()
    for a in tensors:
        a.check_place(device)
    cargs = [(None if a.t is None else ctypes.c_void_p(a.t.data_ptr())) if isinstance(a, _T) else a for a in args]
    with torch.cuda.device(device):
        _check(fn, getattr(lib(), fn)(*cargs, _stream(stream, device)))


def check_status(workspace, stream=None) -> None:
    """Synchronise and raise if a kernel of the last call on `workspace` gave up a wait."""
    _launch("cla_check_status", workspace.device, (_T(workspace, None, "workspace"),), stream)


def selftest_wait_timeout(workspace, stream=None) -> None:
    """Launch the bounded-wait self-test on `workspace` (16-byte aligned, at least the
    256-byte workspace header)."""
    _launch("cla_selftest_wait_timeout", workspace.device,
            (_T(workspace, None, "workspace"), _nbytes(workspace)), stream)


# ---------------------------------------------------------------- diagonal scan
def scan_diag_workspace_size(B, T, D) -> int:
    return int(lib().cla_scan_diag_workspace_size(B, T, D))


def _scan_fwd(fn, a, b, h0, h, hT, workspace, stream, with_ws=True):
    B, T, D = _dims(a, 3, "a")
    dev = a.device
    f32 = torch.float32
    h = _out(h, (B, T, D), f32, dev)
    hT = _out(hT, (B, D), f32, dev)
    bt, bd = (B, T, D), (B, D)
    args = (_T(a, f32, "a", bt), _T(b, f32, "b", bt), _T(h0, f32, "h0", bd),
            _T(h, f32, "h", bt), _T(hT, f32, "hT", bd), B, T, D)
    if with_ws:
        ws = _ws(scan_diag_workspace_size(B, T, D), dev, workspace)
        args += (_T(ws, None, "workspace"), _nbytes(ws))
    _launch(fn, dev, args, stream)
    return h, hT


def scan_diag_fwd(a, b, h0=None, *, h=None, hT=None, workspace=None, stream=None):
    """h_t = a_t h_{t-1} + b_t over axis 1 of [B, T, D] (fp32); returns (h, hT)."""
    return _scan_fwd("cla_scan_diag_fwd", a, b, h0, h, hT, workspace, stream)


def scan_diag_fwd_blelloch(a, b, h0=None, *, h=None, hT=None, workspace=None, stream=None):
    """scan_diag_fwd with a Blelloch tree across the runs of a chunk (a measured
    alternative to Hillis-Steele); returns (h, hT)."""
    return _scan_fwd("cla_scan_diag_fwd_blelloch", a, b, h0, h, hT, workspace, stream)


def scan_diag_fwd_noalloc(a, b, h0=None, *, h=None, hT=None, stream=None):
    """scan_diag_fwd without a workspace: the library's static scratch array
    is used (limited size; overlapping calls race).  Returns (h, hT)."""
    return _scan_fwd("cla_scan_diag_fwd_noalloc", a, b, h0, h, hT, None, stream, with_ws=False)


def scan_diag_noalloc_check_status(stream=None, device=None) -> None:
    """Synchronise and raise if the last scan_diag_fwd_noalloc on `device` gave up a wait."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check("cla_scan_diag_noalloc_check_status",
               lib().cla_scan_diag_noalloc_check_status(_stream(stream, dev)))


def scan_diag_bwd(a, b, h0, h, dh, dhT=None, *, da=None, db=None, dh0=None, workspace=None, stream=None):
    """Adjoint of scan_diag_fwd; returns (da, db, dh0).  h: the forward's states, or None to
    recompute them from (a, b, h0) (then b is required; b may be None when h is given)."""
    B, T, D = _dims(a, 3, "a")
    dev = a.device
    f32 = torch.float32
    da = _out(da, (B, T, D), f32, dev)
    db = _out(db, (B, T, D), f32, dev)
    dh0 = _out(dh0, (B, D), f32, dev)
    ws = _ws(scan_diag_workspace_size(B, T, D), dev, workspace)
    bt, bd = (B, T, D), (B, D)
    _launch("cla_scan_diag_bwd", dev, (
        _T(a, f32, "a", bt), _T(b, f32, "b", bt), _T(h0, f32, "h0", bd), _T(h, f32, "h", bt),
        _T(dh, f32, "dh", bt), _T(dhT, f32, "dhT", bd), _T(da, f32, "da", bt),
        _T(db, f32, "db", bt), _T(dh0, f32, "dh0", bd), B, T, D,
        _T(ws, None, "workspace"), _nbytes(ws)), stream)
    return da, db, dh0


# ---------------------------------------------------------------- selective scan
def selective_scan_workspace_size(B, T, D, N) -> int:
    return int(lib().cla_selective_scan_workspace_size(B, T, D, N))


def selective_scan_ckpt_elems(B, T, D, N) -> int:
    return int(lib().cla_selective_scan_ckpt_elems(B, T, D, N))


def _sel_ckpt_arg(ckpt, B, T, D, N):
    if ckpt is None:
        return None
    need = selective_scan_ckpt_elems(B, T, D, N)
    if ckpt.numel() < need:
        raise ValueError(f"ckpt: need at least {need} fp32 values, got {ckpt.numel()}")
    return _T(ckpt, torch.float32, "ckpt")


def selective_scan_fwd(x, delta, A, Bm, Cm, h0=None, *, y=None, hT=None, ckpt=None, want_ckpt=True,
                       workspace=None, stream=None):
    """Selective scan forward; returns (y, hT, ckpt)."""
    B, T, D = _dims(x, 3, "x")
    N = _dims(A, 2, "A")[1]
    dev = x.device
    f32, bf16 = torch.float32, torch.bfloat16
    y = _out(y, (B, T, D), f32, dev)
    hT = _out(hT, (B, D, N), f32, dev)
    if ckpt is None and want_ckpt:
        ckpt = torch.empty(selective_scan_ckpt_elems(B, T, D, N), dtype=f32, device=dev)
    ws = _ws(selective_scan_workspace_size(B, T, D, N), dev, workspace)
    btd, btn, bdn = (B, T, D), (B, T, N), (B, D, N)
    _launch("cla_selective_scan_fwd", dev, (
        _T(x, bf16, "x", btd), _T(delta, f32, "delta", btd), _T(A, f32, "A", (D, N)),
        _T(Bm, bf16, "Bm", btn), _T(Cm, bf16, "Cm", btn), _T(h0, f32, "h0", bdn),
        _T(y, f32, "y", btd), _T(hT, f32, "hT", bdn), _sel_ckpt_arg(ckpt, B, T, D, N),
        B, T, D, N, _T(ws, None, "workspace"), _nbytes(ws)), stream)
    return y, hT, ckpt


def selective_scan_bwd(x, delta, A, Bm, Cm, h0, ckpt, dy, dhT=None, *, dx=None, ddelta=None, dA=None,
                       dB=None, dC=None, dh0=None, want_dA=True, want_dh0=True, workspace=None, stream=None):
    """Selective scan backward; returns (dx, ddelta, dA, dB, dC, dh0)."""
    B, T, D = _dims(x, 3, "x")
    N = _dims(A, 2, "A")[1]
    dev = x.device
    f32, bf16 = torch.float32, torch.bfloat16
    dx = _out(dx, (B, T, D), f32, dev)
    ddelta = _out(ddelta, (B, T, D), f32, dev)
    dA = _out(dA, (D, N), f32, dev) if (want_dA or dA is not None) else None
    dB = _out(dB, (B, T, N), f32, dev)
    dC = _out(dC, (B, T, N), f32, dev)
    dh0 = _out(dh0, (B, D, N), f32, dev) if (want_dh0 or dh0 is not None) else None
    ws = _ws(selective_scan_workspace_size(B, T, D, N), dev, workspace)
    btd, btn, bdn = (B, T, D), (B, T, N), (B, D, N)
    _launch("cla_selective_scan_bwd", dev, (
        _T(x, bf16, "x", btd), _T(delta, f32, "delta", btd), _T(A, f32, "A", (D, N)),
        _T(Bm, bf16, "Bm", btn), _T(Cm, bf16, "Cm", btn), _T(h0, f32, "h0", bdn),
        _sel_ckpt_arg(ckpt, B, T, D, N), _T(dy, f32, "dy", btd), _T(dhT, f32, "dhT", bdn),
        _T(dx, f32, "dx", btd), _T(ddelta, f32, "ddelta", btd), _T(dA, f32, "dA", (D, N)),
        _T(dB, f32, "dB", btn), _T(dC, f32, "dC", btn), _T(dh0, f32, "dh0", bdn),
        B, T, D, N, _T(ws, None, "workspace"), _nbytes(ws)), stream)
    return dx, ddelta, dA, dB, dC, dh0


# ---------------------------------------------------------------- chunkwise linear attention
def chunk_la_workspace_size(B, H, T, dim_k, dim_v, chunk) -> int:
    return int(lib().cla_chunk_la_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def chunk_la_ckpt_size(B, H, T, dim_k, dim_v, chunk) -> int:
    """Bytes of the segment-state checkpoint the forward can save for the backward."""
    return int(lib().cla_chunk_la_ckpt_size(B, H, T, dim_k, dim_v, int(chunk)))


def chunk_la_ckpt(q, v, *, chunk=64):
    """A device buffer (fp32) for the checkpoint of a forward on q [B, H, T, dk], v [.., dv]."""
    B, H, T, dk = _dims(q, 4, "q")
    n = chunk_la_ckpt_size(B, H, T, dk, v.shape[-1], chunk) // 4
    return torch.empty(max(n, 1), dtype=torch.float32, device=q.device)


def _ckpt_arg(ckpt, B, H, T, dk, dv, chunk):
    if ckpt is None:
        return None
    need = chunk_la_ckpt_size(B, H, T, dk, dv, chunk)
    if _nbytes(ckpt) < need:
        raise ValueError(f"ckpt: need at least {need} bytes, got {_nbytes(ckpt)}")
    return _T(ckpt, torch.float32, "ckpt")


def chunk_la_fwd(q, k, v, log_decay, S0=None, *, chunk=64, o=None, ST=None, ckpt=None, workspace=None,
                 stream=None):
    """Chunkwise decayed linear attention forward; returns (o, ST).  With ckpt (see
    chunk_la_ckpt) it also saves the state entering each segment for chunk_la_bwd."""
    B, H, T, dk = _dims(q, 4, "q")
    dv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    o = _out(o, (B, H, T, dv), f32, dev)
    ST = _out(ST, (B, H, dk, dv), f32, dev)
    ws = _ws(chunk_la_workspace_size(B, H, T, dk, dv, chunk), dev, workspace)
    tk, tv, st = (B, H, T, dk), (B, H, T, dv), (B, H, dk, dv)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", (B, H, T)), _T(S0, f32, "S0", st),
            _T(o, f32, "o", tv), _T(ST, f32, "ST", st))
    tail = (B, H, T, dk, dv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_chunk_la_fwd", dev, args + tail, stream)
    else:
        _launch("cla_chunk_la_fwd_ckpt", dev, args + (_ckpt_arg(ckpt, B, H, T, dk, dv, chunk),) + tail,
                stream)
    return o, ST


def chunk_la_bwd(q, k, v, log_decay, S0, dO, dST=None, *, chunk=64, dq=None, dk=None, dv=None,
                 dlog_decay=None, dS0=None, ckpt=None, workspace=None, stream=None):
    """Chunkwise decayed linear attention backward; returns (dq, dk, dv, dlog_decay, dS0).  ckpt:
    the checkpoint a chunk_la_fwd on the same inputs saved (its states are then not rebuilt)."""
    B, H, T, dkk = _dims(q, 4, "q")
    dvv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    dq = _out(dq, (B, H, T, dkk), f32, dev)
    dk = _out(dk, (B, H, T, dkk), f32, dev)
    dv = _out(dv, (B, H, T, dvv), f32, dev)
    dlog_decay = _out(dlog_decay, (B, H, T), f32, dev)
    dS0 = _out(dS0, (B, H, dkk, dvv), f32, dev)
    ws = _ws(chunk_la_workspace_size(B, H, T, dkk, dvv, chunk), dev, workspace)
    tk, tv, st, bht = (B, H, T, dkk), (B, H, T, dvv), (B, H, dkk, dvv), (B, H, T)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", bht), _T(S0, f32, "S0", st),
            _T(dO, bf16, "dO", tv), _T(dST, f32, "dST", st), _T(dq, f32, "dq", tk),
            _T(dk, f32, "dk", tk), _T(dv, f32, "dv", tv),
            _T(dlog_decay, f32, "dlog_decay", bht), _T(dS0, f32, "dS0", st))
    tail = (B, H, T, dkk, dvv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_chunk_la_bwd", dev, args + tail, stream)
    else:
        _launch("cla_chunk_la_bwd_ckpt", dev, args + (_ckpt_arg(ckpt, B, H, T, dkk, dvv, chunk),) + tail,
                stream)
    return dq, dk, dv, dlog_decay, dS0


# ---------------------------------------------------------------- gated linear attention
def gla_workspace_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    return int(lib().cla_gla_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def gla_ckpt_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    """Bytes of the segment-state checkpoint the GLA forward can save for the backward."""
    return int(lib().cla_gla_ckpt_size(B, H, T, dim_k, dim_v, int(chunk)))


def gla_ckpt(q, v, *, chunk=64):
    """A device buffer (fp32) for the checkpoint of a gla_fwd on q [B, H, T, dk], v [.., dv]."""
    B, H, T, dk = _dims(q, 4, "q")
    n = gla_ckpt_size(B, H, T, dk, v.shape[-1], chunk) // 4
    return torch.empty(max(n, 1), dtype=torch.float32, device=q.device)


def _gla_ckpt_arg(ckpt, B, H, T, dk, dv, chunk):
    need = gla_ckpt_size(B, H, T, dk, dv, chunk)
    if _nbytes(ckpt) < need:
        raise ValueError(f"ckpt: need at least {need} bytes, got {_nbytes(ckpt)}")
    return _T(ckpt, torch.float32, "ckpt")


def gla_fwd(q, k, v, log_decay, S0=None, *, chunk=64, o=None, ST=None, ckpt=None, workspace=None, stream=None):
    """Gated linear attention forward (one decay per key dimension: log_decay [B, H, T, dk]);
    returns (o, ST).  check_status(workspace) reports decays outside the kernel's range.  With
    ckpt (see gla_ckpt) it also saves the state entering every segment for gla_bwd."""
    B, H, T, dk = _dims(q, 4, "q")
    dv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    o = _out(o, (B, H, T, dv), f32, dev)
    ST = _out(ST, (B, H, dk, dv), f32, dev)
    ws = _ws(gla_workspace_size(B, H, T, dk, dv, chunk), dev, workspace)
    tk, tv, st = (B, H, T, dk), (B, H, T, dv), (B, H, dk, dv)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", tk), _T(S0, f32, "S0", st),
            _T(o, f32, "o", tv), _T(ST, f32, "ST", st))
    tail = (B, H, T, dk, dv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_gla_fwd", dev, args + tail, stream)
    else:
        _launch("cla_gla_fwd_ckpt", dev, args + (_gla_ckpt_arg(ckpt, B, H, T, dk, dv, chunk),) + tail, stream)
    return o, ST


def gla_bwd_workspace_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    return int(lib().cla_gla_bwd_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def gla_bwd(q, k, v, log_decay, S0, dO, dST=None, *, chunk=64, dq=None, dk=None, dv=None, dlog_decay=None,
            dS0=None, ckpt=None, workspace=None, stream=None):
    """Gated linear attention backward; returns (dq, dk, dv, dlog_decay [B, H, T, dk], dS0).  ckpt:
    the checkpoint a gla_fwd(..., ckpt=) on the same inputs saved (its dq traversal then starts
    from it)."""
    B, H, T, dkk = _dims(q, 4, "q")
    dvv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    dq = _out(dq, (B, H, T, dkk), f32, dev)
    dk = _out(dk, (B, H, T, dkk), f32, dev)
    dv = _out(dv, (B, H, T, dvv), f32, dev)
    dlog_decay = _out(dlog_decay, (B, H, T, dkk), f32, dev)
    dS0 = _out(dS0, (B, H, dkk, dvv), f32, dev)
    ws = _ws(gla_bwd_workspace_size(B, H, T, dkk, dvv, chunk), dev, workspace)
    tk, tv, st = (B, H, T, dkk), (B, H, T, dvv), (B, H, dkk, dvv)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", tk), _T(S0, f32, "S0", st), _T(dO, bf16, "dO", tv),
            _T(dST, f32, "dST", st), _T(dq, f32, "dq", tk), _T(dk, f32, "dk", tk), _T(dv, f32, "dv", tv),
            _T(dlog_decay, f32, "dlog_decay", tk), _T(dS0, f32, "dS0", st))
    tail = (B, H, T, dkk, dvv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_gla_bwd", dev, args + tail, stream)
    else:
        _launch("cla_gla_bwd_ckpt", dev, args + (_gla_ckpt_arg(ckpt, B, H, T, dkk, dvv, chunk),) + tail, stream)
    return dq, dk, dv, dlog_decay, dS0


# ---------------------------------------------------------------- state passing between slices
def decay_total(log_decay, *, alpha=None, stream=None):
    """exp of the sum over the slice of log_decay: [B, H, T] -> [B, H] (one decay per head) or
    [B, H, T, dk] -> [B, H, dk] (gated)."""
    if log_decay.dim() == 3:
        B, H, T = log_decay.shape
        A, shape = 1, (B, H)
    else:
        B, H, T, A = _dims(log_decay, 4, "log_decay")
        shape = (B, H, A)
    dev = log_decay.device
    alpha = _out(alpha, shape, torch.float32, dev)
    _launch("cla_decay_total", dev, (_T(log_decay, torch.float32, "log_decay", tuple(log_decay.shape)),
                                     _T(alpha, torch.float32, "alpha", shape), B * H, T, A), stream)
    return alpha


def state_compose(alphas, dSs, edge, first, count, step, *, out=None, stream=None):
    """Fold acc <- diag(alpha_j) acc + dS_j over j = first + c * step (c < count) from edge.
    alphas [P, B, H] or [P, B, H, dk]; dSs [P, B, H, dk, dv]; edge [B, H, dk, dv] or None."""
    P, B, H, dk, dv = _dims(dSs, 5, "dSs")
    A = 1 if alphas.dim() == 3 else alphas.shape[3]
    dev = dSs.device
    out = _out(out, (B, H, dk, dv), torch.float32, dev)
    st = (B, H, dk, dv)
    _launch("cla_state_compose", dev, (
        _T(alphas, torch.float32, "alphas", (P, B, H) if A == 1 else (P, B, H, A)),
        _T(dSs, torch.float32, "dSs", (P, B, H, dk, dv)), _T(edge, torch.float32, "edge", st),
        _T(out, torch.float32, "out", st), P, B * H, dk * dv, A, int(first), int(count), int(step)), stream)
    return out


# ---------------------------------------------------------------- delta rule (Gated DeltaNet)
def delta_workspace_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    return int(lib().cla_delta_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def delta_ckpt_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    """Bytes of the checkpoint (the state entering every chunk) the forward can save for the backward."""
    return int(lib().cla_delta_ckpt_size(B, H, T, dim_k, dim_v, int(chunk)))


def delta_ckpt(q, v, *, chunk=64):
    """A device buffer (fp32) for the checkpoint of a delta_fwd on q [B, H, T, dk], v [.., dv]."""
    B, H, T, dk = _dims(q, 4, "q")
    n = delta_ckpt_size(B, H, T, dk, v.shape[-1], chunk) // 4
    return torch.empty(max(n, 1), dtype=torch.float32, device=q.device)


def _delta_ckpt_arg(ckpt, B, H, T, dk, dv, chunk):
    need = delta_ckpt_size(B, H, T, dk, dv, chunk)
    if _nbytes(ckpt) < need:
        raise ValueError(f"ckpt: need at least {need} bytes, got {_nbytes(ckpt)}")
    return _T(ckpt, torch.float32, "ckpt")


def delta_fwd(q, k, v, log_decay, beta, S0=None, *, chunk=64, o=None, ST=None, ckpt=None, workspace=None,
              stream=None):
    """Delta rule with a decay per head: S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
    o_t = q_t S_t; log_decay, beta [B, H, T].  Returns (o, ST).  With ckpt (see delta_ckpt) it also
    saves the state entering every chunk for delta_bwd.  A given workspace needs 256 bytes; the
    size query's amount lets the chunks' (I + A)^-1 be formed beforehand, all at once."""
    B, H, T, dk = _dims(q, 4, "q")
    dv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    o = _out(o, (B, H, T, dv), f32, dev)
    ST = _out(ST, (B, H, dk, dv), f32, dev)
    ws = _ws(delta_workspace_size(B, H, T, dk, dv, chunk), dev, workspace, minimum=256)
    tk, tv, st, bht = (B, H, T, dk), (B, H, T, dv), (B, H, dk, dv), (B, H, T)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", bht), _T(beta, f32, "beta", bht), _T(S0, f32, "S0", st),
            _T(o, f32, "o", tv), _T(ST, f32, "ST", st))
    tail = (B, H, T, dk, dv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_delta_fwd", dev, args + tail, stream)
    else:
        _launch("cla_delta_fwd_ckpt", dev, args + (_delta_ckpt_arg(ckpt, B, H, T, dk, dv, chunk),) + tail, stream)
    return o, ST


def delta_bwd_workspace_size(B, H, T, dim_k, dim_v, chunk=64) -> int:
    return int(lib().cla_delta_bwd_workspace_size(B, H, T, dim_k, dim_v, int(chunk)))


def delta_bwd(q, k, v, log_decay, beta, S0, dO, dST=None, *, chunk=64, dq=None, dk=None, dv=None,
              dlog_decay=None, dbeta=None, dS0=None, ckpt=None, workspace=None, stream=None):
    """Adjoint of delta_fwd (dO bf16 [B, H, T, dv]); returns (dq, dk, dv, dlog_decay, dbeta, dS0).  ckpt:
    the checkpoint a delta_fwd on the same inputs saved (the states are then not recomputed)."""
    B, H, T, dkk = _dims(q, 4, "q")
    dvv = _dims(v, 4, "v")[3]
    dev = q.device
    f32, bf16 = torch.float32, torch.bfloat16
    dq = _out(dq, (B, H, T, dkk), f32, dev)
    dk = _out(dk, (B, H, T, dkk), f32, dev)
    dv = _out(dv, (B, H, T, dvv), f32, dev)
    dlog_decay = _out(dlog_decay, (B, H, T), f32, dev)
    dbeta = _out(dbeta, (B, H, T), f32, dev)
    dS0 = _out(dS0, (B, H, dkk, dvv), f32, dev)
    need = delta_bwd_workspace_size(B, H, T, dkk, dvv, chunk)
    if ckpt is not None:  # no states in the workspace: the header and the partials only
        need = max(need - delta_ckpt_size(B, H, T, dkk, dvv, chunk), 256)
    ws = _ws(need, dev, workspace)
    tk, tv, st, bht = (B, H, T, dkk), (B, H, T, dvv), (B, H, dkk, dvv), (B, H, T)
    args = (_T(q, bf16, "q", tk), _T(k, bf16, "k", tk), _T(v, bf16, "v", tv),
            _T(log_decay, f32, "log_decay", bht), _T(beta, f32, "beta", bht), _T(S0, f32, "S0", st),
            _T(dO, bf16, "dO", tv), _T(dST, f32, "dST", st), _T(dq, f32, "dq", tk), _T(dk, f32, "dk", tk),
            _T(dv, f32, "dv", tv), _T(dlog_decay, f32, "dlog_decay", bht), _T(dbeta, f32, "dbeta", bht),
            _T(dS0, f32, "dS0", st))
    tail = (B, H, T, dkk, dvv, int(chunk), _T(ws, None, "workspace"), _nbytes(ws))
    if ckpt is None:
        _launch("cla_delta_bwd", dev, args + tail, stream)
    else:
        _launch("cla_delta_bwd_ckpt", dev, args + (_delta_ckpt_arg(ckpt, B, H, T, dkk, dvv, chunk),) + tail, stream)
    return dq, dk, dv, dlog_decay, dbeta, dS0
