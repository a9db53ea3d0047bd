"""Float64 CPU oracle for the linear-recurrence hot path.

TEST INFRASTRUCTURE ONLY.  The library never imports this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.
It shares no code with the CUDA path: the arithmetic lives in ``oracle.c``
(plain C, float64 loops) and this module only compiles it, converts arrays to
float64 and calls it.

Each function states the passage it follows in the C source; the summary:

* ``scan_diag_fwd`` / ``scan_diag_bwd`` -- "Parallel Scan", "The scan for one
  number of state" and "The backward pass is a scan in reverse".
* ``selective_fwd`` / ``selective_bwd`` -- the same recurrence per (channel,
  state entry) with a = exp(Delta A), b = Delta B x, y = C . h ("Parallel
  Scan", "When a scan is the wrong tool", Mamba's selective decay).
* ``la_fwd`` / ``la_bwd`` -- decayed linear attention as its per-token
  recurrence and adjoint ("Parallel Scan", "The chunkwise algorithm" and "The
  backward pass of linear attention"; "Lightning Attention-2", eqs. 4, 11-12).
* ``la_dlog_closed_form`` -- the closed-form decay gradient of "The backward
  pass of linear attention".
* ``delta_fwd`` / ``delta_bwd`` -- the delta rule with a decay per head
  (Gated DeltaNet: "Parallel Scan", "What one combine costs", the identity
  minus a rank-one transition that overwrites what a key stores, and "At
  real scale"), S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
  and its adjoint.
* ``decay_total`` / ``state_compose`` -- state passing between slices of one
  sequence ("Parallel Scan", "Splitting one sequence across devices"): a
  slice's total decay, and the fold of slice pairs under the combine.
* ``gla_fwd`` / ``gla_bwd`` / ``gla_dlog_closed_form`` -- gated linear
  attention, one decay per key dimension ("Parallel Scan", "What one combine
  costs" and "The chunkwise algorithm": S_t = G_t (.) S_{t-1} + k_t^T v_t), its
  adjoint, and the per-dimension closed-form decay gradient (Yang et al.'s, as
  "The backward pass of linear attention" cites it).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_scan_diag_fwd.argtypes = [P, P, P, P, P, I, I, I]
            lib.oracle_scan_diag_bwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I]
            lib.oracle_selective_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I]
            lib.oracle_selective_bwd.argtypes = [P] * 14 + [I, I, I, I]
            lib.oracle_la_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
            lib.oracle_la_bwd.argtypes = [P] * 12 + [I, I, I, I, I]
            lib.oracle_la_dlog_closed_form.argtypes = [P] * 7 + [I, I, I, I, I]
            lib.oracle_gla_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
            lib.oracle_gla_bwd.argtypes = [P] * 12 + [I, I, I, I, I]
            lib.oracle_gla_dlog_closed_form.argtypes = [P] * 7 + [I, I, I, I, I]
            lib.oracle_decay_total.argtypes = [P, P, I, I, I]
            lib.oracle_delta_fwd.argtypes = [P] * 8 + [I] * 5
            lib.oracle_delta_bwd.argtypes = [P] * 14 + [I] * 5
            lib.oracle_state_compose.argtypes = [P, P, P, P] + [I] * 7
            for fn in ("oracle_scan_diag_fwd", "oracle_scan_diag_bwd", "oracle_selective_fwd",
                       "oracle_selective_bwd", "oracle_la_fwd", "oracle_la_bwd",
                       "oracle_la_dlog_closed_form", "oracle_gla_fwd", "oracle_gla_bwd",
                       "oracle_gla_dlog_closed_form", "oracle_decay_total", "oracle_state_compose",
                       "oracle_delta_fwd", "oracle_delta_bwd"):
                getattr(lib, fn).restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: take its values exactly
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def scan_diag_fwd(a, b, h0=None):
    """h_t = a_t h_{t-1} + b_t over axis 1 of [B, T, D]; returns (h, h_T)."""
    a, b, h0 = _f64(a), _f64(b), _f64(h0)
    B, T, D = a.shape
    h = np.empty_like(a)
    hT = np.empty((B, D))
    _load().oracle_scan_diag_fwd(_p(a), _p(b), _p(h0), _p(h), _p(hT), B, T, D)
    return h, hT


def scan_diag_bwd(a, b, h0, g, dhT=None):
    """Adjoint of scan_diag_fwd; returns (da, db, dh0)."""
    a, b, h0, g, dhT = _f64(a), _f64(b), _f64(h0), _f64(g), _f64(dhT)
    B, T, D = a.shape
    da = np.empty_like(a)
    db = np.empty_like(a)
    dh0 = np.empty((B, D))
    _load().oracle_scan_diag_bwd(_p(a), _p(b), _p(h0), _p(g), _p(dhT), _p(da), _p(db), _p(dh0), B, T, D)
    return da, db, dh0


def selective_fwd(x, delta, A, Bm, Cm, h0=None):
    """Selective scan forward; returns (y [B,T,D], h_T [B,D,N])."""
    x, delta, A, Bm, Cm, h0 = map(_f64, (x, delta, A, Bm, Cm, h0))
    B, T, D = x.shape
    N = A.shape[1]
    y = np.empty((B, T, D))
    hT = np.empty((B, D, N))
    _load().oracle_selective_fwd(_p(x), _p(delta), _p(A), _p(Bm), _p(Cm), _p(h0), _p(y), _p(hT), B, T, D, N)
    return y, hT


def selective_bwd(x, delta, A, Bm, Cm, h0, dy, dhT=None):
    """Selective scan backward; returns (dx, ddelta, dA, dB, dC, dh0)."""
    x, delta, A, Bm, Cm, h0, dy, dhT = map(_f64, (x, delta, A, Bm, Cm, h0, dy, dhT))
    B, T, D = x.shape
    N = A.shape[1]
    dx = np.empty((B, T, D))
    dd = np.empty((B, T, D))
    dA = np.empty((D, N))
    dB = np.empty((B, T, N))
    dC = np.empty((B, T, N))
    dh0 = np.empty((B, D, N))
    _load().oracle_selective_bwd(_p(x), _p(delta), _p(A), _p(Bm), _p(Cm), _p(h0), _p(dy), _p(dhT),
                                 _p(dx), _p(dd), _p(dA), _p(dB), _p(dC), _p(dh0), B, T, D, N)
    return dx, dd, dA, dB, dC, dh0


def la_fwd(q, k, v, log_a, S0=None):
    """Decayed linear attention forward; q,k [B,H,T,dk], v [B,H,T,dv],
    log_a [B,H,T], S0 [B,H,dk,dv]; returns (o [B,H,T,dv], S_T)."""
    q, k, v, log_a, S0 = map(_f64, (q, k, v, log_a, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    ST = np.empty((B, H, dk, dv))
    _load().oracle_la_fwd(_p(q), _p(k), _p(v), _p(log_a), _p(S0), _p(o), _p(ST), B, H, T, dk, dv)
    return o, ST


def la_bwd(q, k, v, log_a, S0, dO, dST=None):
    """Decayed linear attention backward by the adjoint definition;
    returns (dq, dk, dv, dlog_a, dS0)."""
    q, k, v, log_a, S0, dO, dST = map(_f64, (q, k, v, log_a, S0, dO, dST))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dq = np.empty((B, H, T, dk))
    dkk = np.empty((B, H, T, dk))
    dvv = np.empty((B, H, T, dv))
    dl = np.empty((B, H, T))
    dS0 = np.empty((B, H, dk, dv))
    _load().oracle_la_bwd(_p(q), _p(k), _p(v), _p(log_a), _p(S0), _p(dO), _p(dST),
                          _p(dq), _p(dkk), _p(dvv), _p(dl), _p(dS0), B, H, T, dk, dv)
    return dq, dkk, dvv, dl, dS0


def la_dlog_closed_form(q, k, dq, dk, dST=None, ST=None):
    """dL/dlog a_u = sum_{t>=u} q_t.dq_t - sum_{s>=u} k_s.dk_s (+ <dS_T, S_T>)."""
    q, k, dq, dk, dST, ST = map(_f64, (q, k, dq, dk, dST, ST))
    B, H, T, dkk = q.shape
    dv = ST.shape[-1] if ST is not None else dkk
    out = np.empty((B, H, T))
    _load().oracle_la_dlog_closed_form(_p(q), _p(k), _p(dq), _p(dk), _p(dST), _p(ST), _p(out),
                                       B, H, T, dkk, dv)
    return out


def gla_fwd(q, k, v, log_a, S0=None):
    """Gated linear attention forward, one decay per key dimension: q, k, log_a
    [B,H,T,dk], v [B,H,T,dv], S0 [B,H,dk,dv]; returns (o [B,H,T,dv], S_T)."""
    q, k, v, log_a, S0 = map(_f64, (q, k, v, log_a, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    ST = np.empty((B, H, dk, dv))
    _load().oracle_gla_fwd(_p(q), _p(k), _p(v), _p(log_a), _p(S0), _p(o), _p(ST), B, H, T, dk, dv)
    return o, ST


def gla_bwd(q, k, v, log_a, S0, dO, dST=None):
    """Gated linear attention backward by the adjoint definition; returns
    (dq, dk, dv, dlog_a [B,H,T,dk], dS0)."""
    q, k, v, log_a, S0, dO, dST = map(_f64, (q, k, v, log_a, S0, dO, dST))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dq = np.empty((B, H, T, dk))
    dkk = np.empty((B, H, T, dk))
    dvv = np.empty((B, H, T, dv))
    dl = np.empty((B, H, T, dk))
    dS0 = np.empty((B, H, dk, dv))
    _load().oracle_gla_bwd(_p(q), _p(k), _p(v), _p(log_a), _p(S0), _p(dO), _p(dST),
                           _p(dq), _p(dkk), _p(dvv), _p(dl), _p(dS0), B, H, T, dk, dv)
    return dq, dkk, dvv, dl, dS0


def gla_dlog_closed_form(q, k, dq, dk, dST=None, ST=None):
    """dL/dlog a_u[i] = sum_{t>=u} q_t[i] dq_t[i] - sum_{s>=u} k_s[i] dk_s[i]
    (+ sum_j dS_T[i][j] S_T[i][j])."""
    q, k, dq, dk, dST, ST = map(_f64, (q, k, dq, dk, dST, ST))
    B, H, T, dkk = q.shape
    dv = ST.shape[-1] if ST is not None else dkk
    out = np.empty((B, H, T, dkk))
    _load().oracle_gla_dlog_closed_form(_p(q), _p(k), _p(dq), _p(dk), _p(dST), _p(ST), _p(out),
                                        B, H, T, dkk, dv)
    return out


def decay_total(log_decay):
    """alpha = exp(sum over axis -2 of log_decay) for log_decay [BH..., T, A] given as
    [BH, T, A] (A = 1 for one decay per head); returns [BH, A]."""
    ld = _f64(log_decay)
    BH, T, A = ld.shape
    out = np.empty((BH, A))
    _load().oracle_decay_total(_p(ld), _p(out), BH, T, A)
    return out


def state_compose(alpha, dS, edge, first, count, step):
    """Fold of pairs j = first + c * step (c < count): acc <- alpha_j acc + dS_j from acc = edge.
    alpha [P, BH, A], dS [P, BH, n], edge [BH, n] or None; returns [BH, n]."""
    alpha, dS, edge = _f64(alpha), _f64(dS), _f64(edge)
    P, BH, n = dS.shape
    A = alpha.shape[2]
    out = np.empty((BH, n))
    _load().oracle_state_compose(_p(alpha), _p(dS), _p(edge), _p(out), P, BH, n, A, first, count, step)
    return out


def delta_fwd(q, k, v, log_a, beta, S0=None):
    """Delta rule with a decay per head: q, k [B,H,T,dk], v [B,H,T,dv], log_a, beta [B,H,T],
    S0 [B,H,dk,dv]; returns (o [B,H,T,dv], S_T)."""
    q, k, v, log_a, beta, S0 = map(_f64, (q, k, v, log_a, beta, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    ST = np.empty((B, H, dk, dv))
    _load().oracle_delta_fwd(_p(q), _p(k), _p(v), _p(log_a), _p(beta), _p(S0), _p(o), _p(ST), B, H, T, dk, dv)
    return o, ST


def delta_bwd(q, k, v, log_a, beta, S0, dO, dST=None):
    """Adjoint of delta_fwd; returns (dq, dk, dv, dlog_a, dbeta, dS0)."""
    q, k, v, log_a, beta, S0, dO, dST = map(_f64, (q, k, v, log_a, beta, S0, dO, dST))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dq = np.empty((B, H, T, dk))
    dkk = np.empty((B, H, T, dk))
    dvv = np.empty((B, H, T, dv))
    dl = np.empty((B, H, T))
    db = np.empty((B, H, T))
    dS0 = np.empty((B, H, dk, dv))
    _load().oracle_delta_bwd(_p(q), _p(k), _p(v), _p(log_a), _p(beta), _p(S0), _p(dO), _p(dST), _p(dq), _p(dkk),
                             _p(dvv), _p(dl), _p(db), _p(dS0), B, H, T, dk, dv)
    return dq, dkk, dvv, dl, db, dS0
