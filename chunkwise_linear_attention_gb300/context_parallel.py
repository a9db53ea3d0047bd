"""Context parallelism: one sequence split across devices by state passing.

"Parallel Scan", "Splitting one sequence across devices": every device holds a
contiguous slice of the sequence.  It runs its slice from a zero state, which
gives the slice's affine pair (alpha_p, dS_p) -- the slice's total decay and
its own contribution to the state at its end.  The devices exchange the pairs
(one all-gather of P small pairs), each composes the pairs before it under
the combine (a1, b1) . (a2, b2) = (a1 a2, a2 b1 + b2) onto the initial state,
and reruns its slice from that true incoming state.  Only the composition
waits on other devices; the local work is parallel.  The backward does the
same from the right on the adjoint state: slice p's gradient on its own
initial state is affine in the gradient on its final state,
dS_start = diag(alpha_p) dS_end + dD_p, so the pairs (alpha_p, dD_p) compose
from the last slice to the first, starting from the upstream dS_T.

The functions here are the host-side schedule, SPMD: every rank calls them on
its own slice.  Each step runs in the library's kernels -- the chunkwise
forward and backward (scalar decay: chunk_la_*; one decay per key dimension:
gla_*), decay_total and state_compose -- and the exchange is
torch.distributed.all_gather.  The phase functions (local_pair_fwd,
incoming_state, ...) are exposed so that a schedule can also be stepped
through for several slices in one process.

Work: two passes of the forward (the first only for its final state) and two
of the backward (the first only for its initial-state gradient) per slice.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional


@dataclass
class Ops:
    """The four local steps of the schedule.  `cuda_ops` gives the library's."""

    fwd: Callable      # (q, k, v, log_a, S0) -> (o, S_T)
    bwd: Callable      # (q, k, v, log_a, S0, dO, dST) -> (dq, dk, dv, dlog_a, dS0)
    decay_total: Callable  # log_a -> alpha ([B, H] or [B, H, dk])
    compose: Callable      # (alphas, dSs, edge, first, count, step) -> state


def cuda_ops(kind: str = "la", chunk: int = 64) -> Ops:
    """The library's kernels: kind "la" (one decay per head, chunk 64 or 128) or "gla" (one decay
    per key dimension, chunk 64)."""
    import chunkwise_linear_attention_gb300 as cla

    if kind == "la":
        fwd = lambda q, k, v, la, S0: cla.chunk_la_fwd(q, k, v, la, S0, chunk=chunk)
        bwd = lambda q, k, v, la, S0, dO, dST: cla.chunk_la_bwd(q, k, v, la, S0, dO, dST, chunk=chunk)
    elif kind == "gla":
        fwd = lambda q, k, v, la, S0: cla.gla_fwd(q, k, v, la, S0, chunk=chunk)
        bwd = lambda q, k, v, la, S0, dO, dST: cla.gla_bwd(q, k, v, la, S0, dO, dST, chunk=chunk)
    else:
        raise ValueError(f"kind must be 'la' or 'gla', got {kind!r}")
    return Ops(fwd=fwd, bwd=bwd, decay_total=cla.decay_total, compose=cla.state_compose)


# ---------------------------------------------------------------- phases
def local_pair_fwd(ops: Ops, q, k, v, log_a):
    """The slice's pair: its total decay and its final state from a zero initial state."""
    _, dS = ops.fwd(q, k, v, log_a, None)
    return ops.decay_total(log_a), dS


def incoming_state(ops: Ops, alphas, dSs, rank: int, S0):
    """The state entering slice `rank`: pairs 0..rank-1 folded onto S0."""
    return ops.compose(alphas, dSs, S0, 0, rank, 1)


def local_pair_bwd(ops: Ops, q, k, v, log_a, S_in, dO):
    """The slice's backward pair part: the gradient on its initial state with no upstream
    gradient on its final state (the decay part is the forward's alpha)."""
    return ops.bwd(q, k, v, log_a, S_in, dO, None)[4]


def upstream_state(ops: Ops, alphas, dDs, rank: int, world: int, dST):
    """The gradient on slice `rank`'s final state: pairs world-1 down to rank+1 folded onto dST."""
    return ops.compose(alphas, dDs, dST, world - 1, world - 1 - rank, -1)


# ---------------------------------------------------------------- SPMD entry points
def _gather(x, group):
    import torch
    import torch.distributed as dist

    parts = [torch.empty_like(x) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, x.contiguous(), group=group)
    return torch.stack(parts)


def _rank_world(group):
    import torch.distributed as dist

    return dist.get_rank(group), dist.get_world_size(group)


def forward(q, k, v, log_a, S0=None, *, ops: Optional[Ops] = None, group=None):
    """This rank's slice of the sequence -> (o, S_T, S_in, alpha).  S0 is the sequence's initial
    state (used by the composition on every rank); S_T is the sequence's final state on the last
    rank (this slice's final state elsewhere); keep S_in and alpha for `backward`."""
    ops = ops or cuda_ops("gla" if log_a.dim() == 4 else "la")
    rank, _ = _rank_world(group)
    alpha, dS = local_pair_fwd(ops, q, k, v, log_a)
    alphas, dSs = _gather(alpha, group), _gather(dS, group)
    S_in = incoming_state(ops, alphas, dSs, rank, S0)
    o, ST = ops.fwd(q, k, v, log_a, S_in)
    return o, ST, S_in, alpha


def backward(q, k, v, log_a, S_in, alpha, dO, dST=None, *, ops: Optional[Ops] = None, group=None):
    """Gradients of this rank's slice -> (dq, dk, dv, dlog_a, dS0); dS0 is the gradient on the
    sequence's initial state on rank 0 (on this slice's incoming state elsewhere).  dST: the
    upstream gradient on the sequence's final state (the same on every rank, or None)."""
    ops = ops or cuda_ops("gla" if log_a.dim() == 4 else "la")
    rank, world = _rank_world(group)
    dD = local_pair_bwd(ops, q, k, v, log_a, S_in, dO)
    alphas, dDs = _gather(alpha, group), _gather(dD, group)
    dS_end = upstream_state(ops, alphas, dDs, rank, world, dST)
    return ops.bwd(q, k, v, log_a, S_in, dO, dS_end)
