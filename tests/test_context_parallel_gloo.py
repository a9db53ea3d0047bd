"""Context parallelism by state passing ("Parallel Scan", "Splitting one
sequence across devices") on CPU: 2 and 3 gloo ranks each hold a contiguous,
unequal slice of one sequence and run the library's SPMD schedule
(chunkwise_linear_attention_gb300.context_parallel: local pair, all-gather,
composition, rerun; the adjoint from the right in the backward) with the
float64 oracle as each rank's local step.  Every rank's outputs and
gradients must equal the oracle's on the whole sequence, sliced -- for one
decay per head and for one decay per key dimension."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_ops(kind):
    import torch

    import oracle
    from chunkwise_linear_attention_gb300.context_parallel import Ops

    t = lambda x: torch.from_numpy(x)
    if kind == "la":
        fwd = lambda q, k, v, la, S0: tuple(map(t, oracle.la_fwd(q, k, v, la, S0)))
        bwd = lambda q, k, v, la, S0, dO, dST: tuple(map(t, oracle.la_bwd(q, k, v, la, S0, dO, dST)))
    else:
        fwd = lambda q, k, v, la, S0: tuple(map(t, oracle.gla_fwd(q, k, v, la, S0)))
        bwd = lambda q, k, v, la, S0, dO, dST: tuple(map(t, oracle.gla_bwd(q, k, v, la, S0, dO, dST)))

    def decay_total(la):
        B, H, T = la.shape[:3]
        A = 1 if la.dim() == 3 else la.shape[3]
        a = t(oracle.decay_total(la.reshape(B * H, T, A)))
        return a.reshape(B, H) if la.dim() == 3 else a.reshape(B, H, A)

    def compose(alphas, dSs, edge, first, count, step):
        P, B, H, dk, dv = dSs.shape
        A = 1 if alphas.dim() == 3 else alphas.shape[3]
        out = oracle.state_compose(alphas.reshape(P, B * H, A), dSs.reshape(P, B * H, dk * dv),
                                   None if edge is None else edge.reshape(B * H, dk * dv), first, count, step)
        return t(out).reshape(B, H, dk, dv)

    return Ops(fwd=fwd, bwd=bwd, decay_total=decay_total, compose=compose)


def problem(kind, T=100, dk=8, dv=6):
    import numpy as np
    import torch

    import workloads

    inp = workloads.make("la_long" if kind == "la" else "gla", B=1, H=2, T=T, dk=dk, dv=dv)
    d = {k: (None if v is None else v.double()) for k, v in inp.items()}
    rng = np.random.default_rng(7)
    d["dST"] = torch.from_numpy(rng.normal(0, 0.3, (1, 2, dk, dv)))
    return d


def _rank(rank, world, port, kind, bounds, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from chunkwise_linear_attention_gb300 import context_parallel as cp

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = problem(kind)
        lo, hi = bounds[rank], bounds[rank + 1]
        sl = {k: (v[:, :, lo:hi] if k in ("q", "k", "v", "log_a", "dO") else v) for k, v in d.items()}
        ops = oracle_ops(kind)
        o, ST, S_in, alpha = cp.forward(sl["q"], sl["k"], sl["v"], sl["log_a"], d["S0"], ops=ops)
        g = cp.backward(sl["q"], sl["k"], sl["v"], sl["log_a"], S_in, alpha, sl["dO"], d["dST"], ops=ops)
        fwd = oracle.la_fwd if kind == "la" else oracle.gla_fwd
        bwd = oracle.la_bwd if kind == "la" else oracle.gla_bwd
        ro, rST = fwd(d["q"], d["k"], d["v"], d["log_a"], d["S0"])
        rg = bwd(d["q"], d["k"], d["v"], d["log_a"], d["S0"], d["dO"], d["dST"])
        import numpy as np

        def close(x, r):
            x = x.numpy()
            return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-300))

        errs = {"o": close(o, ro[:, :, lo:hi])}
        for name, x, r in zip(("dq", "dk", "dv", "dlog_a"), g[:4], rg[:4]):
            errs[name] = close(x, r[:, :, lo:hi])
        if rank == world - 1:
            errs["S_T"] = close(ST, rST)
        if rank == 0:
            errs["dS0"] = close(g[4], rg[4])
        q.put((rank, errs))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kind", ["la", "gla"])
@pytest.mark.parametrize("bounds", [(0, 41, 100), (0, 1, 70, 100)])
def test_context_parallel_matches_whole_sequence(kind, bounds):
    world = len(bounds) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, kind, bounds, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0] * world, codes
    got = dict(q.get(timeout=10) for _ in range(world))
    assert sorted(got) == list(range(world))
    for rank, errs in got.items():
        for name, e in errs.items():
            assert e < 1e-11, (rank, name, e)
    assert "S_T" in got[world - 1] and "dS0" in got[0]


def test_schedule_without_exchange_is_wrong():
    """Planted mistake (on the CPU, in the schedule's input): a rank that skips the composition
    (starts from a zero state) no longer matches the whole sequence -- the test above can fail."""
    import numpy as np

    import oracle
    from chunkwise_linear_attention_gb300 import context_parallel as cp

    d = problem("la")
    ops = oracle_ops("la")
    sl = {k: v[:, :, 41:100] for k, v in d.items() if k in ("q", "k", "v", "log_a")}
    o, _ = ops.fwd(sl["q"], sl["k"], sl["v"], sl["log_a"], None)
    ro, _ = oracle.la_fwd(d["q"], d["k"], d["v"], d["log_a"], d["S0"])
    assert np.max(np.abs(o.numpy() - ro[:, :, 41:100])) > 1e-3
    # while the composed incoming state (the schedule's step) restores it
    alpha0, dS0 = cp.local_pair_fwd(ops, *(d[k][:, :, :41] for k in ("q", "k", "v", "log_a")))
    import torch

    S_in = cp.incoming_state(ops, alpha0[None], dS0[None], 1, d["S0"])
    o2, _ = ops.fwd(sl["q"], sl["k"], sl["v"], sl["log_a"], S_in)
    assert np.max(np.abs(o2.numpy() - ro[:, :, 41:100])) < 1e-12
