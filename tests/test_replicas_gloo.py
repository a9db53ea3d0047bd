"""The benchmark's multi-GPU path on CPU: two gloo ranks run bench.py's
barrier, max-over-ranks timing and replica aggregation (each rank is an
independent replica; the job is timed by its slowest rank)."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, step_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._sync_all(torch, True)
        slowest = bench._max_over_ranks(torch, step_ms[rank], True)
        q.put((rank, slowest, bench.replica_throughput(world, 1.0e9, slowest)))
        bench._sync_all(torch, True)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_by_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    step_ms = [1.0, 2.5]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == pytest.approx(2.5)
        # 2 replicas x 1 GB per step / 2.5 ms = 800 GB/s
        assert value == pytest.approx(800.0)


def test_single_replica_throughput():
    import bench

    assert bench.replica_throughput(1, 1.0737e9, 0.2221) == pytest.approx(4834.4, rel=1e-4)
