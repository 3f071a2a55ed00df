"""The bench's multi-rank host logic on CPU: two gloo ranks, each with its own
timing, agree on the max and on the whole-job rate (weak scaling, no data-path
collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    total = bench.max_over_ranks(local_ms, dist, "cpu")
    rate = bench.whole_job_rate(world, units_per_rank=1000, steps=4, total_ms=total)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, total, rate))


def test_two_rank_max_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, total, rate in res:
        assert total == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 1000 * 4 / 0.015)


def test_single_rank_passthrough():
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(1, 10, 2, 1000.0) == pytest.approx(20.0)
