"""bench.py's multi-replica bookkeeping on CPU with two gloo ranks: the timed
region is the slowest rank's, and the value counts every rank's work."""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [10.0, 25.0][rank]                    # rank 1 is the slow replica
    total = bench.slowest_rank_ms(local_ms, world, "cpu")
    value = bench.whole_job_tflops(2e12, 5, world, total)
    q.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, total, value in res:
        assert total == 25.0
        # 2 ranks x 5 steps x 2 TFLOP in 25 ms
        assert value == pytest.approx(2 * 5 * 2e12 / 25e-3 / 1e12)


def test_single_rank_passthrough():
    import bench
    assert bench.slowest_rank_ms(7.5, 1) == 7.5
    assert bench.whole_job_tflops(1e12, 4, 1, 2.0) == pytest.approx(2000.0)
