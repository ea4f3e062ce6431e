"""The benchmark's multi-rank timing reduction (replicas only: no collective
on the data path) on two gloo ranks on CPU: max of the elapsed times, sum of
the units."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.dist_init("gloo")
    assert bench.dist_env() == (rank, rank, world)
    ms, units = bench.reduce_timing(10.0 + 5.0 * rank, 100.0 * (rank + 1), d, torch.device("cpu"))
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_timing_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units in res:
        assert ms == pytest.approx(15.0) and units == pytest.approx(300.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_timing(3.0, 7.0, None) == (3.0, 7.0)
