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


def test_bench_gpus_flag_starts_its_own_ranks(tmp_path):
    """bench.py --gpus 2 outside a launcher runs itself as two ranks
    (torch.distributed.run on 127.0.0.1); the reference arm's rank 0 prints
    the one JSON line, with n_gpus 2.  Under a launcher whose WORLD_SIZE is
    not --gpus it refuses."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl",
                        "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=str(tmp_path))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"
    env.update(WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl",
                        "reference", "--workload", "tiny"], capture_output=True, text=True,
                       env=env, timeout=300, cwd=str(tmp_path))
    assert r.returncode != 0 and "WORLD_SIZE=3" in r.stderr


def test_reference_arm_config_matches_the_gpu_arm():
    """Both arms describe the workload with the same config object."""
    import bench
    import gk_inputs as gi
    w = gi.get("gptoss_b64")
    c = gi.make_control(w)
    assert bench.workload_config(w, c, bench.kv_layout_desc()) == bench.workload_config(w, c)
