"""Replica aggregation of bench.py across ranks, world_size 2 over gloo on CPU:
the slowest rank's time sets the step time and the job throughput counts the
work of every rank (the attention forward shards with no exchange)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]              # rank 1 is the slow replica
    t = bench.max_over_ranks(ms, world, torch.device("cpu"))
    v = bench.job_rate(2.0e12, t, world, "causal")
    results[rank] = (t, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        t, v = results[r]
        assert t == 5.0                                   # max over ranks
        assert abs(v - 2 * 2.0e12 / 5e-3 / 1e12) < 1e-9   # TFLOP/s of both replicas


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_rate(1e12, 1.0, 1, "causal") == pytest.approx(1000.0)
    assert bench.job_rate(2e9, 1.0, 1, "decode") == pytest.approx(2000.0)


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` started outside torchrun re-launches itself with two
    ranks (torch.distributed.run); --dry-run keeps it on the CPU (gloo)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run",
                        "--steps", "4", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2
    assert d["max_over_ranks"] == 2.0       # ranks report 1 and 2; the max wins
