"""The benchmark's multi-rank host logic on CPU: two gloo ranks (world size 2,
127.0.0.1 rendezvous) agree on the slowest rank's time, the whole-job figure
counts every replica, and the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [3.0, 7.5][rank]
    slowest = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, slowest, bench.job_throughput(world, 10**9, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [7.5, 7.5]
    # 2 replicas x 1 GB per step in 7.5 ms
    assert all(abs(g[2] - 2e9 / 7.5e-3 / 1e9) < 1e-6 for g in got)


def test_reference_arm_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mha", "--steps", "1", "--warmup", "3", "--gpus", "2"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
