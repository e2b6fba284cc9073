"""The bench's N > 1 host logic on CPU with two gloo ranks: replicas only, the
timed region's length is the slowest rank's, the job's throughput counts
every rank's units over that time."""
import json
import os
import socket
import subprocess
import sys

from conftest import ROOT

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
bench.barrier(dist)
t = bench.slowest_replica_ms(10.0 + 5.0 * rank, dist)
rate = bench.job_rate(8 * 100, world, t)
bench.barrier(dist)
print(json.dumps({"rank": rank, "world": world, "total_ms": t, "rate": rate}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), BENCH_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["total_ms"] == 15.0                   # rank 1's 15 ms, not rank 0's 10 ms
        assert o["rate"] == 8 * 100 * 2 / 0.015        # both ranks' units over the slowest time


def test_single_process_is_one_replica():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: v for k, v in os.environ.items() if k != "RANK"}
    old = dict(os.environ)
    try:
        os.environ.clear()
        os.environ.update(env)
        assert bench.dist_setup(4) == (0, 1, None)   # no launcher: one process, no group
    finally:
        os.environ.clear()
        os.environ.update(old)
    assert bench.slowest_replica_ms(12.5, None) == 12.5
    assert bench.job_rate(100, 1, 50.0) == 2000.0
