"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1).  The
attention path has no exchange step, so N GPUs run N independent replicas;
what must hold is the cross-rank bookkeeping: the job time is the slowest
rank's, the whole-job throughput counts every rank's work, and the
reference arm does its work on rank 0 only."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank={rank}, world_size=2)
rank = dist.get_rank()
times = [1.0 + rank, 0.5 * (2 - rank)]
mx = bench.max_over_ranks(times, 2)
tp = bench.job_throughput(100.0, 2, 4, mx[0])
dist.barrier()
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "max": mx, "throughput": tp}}))
"""


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_aggregate_like_the_bench():
    pytest.importorskip("torch")
    port = free_port()
    procs = [subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT, port=port, rank=r)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=120)
        assert pr.returncode == 0, err
        outs.append(__import__("json").loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["max"] == [2.0, 1.0]                  # slowest rank per entry
        assert o["throughput"] == 2 * 4 * 100.0 / 2.0  # every rank's units over the slowest time


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
