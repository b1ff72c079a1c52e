"""The replicated multi-process path on CPU (world size 2, gloo): the
max-over-ranks time and whole-job value bench.py reports, and the reference
arm under torchrun, where rank 0 alone runs and prints its line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [250.0, 262.5][rank]  # this rank's time for its steps
    out[rank] = bench.max_over_ranks(local, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    assert out[0] == out[1] == 262.5  # every rank reports the slowest rank's time


def test_whole_job_value():
    sys.path.insert(0, ROOT)
    import bench

    # two replicas of 100 steps each in 25 ms (the slowest rank): 8000 steps/s
    assert bench.whole_job_value(2, 100, 25.0) == pytest.approx(8000.0)
    assert bench.whole_job_value(1, 10, 2.5) == pytest.approx(4000.0)


def test_reference_arm_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_fp32"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["config"]["workload"] == "tiny_fp32"
