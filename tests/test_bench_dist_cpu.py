"""The multi-process plumbing of bench.py on CPU (gloo, world size 2): the
path runs independent replicas, so what has to hold is the rendezvous, the
barrier, the max over ranks of the timed region and that rank 0 alone prints
the JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, os.environ["PTI_ROOT"])
import bench
rank, world, local = bench.dist_setup(2)
assert world == 2 and rank == int(os.environ["RANK"])
bench.barrier(world)
v = bench.max_over_ranks(1.5 + rank, world)   # each rank times something different
assert v == 2.5, v
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print(f"rank {rank} ok")
"""


def torchrun(args, timeout=240):
    env = dict(os.environ, PTI_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_ranks_meet_and_take_the_max(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    r = torchrun([str(script)])
    assert r.returncode == 0, r.stdout + r.stderr
    assert "rank 0 ok" in r.stdout and "rank 1 ok" in r.stdout


def test_reference_arm_prints_one_line_from_rank_zero():
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--workload", "q8", "--steps", "1",
                  "--warmup", "3"])
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["cpu_baseline"]["kind"] == "oracle"
