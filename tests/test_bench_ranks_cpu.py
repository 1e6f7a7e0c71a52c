"""The benchmark's multi-rank logic on CPU with the gloo backend (world size
2): max-over-ranks timing, whole-job throughput, and the reference arm
printing on rank 0 only."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
r = dist.get_rank()
m = bench.max_over_ranks(1.5 + 2.0 * r)        # rank 0: 1.5 ms, rank 1: 3.5 ms
assert m == 3.5, m
v = bench.job_throughput(1000, dist.get_world_size(), m)
assert abs(v - 2000 / 3.5e-3) < 1e-6, v
dist.barrier()
print(f"rank{r} ok")
dist.destroy_process_group()
"""


def _torchrun(args, extra_env=None, timeout=300):
    env = dict(os.environ, ROOT=ROOT, OMP_NUM_THREADS="1")
    if extra_env:
        env.update(extra_env)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29517"] + args
    return subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout,
                          cwd=ROOT)


def test_max_over_ranks_and_throughput_gloo(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    r = _torchrun([str(script)])
    assert r.returncode == 0, r.stdout + r.stderr
    assert "rank0 ok" in r.stdout and "rank1 ok" in r.stdout


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25) == 2.25
    assert bench.job_throughput(16384, 1, 1.0) == pytest.approx(16384e3)
