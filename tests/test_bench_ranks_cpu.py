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


def _reference_lines(stdout):
    import json
    return [json.loads(l) for l in stdout.splitlines() if l.startswith("{")]


def test_reference_arm_json_line():
    # the reference arm is the float64 oracle on the host cores: one JSON line
    # with the contract's keys, its own cpu_baseline and a host-only e2e
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "fp32_256_b32"], capture_output=True,
                       text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = _reference_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "fp32_256_b32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_prints_on_rank_zero_only():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0", "--workload", "fp32_256_b32"])
    assert r.returncode == 0, r.stdout + r.stderr
    lines = _reference_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference"


def test_l2_rule_per_workload():
    # a single projection whose x, dy and W0 are under twice the L2 is timed
    # step by step after a flush; the larger ones run back to back, and the
    # config says which, with the input size
    sys.path.insert(0, ROOT)
    import bench
    from orthogonal_reparameterized_packed_gb300.inputs import WORKLOADS
    w = WORKLOADS["llama3_8b_qo"]
    assert bench.input_bytes(w) == 2 * (16384 * 8192 + 4096 * 4096)
    assert bench.input_bytes(WORKLOADS["fp32_256_b32"]) == 4 * (512 * 512 + 256 * 256)
    assert not bench.flush_between_steps("llama3_8b_qo")
    assert bench.flush_between_steps("fp32_256_b32")
    assert bench.flush_between_steps("bf16_2048x5632")
    assert not bench.flush_between_steps("llama3_8b_block")  # composites: not single projections
    for name in WORKLOADS:
        l2 = bench.config_json(name, 1)["l2"]
        assert l2.startswith("flushed" if bench.flush_between_steps(name) else "inputs larger"), l2
        big = bench.input_bytes(WORKLOADS[name]) >= 2 * bench.L2_BYTES
        assert big != bench.flush_between_steps(name)
