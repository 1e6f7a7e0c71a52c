"""POET-X layer forward+backward throughput on GB300.

One step = the whole hot path for one projection: build the P and R blocks
from their packed parameters, forward y = R (W0 (P x)), backward to dx and
the packed dtheta_P, dtheta_R.  Default workload: the Llama-3-8B q/o
projection, 4096 x 4096, b = 256, k = 3, 16384 tokens, bf16 with fp32
accumulation.  Inputs are synthetic (seeded Gaussians of the documented
shapes) and already resident in HBM; x, dy (128 MiB each) and the step's
other tensors exceed the 129 MB L2, so no separate flush is needed.

--gpus N under torchrun runs N independent replicas (the layer does not
shard); value = tokens of all ranks / max time over ranks.
--impl reference times the float64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from orthogonal_reparameterized_packed_gb300.inputs import (COMPOSITES, WORKLOADS,  # noqa
                                                            make_layer_inputs)

METRIC = "POET-X layer fwd+bwd tokens/s (d=4096,b=256,bf16); % HBM / tensor-core roofline"
UNIT = "tokens/s"

# the isolated block-diagonal transform sweep: d = 4096, 8192 tokens, bf16
SWEEP = "transform_sweep"
SWEEP_D, SWEEP_T = 4096, 8192
SWEEP_CASES = [(b, k) for b in (32, 64, 128, 256, 512) for k in (1, 3, 5)]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="poetx", choices=["poetx", "reference"])
    ap.add_argument("--workload", default="llama3_8b_qo",
                    choices=sorted(WORKLOADS) + sorted(COMPOSITES) + [SWEEP],
                    help="one projection, or a composite run as its projections in sequence "
                         "(llama3_8b_block: the 7 of a Llama-3-8B decoder block; "
                         "llama_1p3b_model: all 168 of the 1.3B-shaped model)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--permute", action="store_true",
                    help="permuted block-diagonal factors (index maps around the plain step; "
                         "the two inner permutations folded into W0 once, before timing)")
    ap.add_argument("--train-step", action="store_true",
                    help="each step also applies Adam to theta_P and theta_R; the merge "
                         "W0 <- R W0 P is timed separately after the timed region")
    ap.add_argument("--w0-int8", action="store_true",
                    help="frozen weight held as INT8 codes with per-row scales, dequantised "
                         "into a bf16 buffer inside every step")
    ap.add_argument("--fuse-epilogue", action="store_true",
                    help="apply the block-diagonal factors in the W0 GEMMs' epilogues "
                         "(y = R v, dx = du P) instead of separate block transforms")
    ap.add_argument("--no-split-tail", action="store_true",
                    help="W0 GEMMs: every tile sums K in one CTA (no K split of the last "
                         "partial round of tiles across a cluster's two CTAs)")
    ap.add_argument("--profile-pass", action="store_true",
                    help="for profilers: W warm-up steps, then K eager steps and exit (no "
                         "timing repeats, graph, end-to-end leg or CPU baseline)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (profiling a smaller case)")
    ap.add_argument("--recompute-v", action="store_true",
                    help="backward recomputes v = W0 P x instead of reading it (saves T x d_out)")
    ap.add_argument("--sweep-case", default=None, metavar="B,K",
                    help="transform sweep: run only the case (b, k), e.g. 32,3 (profiling one "
                         "path of the sweep)")
    return ap.parse_args()


TOKENS_OVERRIDE = None


def workload_config(name):
    w = dict(WORKLOADS[name])
    if TOKENS_OVERRIDE is not None:
        w["tokens"] = TOKENS_OVERRIDE
    return w


def projections(name):
    """The (projection, workload key) pairs one step runs, in order."""
    return COMPOSITES[name] if name in COMPOSITES else [(name, name)]


def step_shapes(name):
    """Distinct workload keys of a step and how often each runs."""
    counts = {}
    for _, key in projections(name):
        counts[key] = counts.get(key, 0) + 1
    return counts


L2_BYTES = 129 * 10 ** 6


def input_bytes(w):
    """x, dy and W0 of one single-projection workload."""
    el = 4 if w["dtype"] == "f32" else 2
    return el * (w["tokens"] * (w["d_in"] + w["d_out"]) + w["d_in"] * w["d_out"])


def flush_between_steps(name):
    """A single projection whose inputs are under twice the L2: the next
    step would find much of them in L2, so the bench flushes L2 before every
    timed step instead of timing steps back to back."""
    return name in WORKLOADS and input_bytes(WORKLOADS[name]) < 2 * L2_BYTES


def config_json(name, n, args=None):
    counts = step_shapes(name)
    w = WORKLOADS[next(iter(counts))]
    c = {"workload": name, "b": w["b"], "k": w["k"], "tokens_per_gpu": w["tokens"],
         "dtype": w["dtype"], "parallelism": f"replicas{n}"}
    if name in WORKLOADS:
        c["d_in"], c["d_out"] = w["d_in"], w["d_out"]
        mib = input_bytes(w) / 2 ** 20
        c["l2"] = (f"flushed before every timed step (a 256 MiB write, then a 256 MiB read); "
                   f"each step timed alone: x, dy and W0 are {mib:.1f} MiB"
                   if flush_between_steps(name) else
                   f"inputs larger than L2 (x, dy and W0: {mib:.0f} MiB; more touched per step)")
    else:
        c["projections"] = len(projections(name))
        c["shapes"] = {key: {"d_in": WORKLOADS[key]["d_in"], "d_out": WORKLOADS[key]["d_out"],
                             "count": cnt} for key, cnt in counts.items()}
        c["l2"] = "every projection's activations exceed L2 or are evicted by the next ones"
    if args is not None and getattr(args, "permute", False):
        c["permuted_blocks"] = True
    if args is not None and getattr(args, "recompute_v", False):
        c["recompute_v"] = True
    if args is not None and getattr(args, "fuse_epilogue", False):
        c["block_epilogue"] = "fused into the W0 GEMMs"
    if args is not None and getattr(args, "no_split_tail", False):
        c["w0_split_tail"] = False
    if args is not None and getattr(args, "w0_int8", False):
        c["w0"] = "int8, per-row scales, dequantised each step"
    if args is not None and getattr(args, "train_step", False):
        c["optimizer"] = "adam (fused, in the step)"
    return c


# ----------------------------------------------------------- CPU oracle

def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("num_threads")]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(inp, sample_tokens):
    """Time the oracle on a bounded sample: the token-independent part (block
    build and CNP adjoint of both sides) once, and forward+backward on the
    first `sample_tokens` tokens.  Returns (t_fixed_s, t_per_token_s)."""
    import oracle
    b, k = inp.b, inp.k
    t0 = time.perf_counter()
    QP = oracle.unpack(inp.theta_P, b)
    QR = oracle.unpack(inp.theta_R, b)
    P = oracle.cayley_neumann(QP, k)
    R = oracle.cayley_neumann(QR, k)
    t1 = time.perf_counter()
    x = inp.x[:sample_tokens]
    dy = inp.dy[:sample_tokens]
    y, u, v = oracle.forward(x, inp.W0, P, R)
    dx, G_P, G_R = oracle.backward(dy, x, inp.W0, P, R, v)
    t2 = time.perf_counter()
    oracle.pack_skew_grad(oracle.cnp_adjoint(QP, G_P, k))
    oracle.pack_skew_grad(oracle.cnp_adjoint(QR, G_R, k))
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2), (t2 - t1) / sample_tokens


# tokens of each distinct projection shape the oracle runs per step (both
# oracle legs use the same sample, so their figures agree)
ORACLE_SAMPLE_TOKENS = 2048


def oracle_step(name, inps, sample_tokens):
    """One oracle step on the bounded sample: each distinct projection shape
    once (block build, forward + backward on `sample_tokens` tokens, CNP
    adjoint).  Returns the measured wall time (s) of each shape and the
    linear extrapolation of the full step (each shape's fixed part plus its
    per-token time times the full token count, weighted by how often the
    step runs the shape)."""
    counts = step_shapes(name)
    wall, full = {}, 0.0
    for key, inp in inps.items():
        t0 = time.perf_counter()
        t_fixed, t_tok = oracle_sample(inp, sample_tokens)
        wall[key] = time.perf_counter() - t0
        full += counts[key] * (t_fixed + t_tok * inp.tokens)
    return wall, full


def oracle_rates(name, inps, sample_tokens, wall, full_s, steps):
    """(measured tokens/s, extrapolated tokens/s) over `steps` steps whose
    per-shape wall times were summed into `wall`.  Measured: the sampled
    tokens / the wall time they took (fixed parts included); for a
    composite, each shape's time counts as often as the step runs it."""
    counts = step_shapes(name)
    weighted = sum(counts[key] * t for key, t in wall.items())
    T = next(iter(inps.values())).tokens
    return sample_tokens * steps / weighted, T * steps / full_s


def cpu_baseline(name, sample_tokens, seed=0):
    """The oracle on a bounded sample of the step's workload (one step)."""
    inps = {key: make_layer_inputs(**WORKLOADS[key], seed=seed) for key in step_shapes(name)}
    wall, full = oracle_step(name, inps, sample_tokens)
    measured, extrap = oracle_rates(name, inps, sample_tokens, wall, full, 1)
    T = next(iter(inps.values())).tokens
    return {"value": measured, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": (f"float64 numpy oracle, one step on a bounded sample: block build + CNP "
                       f"adjoint of both sides and forward+backward on {sample_tokens} of {T} "
                       f"tokens" + ("" if name in WORKLOADS else
                                    f" for each of the {len(inps)} distinct shapes, weighted by "
                                    f"its count in the {len(projections(name))} projections")
                       + f"; value = sampled tokens / measured {sum(wall.values()):.2f} s"),
            "extrapolated_full_step": {"value": extrap, "unit": UNIT, "s_per_step": full,
                                       "note": "linear in tokens to the full token count; "
                                               "not a measured time"}}


def run_reference_sweep(args):
    """The oracle's isolated transform (build, z = B x, dx and packed dtheta)
    for every (b, k) of the sweep on a bounded token sample."""
    import oracle
    d, T, sample = SWEEP_D, SWEEP_T, 512
    base = make_layer_inputs(d, d, 256, 3, sample, dtype="bf16", seed=0)
    thetas = {(b, k): (np.random.default_rng(10 * b + k).standard_normal(
        (d // b, b * (b - 1) // 2)) * 0.02).astype(np.float32) for b, k in SWEEP_CASES}

    def one_step():
        for (b, k), th in thetas.items():
            oracle.transform(th, base.x, base.dy, b, k)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    wall = time.perf_counter() - t0
    value = sample * len(SWEEP_CASES) * args.steps / wall
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": SWEEP, "d": d, "tokens_per_gpu": T, "dtype": "bf16"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(),
                             "kind": "oracle",
                             "sample": f"each step: every (b, k) of the sweep on {sample} of "
                                       f"{T} tokens; ms_per_step is the measured wall time"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    name = args.workload
    if name == SWEEP:
        run_reference_sweep(args)
        return
    inps = {key: make_layer_inputs(**WORKLOADS[key], seed=0) for key in step_shapes(name)}
    T = next(iter(inps.values())).tokens
    sample = ORACLE_SAMPLE_TOKENS
    for _ in range(args.warmup):
        oracle_step(name, inps, sample)
    wall = {key: 0.0 for key in inps}
    full = 0.0
    for _ in range(args.steps):
        w_, f_ = oracle_step(name, inps, sample)
        for key, t in w_.items():
            wall[key] += t
        full += f_
    value, extrap = oracle_rates(name, inps, sample, wall, full, args.steps)
    cores = blas_threads()
    sample_txt = (f"each step: block build + CNP adjoint of both sides and forward+backward "
                  f"on {sample} of {T} tokens" +
                  ("" if name in WORKLOADS else " per distinct projection shape, weighted by "
                   "the shape's count") + "; ms_per_step is the measured wall time of that")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(wall.values()) / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_json(name, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample_txt},
            "extrapolated_full_step": {"value": extrap, "unit": UNIT,
                                       "ms_per_step": 1e3 * full / args.steps,
                                       "note": "linear in tokens to the full token count; "
                                               "not a measured time"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ ranks

def max_over_ranks(x, device="cpu"):
    """Largest value of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_max):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max * 1e-3)


# -------------------------------------------------------------- GPU arm

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
        "fallback"


# the files each kernel is compiled from: its DRAM counters stay valid while
# these are unchanged
GEMM_SOURCES = ("gemm_tc.cu", "tc_common.cuh", "ptx.cuh", "internal.h")
PAIR_SOURCES = ("gemm_pair.cu", "tc_common.cuh", "ptx.cuh", "internal.h")
KERNEL_SOURCES = {
    "gemm_w0": PAIR_SOURCES, "gemm_w0_dgrad": PAIR_SOURCES, "transform": GEMM_SOURCES,
    "transform_t": GEMM_SOURCES, "outer": GEMM_SOURCES,
    "transform_sum": ("transform_sum_tc.cu", "tc_common.cuh", "ptx.cuh", "internal.h"),
}


def source_hash(files=GEMM_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, "orthogonal_reparameterized_packed_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(workload, tag):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is for other sources (of that kernel) or another workload."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    if not os.path.exists(p) or tag not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    k = d.get("kernels", {}).get(tag)
    if k is None or k.get("source_hash") != source_hash(KERNEL_SOURCES[tag]):
        return None
    return k["dram_read"] + k["dram_write"]


def algorithmic_work(tag, w):
    """(amount, unit, bound) per launch for a kernel tag of one step."""
    T, di, do, b = w["tokens"], w["d_in"], w["d_out"], w["b"]
    if tag in ("gemm_w0", "gemm_w0_dgrad"):
        return 2.0 * T * di * do / 1e12, "TFLOP", "tensor", "2*T*d_in*d_out"
    if tag == "gemm_w0_r":  # v = u W0^T with y = v R^T in the epilogue
        return 2.0 * T * do * (di + b) / 1e12, "TFLOP", "tensor", "2*T*d_out*(d_in+b)"
    if tag == "gemm_w0_dgrad_p":  # du = dv W0 with dx = du P in the epilogue
        return 2.0 * T * di * (do + b) / 1e12, "TFLOP", "tensor", "2*T*d_in*(d_out+b)"
    if tag in ("gemm_w0_fused", "gemm_w0_dgrad_fused"):  # both block factors and W0, one launch
        return (2.0 * T * (di * b + di * do + do * b) / 1e12, "TFLOP", "tensor",
                "2*T*(d_in*b+d_in*d_out+d_out*b)")
    return None


def time_merge(poetx, layer, dev, w, stream, peaks, reps=20):
    """Time the merge W0 <- R W0 P (into a copy of W0, factors kept) with CUDA
    events after the timed region: it runs once per merge period, not per step."""
    import torch
    W = dev["W0"].clone()
    for _ in range(3):
        poetx.poetx_merge(dev["W0"], layer.P_blocks, layer.R_blocks, W, None, None, w["d_in"],
                          w["d_out"], w["b"], layer.code, layer.workspace, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        poetx.poetx_merge(dev["W0"], layer.P_blocks, layer.R_blocks, W, None, None, w["d_in"],
                          w["d_out"], w["b"], layer.code, layer.workspace, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    S = max(w["b"], 256)
    flop = 4.0 * w["d_in"] * w["d_out"] * S  # W0 P and R (W0 P), superblock width S
    moved = 2.0 * 2 * w["d_in"] * w["d_out"]  # read W0, write W0_out (bf16)
    return {"us": us, "tflops": flop / (us * 1e-6) / 1e12,
            "hbm_gbs_min_bytes": moved / (us * 1e-6) / 1e9, "hbm_peak_gbs": peaks["hbm_gbs"],
            "note": "two launches (W0 P, then R M); once per merge period, not per step"}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import orthogonal_reparameterized_packed_gb300 as poetx
    from orthogonal_reparameterized_packed_gb300.layer import PoetxAdam, PoetxLayer, to_device

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    poetx.load_library()
    poetx.poetx_set_block_epilogue_fusion(args.fuse_epilogue)
    poetx.poetx_set_w0_split_tail(not args.no_split_tail)

    name = args.workload
    projs = projections(name)
    counts = step_shapes(name)
    single = name in WORKLOADS
    keys = list(counts)
    w = workload_config(keys[0])  # the (first) projection shape
    stream = torch.cuda.current_stream()
    shared = {}  # per-weight preparation shared by every layer instance

    def make_step(w, dev, acts):
        """A layer instance of shape w and its step over the weights and
        parameters in dev and the activation buffers `acts` (x, dy); every
        instance has its own outputs and workspace."""
        if args.permute:
            from orthogonal_reparameterized_packed_gb300.layer import PoetxPermutedLayer
            prng = np.random.default_rng(1000 + rank)
            lay = PoetxPermutedLayer(w["d_in"], w["d_out"], w["b"], w["k"], w["tokens"],
                                     prng.permutation(w["d_in"]), prng.permutation(w["d_out"]),
                                     dtype=w["dtype"])
            lay.fold(dev["W0"])  # once per weight, outside the timed steps

            def fn():
                lay.step(dev["theta_P"], dev["theta_R"], acts["x"], acts["dy"])
        elif args.w0_int8:
            from orthogonal_reparameterized_packed_gb300.layer import PoetxQLayer, quantize
            lay = PoetxQLayer(w["d_in"], w["d_out"], w["b"], w["k"], w["tokens"],
                              dtype=w["dtype"], recompute_v=args.recompute_v)
            wkey = id(dev["W0"])
            if wkey not in shared:  # once per weight
                shared[wkey] = quantize(dev["W0"], lay.code)
            W0_q, scales = shared[wkey]

            def fn():
                lay.step(dev["theta_P"], dev["theta_R"], W0_q, scales, acts["x"], acts["dy"])
        else:
            lay = PoetxLayer(w["d_in"], w["d_out"], w["b"], w["k"], w["tokens"],
                             dtype=w["dtype"], recompute_v=args.recompute_v)
            if args.train_step:
                # the graph replays the captured launch's bias correction;
                # theta_P, theta_R (and dtheta_P, dtheta_R) are one buffer: one launch
                opt = PoetxAdam([dev["theta"]], lr=1e-4)

                def fn():
                    lay.step(dev["theta_P"], dev["theta_R"], dev["W0"], acts["x"], acts["dy"])
                    opt.step([lay.dtheta])
            else:
                def fn():
                    lay.step(dev["theta_P"], dev["theta_R"], dev["W0"], acts["x"], acts["dy"])
        return lay, fn

    insts = {}  # per distinct projection shape: inputs on the device, layer, step
    for i, key in enumerate(keys):
        wk = workload_config(key)
        inp_k = make_layer_inputs(**wk, seed=rank if single else 1000 * rank + i)
        dev_k = to_device(inp_k)
        lay_k, fn_k = make_step(wk, dev_k, dev_k)
        insts[key] = {"w": wk, "dev": dev_k, "layer": lay_k, "step": fn_k}
    dev, layer = insts[keys[0]]["dev"], insts[keys[0]]["layer"]
    order = [insts[key]["step"] for _, key in projs]
    if len(projs) > 1 and not (args.permute or args.w0_int8 or args.train_step):
        # a model step: every projection's factors built by one call at the
        # start (its own packed parameters, copied from its shape's seeded
        # inputs), then each projection's forward and backward on its blocks
        from orthogonal_reparameterized_packed_gb300.layer import BlockStack
        stack = BlockStack([(insts[key]["w"]["d_in"], insts[key]["w"]["d_out"])
                            for _, key in projs], w["b"], w["k"], dtype=w["dtype"])
        for i, (_, key) in enumerate(projs):
            tp, tr = stack.theta_views(i)
            tp.copy_(insts[key]["dev"]["theta_P"])
            tr.copy_(insts[key]["dev"]["theta_R"])

        def proj_fn(i, key):
            lay_i, dev_i = insts[key]["layer"], insts[key]["dev"]
            tp, tr = stack.theta_views(i)
            P, R = stack.block_views(i)

            def fn():
                lay_i.forward(dev_i["x"], dev_i["W0"], P_blocks=P, R_blocks=R)
                lay_i.backward(dev_i["dy"], dev_i["x"], dev_i["W0"], tp, tr, P_blocks=P,
                               R_blocks=R)
            return fn
        order = [stack.build] + [proj_fn(i, key) for i, (_, key) in enumerate(projs)]

    def step():
        for fn in order:
            fn()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if poetx.poetx_device_status() != 0:
        raise RuntimeError("device status not OK after warm-up")
    if args.profile_pass:
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        status = poetx.poetx_device_status()
        if rank == 0:
            print(json.dumps({"profile_pass": name, "steps": args.steps, "tokens": w["tokens"],
                              "device_status": status}), flush=True)
        if status != 0:
            raise RuntimeError("device status not OK")
        return

    # (1) eager pass: every launch bracketed by CUDA events on its stream,
    #     giving the per-kernel durations the roofline uses.  Like the timed
    #     region below it runs for about a second (whole K-step rounds), so
    #     the kernels are timed in the same sustained power state.
    # (a composite step profiles a few steps: its launch count is large)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step()
    t1.record(stream)
    torch.cuda.synchronize()
    est_ms = max(t0.elapsed_time(t1), 1e-3)
    if single:
        rounds = max(1, min(100, int(1000.0 / (est_ms * args.steps)) + 1))
        prof_steps = args.steps * rounds
    else:
        prof_steps = min(args.steps, 3)
    launches0 = poetx.poetx_launch_count()
    poetx.poetx_profile_start(16 * len(projs) * prof_steps)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(prof_steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    poetx.poetx_profile_stop()
    launches_per_step = (poetx.poetx_launch_count() - launches0) // prof_steps
    ms_eager = t0.elapsed_time(t1) / prof_steps

    # (2) the same step captured once in a CUDA graph and replayed: the timed
    #     region of the headline number (no host launch overhead between kernels)
    def capture(fn):
        """A replayable form of fn: its CUDA graph, or fn itself (with the
        reason) when capture is refused."""
        if args.no_graph:
            return fn, None
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                fn()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            graphs.append(g)
            return g.replay, None
        except Exception as exc:  # capture refused: time eager launches instead
            torch.cuda.synchronize()
            return fn, repr(exc)[:200]

    graphs = []
    run_step, graph_error = capture(step)
    graph = graphs[0] if graphs else None

    # the timed region: exactly K steps between a barrier + synchronize on
    # each side, repeated until the repeats cover at least a second (so the
    # clock sampler sees a loaded GPU); ms_per_step is the median repeat
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    region_ms = []
    # small inputs: each step timed alone after an L2 flush that leaves no
    # dirty line behind (the region's time is the sum of its steps' times)
    flush_each = flush_between_steps(name)
    if flush_each:
        flush_w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        flush_r = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    while len(region_ms) < 3 or (sum(region_ms) < 1000.0 and len(region_ms) < 500):
        barrier()
        torch.cuda.synchronize()
        if flush_each:
            for e0, e1 in step_ev:
                flush_w.zero_()
                flush_r.sum()
                e0.record(stream)
                run_step()
                e1.record(stream)
            torch.cuda.synchronize()
            barrier()
            region_ms.append(sum(e0.elapsed_time(e1) for e0, e1 in step_ev))
            continue
        t0.record(stream)
        for _ in range(args.steps):
            run_step()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        region_ms.append(t0.elapsed_time(t1))
    clk = clocks.stop()
    launches = launches_per_step * args.steps * len(region_ms)  # every repeat of the region
    ms = statistics.median(region_ms) / args.steps
    ms_max = max_over_ranks(ms, "cuda")
    per_step = sorted(r / args.steps for r in region_ms)
    repeats = {"regions": len(region_ms), "steps_each": args.steps,
               "ms_per_step_median": ms, "ms_per_step_min": per_step[0],
               "ms_per_step_max": per_step[-1],
               "ms_per_step_p10": per_step[len(per_step) // 10],
               "ms_per_step_p90": per_step[(9 * len(per_step)) // 10],
               "total_s": sum(region_ms) / 1e3}
    status = poetx.poetx_device_status()

    # per-kernel times over the timed region
    tags = ["build", "unpack", "identity_plus", "expand_superblocks", "transform",
            "transform_t", "gemm_w0", "gemm_w0_dgrad", "gemm_w0_r", "gemm_w0_dgrad_p",
            "gemm_w0_fused", "gemm_w0_dgrad_fused", "outer", "reduce_extract", "cnp_bwd",
            "pack_skew", "f32_to_bf16", "chain", "prep_tiles", "pack_tiles", "permute", "adam",
            "transform_sum", "cnp_build", "cnp_sums", "cnp_adjoint",
            "dequantize", "quantize"]
    kernels = {}
    for t in tags:
        n, tot = poetx.poetx_profile_query(t)
        if n:
            kernels[t] = {"launches": n, "total_ms": tot, "avg_us": 1e3 * tot / n}
    peaks, peak_src = load_peaks()
    shapes = [insts[key]["w"] for _, key in projs]  # one entry per projection of the step

    def per_step(fn):
        return sum(fn(wp) for wp in shapes)

    # the dominant kernel: algorithmic work of all its launches / their summed time
    dom = max((t for t in kernels if algorithmic_work(t, w)), key=lambda t: kernels[t]["total_ms"])
    _, unit, bound, formula = algorithmic_work(dom, w)
    work = per_step(lambda wp: algorithmic_work(dom, wp)[0])
    achieved = work * prof_steps / (kernels[dom]["total_ms"] * 1e-3)
    # the sustained peak for a kernel inside a long step (a whole-model step of
    # 10 ms or more) or a profiled region of a second or more, the burst
    # peak otherwise
    long_region = ms_eager > 10.0 or ms_eager * prof_steps >= 900.0
    if w["dtype"] == "bf16":
        peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        peak_note = f"{peak_src} bf16 ({'sustained' if long_region else 'burst'})"
    else:  # fp32 FFMA on the CUDA cores: 128 lanes x 2 flop per SM per clock
        bound = "alu"
        sm_mhz = (clk or {}).get("sm_max_mhz") or 2070.0
        peak = torch.cuda.get_device_properties(local).multi_processor_count * 128 * 2 * \
            sm_mhz * 1e6 / 1e12
        peak_note = f"fp32 FFMA: SMs x 128 lanes x 2 flop x {sm_mhz:.0f} MHz"
    roofline = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": captured_traffic(name, dom) if single else None,
                "peak_source": peak_note,
                "per_launch": (f"{formula} = {work:.4f} TFLOP" if single else
                               f"{formula} summed over the {len(projs)} projections: "
                               f"{work:.4f} TFLOP per step"),
                "timing": f"CUDA events around each launch, eager pass of {prof_steps} steps "
                          f"({ms_eager * prof_steps / 1e3:.2f} s)"}

    # the HBM-bound kernels: algorithmic bytes of all their launches in the
    # timed steps / their summed event time
    def hbm_bytes(tag, wp):
        T, di, do = wp["tokens"], wp["d_in"], wp["d_out"]
        S = max(wp["b"], 256)
        return {
            # u = P x and y = R v: read + write bf16 activations, the superblocks
            "transform": 4.0 * T * (di + do) + 2.0 * S * (di + do),
            "transform_t": 4.0 * T * (di + do) + 2.0 * S * (di + do),
            # dv = dy R with sum_t v dy^T, dx = du P with sum_t x du^T: two reads, one write
            "transform_sum": 6.0 * T * (di + do) + 2.0 * S * (di + do),
            "outer": 4.0 * T * (di + do),
            # index maps: 2 over d_in, 2 over d_out, each reads and writes T x d bf16
            "permute": 8.0 * T * (di + do),
            # INT8 -> bf16 weight: 1 + 2 bytes per entry
            "dequantize": 3.0 * di * do,
        }[tag]

    hbm = []
    for tag in ("transform", "transform_t", "transform_sum", "outer", "permute", "dequantize"):
        if tag in kernels and w["dtype"] == "bf16":
            kt = kernels[tag]
            bytes_step = per_step(lambda wp: hbm_bytes(tag, wp))
            gbs = bytes_step * prof_steps / (kt["total_ms"] * 1e-3) / 1e9
            hbm.append({"kernel": tag, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                        "bytes_per_step": bytes_step,
                        "traffic": captured_traffic(name, tag) if single else None})
    roofline["hbm_kernels"] = hbm

    merge = None
    if single and args.train_step and not args.permute and not args.w0_int8:
        merge = time_merge(poetx, layer, dev, w, stream, peaks)

    # whole step against the HBM floor of a fully fused layer: x, y, v in the
    # forward, dy, v, x in and dx out in the backward (bf16), W0 read twice
    min_step_bytes = (per_step(lambda wp: wp["tokens"] * ((2 * wp["d_in"] + 4 * wp["d_out"]) +
                                                          (4 * wp["d_in"] + 4 * wp["d_out"])) +
                               4.0 * wp["d_in"] * wp["d_out"])
                      if w["dtype"] == "bf16" else None)

    # whole-step algorithmic tensor work for context
    step_flop = per_step(lambda wp: wp["tokens"] * (4.0 * wp["d_in"] * wp["d_out"] +
                                                    6.0 * wp["b"] * (wp["d_in"] + wp["d_out"])))
    value = job_throughput(w["tokens"], world, ms_max)

    # end to end through the C ABI from pinned host buffers: every step's x and
    # dy go host -> device and its results (y, dx and the packed dtheta)
    # device -> host inside the timed region.  Two buffer sets: step i+1's
    # inputs upload (copy stream) while step i computes, and step i's results
    # read back (another copy stream) during step i+1.
    e2e = None
    if single and not args.no_e2e:
        hx = dev["x"].cpu().pin_memory()
        hdy = dev["dy"].cpu().pin_memory()
        acts2 = {"x": torch.empty_like(dev["x"]), "dy": torch.empty_like(dev["dy"])}
        acts2["x"].copy_(dev["x"])
        acts2["dy"].copy_(dev["dy"])
        layer2, step2 = make_step(w, dev, acts2)
        step2()
        torch.cuda.synchronize()
        run_step2, _ = capture(step2)
        sets = [(dev, layer, run_step), (acts2, layer2, run_step2)]

        def host_like(t):
            return torch.empty(t.shape, dtype=t.dtype).pin_memory()

        outs = [{"y": host_like(lay.y), "dx": host_like(lay.dx), "dtheta": host_like(lay.dtheta)}
                for lay in (layer, layer2)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        down = [torch.cuda.Event() for _ in range(2)]

        def upload(j, after=None):
            with torch.cuda.stream(h2d):
                if after is not None:
                    h2d.wait_event(after)  # the set's previous step has read its inputs
                sets[j][0]["x"].copy_(hx, non_blocking=True)
                sets[j][0]["dy"].copy_(hdy, non_blocking=True)
                up[j].record(h2d)

        def pipeline(k, start):
            h2d.wait_event(start)
            d2h.wait_event(start)
            upload(0)
            for i in range(k):
                j = i % 2
                stream.wait_event(up[j])
                if i >= 2:
                    stream.wait_event(down[j])  # the set's results have been read back
                sets[j][2]()
                done[j].record(stream)
                if i + 1 < k:
                    upload((i + 1) % 2, done[(i + 1) % 2] if i >= 1 else None)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(done[j])
                    lay = sets[j][1]
                    outs[j]["y"].copy_(lay.y, non_blocking=True)
                    outs[j]["dx"].copy_(lay.dx, non_blocking=True)
                    outs[j]["dtheta"].copy_(lay.dtheta, non_blocking=True)
                    down[j].record(d2h)
            stream.wait_stream(d2h)
            stream.wait_stream(h2d)

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pipeline(2, e0)  # warm-up
        torch.cuda.synchronize()
        barrier()
        # at least the driver's K steps and at least ~0.5 s of them
        ksteps = max(args.steps, int(500.0 / max(ms, 1e-3) / 1.6) + 1)
        e0.record(stream)
        pipeline(ksteps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1) / ksteps, "cuda")
        nbytes = lambda t: t.numel() * t.element_size()  # noqa: E731
        e2e = {"value": job_throughput(w["tokens"], world, ems), "unit": UNIT,
               "h2d_bytes_per_step": nbytes(hx) + nbytes(hdy),
               "d2h_bytes_per_step": sum(nbytes(t) for t in outs[0].values()),
               "steps": ksteps, "ms_per_step": ems,
               "copies": "x, dy in; y, dx and the packed dtheta out, every step",
               "overlap": "double-buffered: while step i computes, step i+1's inputs upload "
                          "and step i-1's results read back on two copy streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, ORACLE_SAMPLE_TOKENS if single else 512, seed=rank)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": w["dtype"].replace("f32", "fp32"), "data": "synthetic",
                "config": config_json(name, world, args),
                "gpu_launches": launches, "gpu_launches_per_step": launches_per_step,
                "launch": "cuda_graph" if graph is not None else "eager",
                "graph_error": graph_error,
                "ms_per_step_eager": ms_eager, "roofline": roofline,
                "step_tflops": step_flop / (ms_max * 1e-3) / 1e12,
                "step_hbm": None if min_step_bytes is None else {
                    "min_bytes": min_step_bytes,
                    "achieved_gbs": min_step_bytes / (ms_max * 1e-3) / 1e9,
                    "frac": min_step_bytes / (ms_max * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    "note": "algorithmic floor of a fully fused layer step / step time"},
                "timed_repeats": repeats,
                "kernels": kernels, "merge": merge, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
                "device_status": status}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def sweep_bytes(b, d=SWEEP_D, T=SWEEP_T):
    """Algorithmic HBM bytes of the isolated transform: forward reads x and
    the blocks and writes z; backward reads dout, x and the blocks and
    writes dx and the packed dtheta (bf16 activations and blocks, fp32
    dtheta)."""
    blocks = 2.0 * d * b
    fwd = 4.0 * d * T + blocks
    bwd = 6.0 * d * T + blocks + 4.0 * d * (b - 1) / 2
    return fwd, bwd


def run_sweep(args):
    """Each (b, k) of the sweep: block build, forward z = B x and backward
    (dx, packed dtheta) timed call by call with CUDA events; L2 is flushed
    (a 256 MiB write, then a 256 MiB read) before every timed call, since x
    (64 MiB) fits in L2."""
    import torch

    import orthogonal_reparameterized_packed_gb300 as poetx

    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    poetx.load_library()
    d, T, c = SWEEP_D, SWEEP_T, poetx.BF16
    stream = torch.cuda.current_stream()
    base = make_layer_inputs(d, d, 256, 3, T, dtype="bf16", seed=rank)
    x = torch.from_numpy(base.x).cuda().to(torch.bfloat16)
    dout = torch.from_numpy(base.dy).cuda().to(torch.bfloat16)
    z = torch.empty_like(x)
    dx = torch.empty_like(x)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    # read after the write: its lines displace the flush's dirty ones, so the
    # timed call starts with an L2 that holds none of its data and owes no
    # write-backs of someone else's
    flush_read = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn, reps):
        tot = 0.0
        for _ in range(reps):
            flush.zero_()
            flush_read.sum()
            ev[0].record(stream)
            fn()
            ev[1].record(stream)
            torch.cuda.synchronize()
            tot += ev[0].elapsed_time(ev[1])
        return tot / reps

    sweep_cases = SWEEP_CASES
    if args.sweep_case:
        b_k = tuple(int(t) for t in args.sweep_case.split(","))
        if b_k not in SWEEP_CASES:
            raise SystemExit(f"--sweep-case {args.sweep_case}: not a case of the sweep")
        sweep_cases = [b_k]
    cases = []
    flush.zero_()  # the flush's own kernels warmed up before the first timed call
    flush_read.sum()
    torch.cuda.synchronize()
    launches0 = poetx.poetx_launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    for b, k in sweep_cases:
        rng = np.random.default_rng(1000 * rank + 10 * b + k)
        theta = torch.from_numpy((rng.standard_normal((d // b, b * (b - 1) // 2)) *
                                  0.02).astype(np.float32)).cuda()
        blocks = torch.empty((d // b, b, b), dtype=torch.bfloat16, device="cuda")
        dtheta = torch.empty_like(theta)
        ws = torch.empty((max(poetx.poetx_build_workspace_size(d, b, k, c),
                              poetx.poetx_transform_workspace_size(d, b, k, T, c), 16),),
                         dtype=torch.uint8, device="cuda")

        def build():
            poetx.poetx_build_blocks(theta, d, b, k, c, blocks, ws)

        def fwd():
            poetx.poetx_transform_forward(x, blocks, z, d, b, T, c, ws)

        def bwd():
            poetx.poetx_transform_backward(dout, x, theta, blocks, dx, dtheta, d, b, k, T, c, ws)

        for _ in range(max(args.warmup, 3)):
            build()
            fwd()
            bwd()
        torch.cuda.synchronize()
        reps = max(args.steps, 5)
        ms_b, ms_f, ms_w = timed(build, reps), timed(fwd, reps), timed(bwd, reps)
        fb, wb = sweep_bytes(b)
        cases.append({"b": b, "k": k, "build_us": 1e3 * ms_b, "fwd_us": 1e3 * ms_f,
                      "bwd_us": 1e3 * ms_w,
                      "fwd_gbs": fb / (ms_f * 1e-3) / 1e9, "bwd_gbs": wb / (ms_w * 1e-3) / 1e9,
                      "fwd_frac": fb / (ms_f * 1e-3) / 1e9 / hbm,
                      "bwd_frac": wb / (ms_w * 1e-3) / 1e9 / hbm})
    clk = clocks.stop()
    status = poetx.poetx_device_status()
    launches = poetx.poetx_launch_count() - launches0
    t_all = sum(cs["build_us"] + cs["fwd_us"] + cs["bwd_us"] for cs in cases) * 1e-6
    bytes_all = sum(sum(sweep_bytes(cs["b"])) for cs in cases)
    t_tr = sum(cs["fwd_us"] + cs["bwd_us"] for cs in cases) * 1e-6
    achieved = bytes_all / t_tr / 1e9
    if rank == 0:
        line = {"metric": METRIC, "value": T * len(cases) / t_all, "unit": UNIT, "n_gpus": 1,
                "steps": args.steps, "warmup": max(args.warmup, 3),
                "ms_per_step": 1e3 * t_all, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": SWEEP, "d": d, "tokens_per_gpu": T, "dtype": "bf16",
                           "cases": [f"b{b}_k{k}" for b, k in sweep_cases],
                           "l2": "flushed before every timed call: a 256 MiB write, then a "
                                 "256 MiB read that leaves no dirty line in L2"},
                "gpu_launches": launches, "launch": "eager",
                "roofline": {"bound": "hbm", "kernel": "block transform fwd + bwd, all cases",
                             "achieved": achieved, "peak": hbm, "unit": "GB/s",
                             "frac": achieved / hbm, "traffic": None,
                             "peak_source": f"{peak_src} copy bandwidth",
                             "per_launch": "fwd 4dT + 2db, bwd 6dT + 2db + 2d(b-1) bytes"},
                "sweep": cases, "clocks": clk, "e2e": None, "cpu_baseline": None,
                "device_status": status,
                "note": "value = tokens of all cases / the summed build + fwd + bwd time; "
                        "one step = the whole sweep once"}
        print(json.dumps(line), flush=True)


def main():
    global TOKENS_OVERRIDE
    args = parse()
    TOKENS_OVERRIDE = args.tokens
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == SWEEP:
        run_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
