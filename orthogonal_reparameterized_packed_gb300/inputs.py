"""Seeded synthetic inputs for the POET-X layer (shared by the oracle tests,
the GPU tests and the benchmark).

This module holds no arithmetic of the method itself: it only draws
Gaussian tensors with a fixed generator and rounds them to the working
precision, so that the CUDA path and the float64 oracle see identical
values.

Recipe (one ``numpy.random.default_rng(seed)`` stream, PCG64, drawn in this
fixed order):
  theta_P ~ N(0, sigma_theta^2)  shape [d_in/b][b(b-1)/2]   float32
  theta_R ~ N(0, sigma_theta^2)  shape [d_out/b][b(b-1)/2]  float32
  W0      ~ N(0, 1/d_in)         shape [d_out][d_in]        working dtype
  x       ~ N(0, 1)              shape [T][d_in]            working dtype
  dy      ~ N(0, 1)              shape [T][d_out]           working dtype
Working-dtype tensors are drawn in float64, rounded to float32 and then
(for bf16) rounded to nearest-even bfloat16; theta is always float32.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even); returns float32 values
    that are exactly representable in bfloat16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exact bfloat16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def packed_len(b: int) -> int:
    return b * (b - 1) // 2


@dataclasses.dataclass
class LayerInputs:
    d_in: int
    d_out: int
    b: int
    k: int
    tokens: int
    dtype: str            # "f32" or "bf16"
    theta_P: np.ndarray   # float32 [d_in/b][b(b-1)/2]
    theta_R: np.ndarray   # float32 [d_out/b][b(b-1)/2]
    W0: np.ndarray        # float32 values (bf16-exact in bf16 mode) [d_out][d_in]
    x: np.ndarray         # [T][d_in]
    dy: np.ndarray        # [T][d_out]


def _round(a: np.ndarray, dtype: str) -> np.ndarray:
    a32 = a.astype(np.float32)
    return round_to_bf16(a32) if dtype == "bf16" else a32


def make_layer_inputs(d_in: int, d_out: int, b: int, k: int, tokens: int,
                      dtype: str = "bf16", sigma_theta: float = 0.02,
                      seed: int = 0) -> LayerInputs:
    if dtype not in ("f32", "bf16"):
        raise ValueError(f"dtype must be 'f32' or 'bf16', got {dtype!r}")
    if d_in % b or d_out % b:
        raise ValueError("d_in and d_out must be multiples of b")
    rng = np.random.default_rng(seed)
    m = packed_len(b)
    theta_P = (rng.standard_normal((d_in // b, m)) * sigma_theta).astype(np.float32)
    theta_R = (rng.standard_normal((d_out // b, m)) * sigma_theta).astype(np.float32)
    W0 = _round(rng.standard_normal((d_out, d_in)) / np.sqrt(d_in), dtype)
    x = _round(rng.standard_normal((tokens, d_in)), dtype)
    dy = _round(rng.standard_normal((tokens, d_out)), dtype)
    return LayerInputs(d_in, d_out, b, k, tokens, dtype, theta_P, theta_R, W0, x, dy)


# The workloads the layer is exercised on (token counts are the full ones;
# tests slice tokens where the oracle would be too slow).
WORKLOADS = {
    # single layer, fp32, tiny
    "fp32_256_b32": dict(d_in=256, d_out=256, b=32, k=3, tokens=512, dtype="f32",
                         sigma_theta=0.01),
    # single layer, bf16, 2048 -> 5632 (batch 4 x seq 2048)
    "bf16_2048x5632": dict(d_in=2048, d_out=5632, b=256, k=3, tokens=8192, dtype="bf16"),
    # Llama-3-8B-shaped q/o projection, 16384 tokens (batch 4 x seq 4096)
    "llama3_8b_qo": dict(d_in=4096, d_out=4096, b=256, k=3, tokens=16384, dtype="bf16"),
    "llama3_8b_kv": dict(d_in=4096, d_out=1024, b=256, k=3, tokens=16384, dtype="bf16"),
    "llama3_8b_gate_up": dict(d_in=4096, d_out=14336, b=256, k=3, tokens=16384, dtype="bf16"),
    "llama3_8b_down": dict(d_in=14336, d_out=4096, b=256, k=3, tokens=16384, dtype="bf16"),
}

# 1.3B-shaped Llama-style model (d_model 2048, ffn 5632), 16384 tokens (batch 8 x seq 2048)
WORKLOADS.update({
    "llama_1p3b_attn": dict(d_in=2048, d_out=2048, b=256, k=3, tokens=16384, dtype="bf16"),
    "llama_1p3b_up": dict(d_in=2048, d_out=5632, b=256, k=3, tokens=16384, dtype="bf16"),
    "llama_1p3b_down": dict(d_in=5632, d_out=2048, b=256, k=3, tokens=16384, dtype="bf16"),
})

# Llama-3-8B decoder block: the seven projections (name, workload key)
LLAMA3_8B_BLOCK = [("q", "llama3_8b_qo"), ("k", "llama3_8b_kv"), ("v", "llama3_8b_kv"),
                   ("o", "llama3_8b_qo"), ("gate", "llama3_8b_gate_up"),
                   ("up", "llama3_8b_gate_up"), ("down", "llama3_8b_down")]

# one layer of the 1.3B-shaped model; the model has 24 of them (168 projections)
LLAMA_1P3B_LAYER = [("q", "llama_1p3b_attn"), ("k", "llama_1p3b_attn"), ("v", "llama_1p3b_attn"),
                    ("o", "llama_1p3b_attn"), ("gate", "llama_1p3b_up"), ("up", "llama_1p3b_up"),
                    ("down", "llama_1p3b_down")]

# workloads made of several projections run one after another in a step
# (all with the same token count): (projection name, workload key) lists
COMPOSITES = {
    "llama3_8b_block": LLAMA3_8B_BLOCK,
    "llama_1p3b_model": [(f"L{i}.{n}", key) for i in range(24) for n, key in LLAMA_1P3B_LAYER],
}
