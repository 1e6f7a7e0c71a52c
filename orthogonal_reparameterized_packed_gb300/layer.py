"""One POET-X layer step through the C ABI: device buffers held in torch
tensors, one shared workspace, and the four calls of a training step
(build P blocks, build R blocks, forward, backward) enqueued on one stream.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (BF16, F32, poetx_adam_update, poetx_backward, poetx_backward_workspace_size,
               poetx_build_blocks, poetx_build_workspace_size, poetx_dequantize_w0,
               poetx_fold_permutations, poetx_forward, poetx_forward_workspace_size,
               poetx_merge, poetx_merge_workspace_size, poetx_packed_size,
               poetx_permute_features, poetx_quantize_w0)

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def dtype_code(name: str) -> int:
    return {"f32": F32, "bf16": BF16}[name]


def adjacent(a, b):
    """The combined tensor if float32 tensors a and b lie back to back in one
    allocation (a first), else None."""
    if not (a.is_contiguous() and b.is_contiguous() and a.dtype == b.dtype == torch.float32):
        return None
    if a.data_ptr() + a.numel() * 4 != b.data_ptr():
        return None
    if a.untyped_storage().data_ptr() != b.untyped_storage().data_ptr():
        return None
    base = a.untyped_storage()
    off = (a.data_ptr() - base.data_ptr()) // 4
    return torch.empty(0, dtype=torch.float32, device=a.device).set_(
        base, off, (a.numel() + b.numel(),), (1,))


class PoetxLayer:
    """Buffers for one projection y = R (W0 (P x)) with `tokens` tokens.

    The P and R blocks (and dtheta_P, dtheta_R) are views of one allocation,
    P first: blocks are independent, so when theta_P and theta_R also lie
    back to back the two factors are built by a single call over
    d_in + d_out features."""

    def __init__(self, d_in, d_out, b, k, tokens, dtype="bf16", device="cuda",
                 recompute_v=False):
        self.d_in, self.d_out, self.b, self.k, self.tokens = d_in, d_out, b, k, tokens
        self.code = dtype_code(dtype)
        self.recompute_v = recompute_v
        tdt = _TORCH_DTYPE[self.code]
        dev = torch.device(device)
        nP, nR = d_in // b, d_out // b
        self.blocks = torch.empty((nP + nR, b, b), dtype=tdt, device=dev)
        self.P_blocks = self.blocks[:nP]
        self.R_blocks = self.blocks[nP:]
        self.y = torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.v = None if recompute_v else torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.dx = torch.empty((tokens, d_in), dtype=tdt, device=dev)
        mP, mR = poetx_packed_size(d_in, b), poetx_packed_size(d_out, b)
        self.dtheta = torch.empty((mP + mR,), dtype=torch.float32, device=dev)
        self.dtheta_P = self.dtheta[:mP]
        self.dtheta_R = self.dtheta[mP:]
        ws = max(poetx_build_workspace_size(d_in, b, k, self.code),
                 poetx_build_workspace_size(d_out, b, k, self.code),
                 poetx_build_workspace_size(d_in + d_out, b, k, self.code),
                 poetx_forward_workspace_size(d_in, d_out, b, tokens, self.code),
                 poetx_backward_workspace_size(d_in, d_out, b, k, tokens, self.code,
                                               recompute_v),
                 poetx_merge_workspace_size(d_in, d_out, b, self.code))
        self.workspace = torch.empty((max(ws, 16),), dtype=torch.uint8, device=dev)

    def build(self, theta_P, theta_R, stream=None):
        theta = adjacent(theta_P, theta_R)
        if theta is not None:  # both factors in one call
            poetx_build_blocks(theta, self.d_in + self.d_out, self.b, self.k, self.code,
                               self.blocks, self.workspace, stream)
            return
        poetx_build_blocks(theta_P, self.d_in, self.b, self.k, self.code, self.P_blocks,
                           self.workspace, stream)
        poetx_build_blocks(theta_R, self.d_out, self.b, self.k, self.code, self.R_blocks,
                           self.workspace, stream)

    def forward(self, x, W0, stream=None, P_blocks=None, R_blocks=None):
        """P_blocks, R_blocks: blocks built elsewhere (e.g. by a BlockStack)
        instead of this layer's own."""
        P = self.P_blocks if P_blocks is None else P_blocks
        R = self.R_blocks if R_blocks is None else R_blocks
        poetx_forward(x, W0, P, R, self.y, self.v, self.d_in, self.d_out, self.b, self.tokens,
                      self.code, self.workspace, stream)
        return self.y

    def backward(self, dy, x, W0, theta_P, theta_R, stream=None, P_blocks=None, R_blocks=None):
        P = self.P_blocks if P_blocks is None else P_blocks
        R = self.R_blocks if R_blocks is None else R_blocks
        poetx_backward(dy, x, W0, theta_P, theta_R, P, R, self.v, self.dx, self.dtheta_P,
                       self.dtheta_R, self.d_in, self.d_out, self.b, self.k, self.tokens,
                       self.code, self.workspace, stream)
        return self.dx, self.dtheta_P, self.dtheta_R

    def step(self, theta_P, theta_R, W0, x, dy, stream=None):
        """Build both sides, forward, backward (one training step's layer work)."""
        self.build(theta_P, theta_R, stream)
        self.forward(x, W0, stream)
        self.backward(dy, x, W0, theta_P, theta_R, stream)
        return self.y, self.dx, self.dtheta_P, self.dtheta_R


    def merge(self, W0, theta_P, theta_R, stream=None):
        """Fold the current blocks into the weight, W0 <- R W0 P (in place),
        and restart both factors at the identity (theta_P = theta_R = 0).
        Uses the blocks of the last build()."""
        poetx_merge(W0, self.P_blocks, self.R_blocks, W0, theta_P, theta_R, self.d_in,
                    self.d_out, self.b, self.code, self.workspace, stream)


class PoetxQLayer(PoetxLayer):
    """The layer with its frozen weight held as INT8 codes and per-row
    scales.  Each step dequantises W0 into a bf16 (or fp32) buffer that the
    forward and backward read; the buffer is scratch shared by nothing
    else, so a model can reuse one for all its layers."""

    def __init__(self, d_in, d_out, b, k, tokens, dtype="bf16", device="cuda",
                 recompute_v=False):
        super().__init__(d_in, d_out, b, k, tokens, dtype=dtype, device=device,
                         recompute_v=recompute_v)
        self.W0 = torch.empty((d_out, d_in), dtype=_TORCH_DTYPE[self.code],
                              device=torch.device(device))

    def dequantize(self, W0_q, scales, stream=None):
        poetx_dequantize_w0(W0_q, scales, self.W0, self.d_in, self.d_out, self.code, stream)
        return self.W0

    def step(self, theta_P, theta_R, W0_q, scales, x, dy, stream=None):
        self.build(theta_P, theta_R, stream)
        self.dequantize(W0_q, scales, stream)
        self.forward(x, self.W0, stream)
        self.backward(dy, x, self.W0, theta_P, theta_R, stream)
        return self.y, self.dx, self.dtheta_P, self.dtheta_R

    def merge_quantized(self, W0_q, scales, theta_P, theta_R, stream=None):
        """W0 <- R W0 P on the dequantised weight, then re-quantised in place;
        the factors restart at the identity.  Uses the blocks of the last
        build()."""
        self.dequantize(W0_q, scales, stream)
        self.merge(self.W0, theta_P, theta_R, stream)
        poetx_quantize_w0(self.W0, W0_q, scales, self.d_in, self.d_out, self.code, stream)


def quantize(W0, code, stream=None):
    """INT8 codes and float32 scales of a [d_out][d_in] weight tensor."""
    d_out, d_in = W0.shape
    q = torch.empty((d_out, d_in), dtype=torch.int8, device=W0.device)
    s = torch.empty((d_out,), dtype=torch.float32, device=W0.device)
    poetx_quantize_w0(W0, q, s, d_in, d_out, code, stream)
    return q, s


class PoetxAdam:
    """Adam on packed parameter vectors (float32 device tensors), one fused
    launch per vector per step."""

    def __init__(self, params, lr, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0):
        self.params = list(params)
        self.lr, self.betas, self.eps, self.weight_decay = lr, betas, eps, weight_decay
        self.m = [torch.zeros_like(p) for p in self.params]
        self.v = [torch.zeros_like(p) for p in self.params]
        self.t = 0

    def reset(self):
        """Zero the moments (after a merge restarts the factors)."""
        for m, v in zip(self.m, self.v):
            m.zero_()
            v.zero_()
        self.t = 0

    def step(self, grads, stream=None):
        self.t += 1
        for p, g, m, v in zip(self.params, grads, self.m, self.v):
            poetx_adam_update(p, g, m, v, p.numel(), self.t, self.lr, self.betas[0],
                              self.betas[1], self.eps, self.weight_decay, stream)


def to_device(inp, device="cuda"):
    """Upload a LayerInputs (numpy) to torch tensors in the working dtype.
    theta_P and theta_R are views of one buffer `theta` (P first)."""
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def act(a):
        return torch.from_numpy(a).to(device=device).to(tdt).contiguous()

    nP = inp.theta_P.size
    theta = torch.from_numpy(np.concatenate([inp.theta_P.ravel(), inp.theta_R.ravel()])).to(
        device)
    return dict(theta=theta, theta_P=theta[:nP].view(inp.theta_P.shape),
                theta_R=theta[nP:].view(inp.theta_R.shape),
                W0=act(inp.W0), x=act(inp.x), dy=act(inp.dy))


class BlockStack:
    """The packed parameters and blocks of many projections (same b, k and
    dtype) in two allocations, so that one poetx_build_blocks call builds
    every factor of a model at the start of a step (blocks are independent).
    `shapes` lists (d_in, d_out) per projection; theta(i) and blocks(i) give
    projection i's (theta_P, theta_R) and (P_blocks, R_blocks) views."""

    def __init__(self, shapes, b, k, dtype="bf16", device="cuda"):
        self.b, self.k, self.code = b, k, dtype_code(dtype)
        dev = torch.device(device)
        self.shapes = list(shapes)
        self.d = sum(di + do for di, do in self.shapes)
        self._theta_off, self._block_off = [], []
        t = n = 0
        for di, do in self.shapes:
            self._theta_off.append(t)
            self._block_off.append(n)
            t += poetx_packed_size(di, b) + poetx_packed_size(do, b)
            n += (di + do) // b
        self.theta = torch.zeros((t,), dtype=torch.float32, device=dev)
        self.blocks = torch.empty((n, b, b), dtype=_TORCH_DTYPE[self.code], device=dev)
        ws = poetx_build_workspace_size(self.d, b, k, self.code)
        self.workspace = torch.empty((max(ws, 16),), dtype=torch.uint8, device=dev)

    def theta_views(self, i):
        di, do = self.shapes[i]
        mP, mR = poetx_packed_size(di, self.b), poetx_packed_size(do, self.b)
        o = self._theta_off[i]
        return (self.theta[o:o + mP].view(di // self.b, -1),
                self.theta[o + mP:o + mP + mR].view(do // self.b, -1))

    def block_views(self, i):
        di, do = self.shapes[i]
        o = self._block_off[i]
        return self.blocks[o:o + di // self.b], self.blocks[o + di // self.b:o + (di + do) // self.b]

    def build(self, stream=None):
        """Every factor of every projection, one call."""
        poetx_build_blocks(self.theta, self.d, self.b, self.k, self.code, self.blocks,
                           self.workspace, stream)


class PoetxPermutedLayer:
    """One projection with permuted block-diagonal factors,
    R = Pi_R^T B_R Pi_R and P = Pi_P^T B_P Pi_P.  The two inner permutations
    are folded into the weight once (fold()); each step applies the outer two
    to the activations as index maps around a plain PoetxLayer step."""

    def __init__(self, d_in, d_out, b, k, tokens, perm_P, perm_R, dtype="bf16", device="cuda"):
        self.inner = PoetxLayer(d_in, d_out, b, k, tokens, dtype=dtype, device=device)
        self.code = self.inner.code
        dev = torch.device(device)

        def as_dev(p):
            return torch.from_numpy(np.ascontiguousarray(p, dtype=np.int32)).to(dev)

        perm_P = np.asarray(perm_P)
        perm_R = np.asarray(perm_R)
        self.perm_P, self.perm_R = as_dev(perm_P), as_dev(perm_R)
        self.inv_P, self.inv_R = as_dev(np.argsort(perm_P)), as_dev(np.argsort(perm_R))
        tdt = _TORCH_DTYPE[self.code]
        self.W0_folded = torch.empty((d_out, d_in), dtype=tdt, device=dev)
        self.xp = torch.empty((tokens, d_in), dtype=tdt, device=dev)
        self.dyp = torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.y = torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.dx = torch.empty((tokens, d_in), dtype=tdt, device=dev)

    @property
    def dtheta_P(self):
        return self.inner.dtheta_P

    @property
    def dtheta_R(self):
        return self.inner.dtheta_R

    def fold(self, W0, stream=None):
        """W0' = Pi_R W0 Pi_P^T, once per weight."""
        poetx_fold_permutations(W0, self.perm_R, self.perm_P, self.W0_folded, self.inner.d_in,
                                self.inner.d_out, self.code, stream)

    def step(self, theta_P, theta_R, x, dy, stream=None):
        L = self.inner
        T = L.tokens
        poetx_permute_features(x, self.perm_P, self.xp, T, L.d_in, self.code, stream)
        L.build(theta_P, theta_R, stream)
        L.forward(self.xp, self.W0_folded, stream)
        poetx_permute_features(L.y, self.inv_R, self.y, T, L.d_out, self.code, stream)
        poetx_permute_features(dy, self.perm_R, self.dyp, T, L.d_out, self.code, stream)
        L.backward(self.dyp, self.xp, self.W0_folded, theta_P, theta_R, stream)
        poetx_permute_features(L.dx, self.inv_P, self.dx, T, L.d_in, self.code, stream)
        return self.y, self.dx, L.dtheta_P, L.dtheta_R
