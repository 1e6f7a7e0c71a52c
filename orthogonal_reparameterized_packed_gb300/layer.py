"""One POET-X layer step through the C ABI: device buffers held in torch
tensors, one shared workspace, and the four calls of a training step
(build P blocks, build R blocks, forward, backward) enqueued on one stream.
"""

from __future__ import annotations

import torch

from . import (BF16, F32, poetx_adam_update, poetx_backward, poetx_backward_workspace_size,
               poetx_build_blocks, poetx_build_workspace_size, poetx_fold_permutations,
               poetx_forward, poetx_forward_workspace_size, poetx_merge,
               poetx_merge_workspace_size, poetx_packed_size, poetx_permute_features)

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def dtype_code(name: str) -> int:
    return {"f32": F32, "bf16": BF16}[name]


class PoetxLayer:
    """Buffers for one projection y = R (W0 (P x)) with `tokens` tokens."""

    def __init__(self, d_in, d_out, b, k, tokens, dtype="bf16", device="cuda",
                 recompute_v=False):
        self.d_in, self.d_out, self.b, self.k, self.tokens = d_in, d_out, b, k, tokens
        self.code = dtype_code(dtype)
        self.recompute_v = recompute_v
        tdt = _TORCH_DTYPE[self.code]
        dev = torch.device(device)
        nP, nR = d_in // b, d_out // b
        self.P_blocks = torch.empty((nP, b, b), dtype=tdt, device=dev)
        self.R_blocks = torch.empty((nR, b, b), dtype=tdt, device=dev)
        self.y = torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.v = None if recompute_v else torch.empty((tokens, d_out), dtype=tdt, device=dev)
        self.dx = torch.empty((tokens, d_in), dtype=tdt, device=dev)
        self.dtheta_P = torch.empty((poetx_packed_size(d_in, b),), dtype=torch.float32,
                                    device=dev)
        self.dtheta_R = torch.empty((poetx_packed_size(d_out, b),), dtype=torch.float32,
                                    device=dev)
        ws = max(poetx_build_workspace_size(d_in, b, k, self.code),
                 poetx_build_workspace_size(d_out, b, k, self.code),
                 poetx_forward_workspace_size(d_in, d_out, b, tokens, self.code),
                 poetx_backward_workspace_size(d_in, d_out, b, k, tokens, self.code,
                                               recompute_v),
                 poetx_merge_workspace_size(d_in, d_out, b, self.code))
        self.workspace = torch.empty((max(ws, 16),), dtype=torch.uint8, device=dev)

    def build(self, theta_P, theta_R, stream=None):
        poetx_build_blocks(theta_P, self.d_in, self.b, self.k, self.code, self.P_blocks,
                           self.workspace, stream)
        poetx_build_blocks(theta_R, self.d_out, self.b, self.k, self.code, self.R_blocks,
                           self.workspace, stream)

    def forward(self, x, W0, stream=None):
        poetx_forward(x, W0, self.P_blocks, self.R_blocks, self.y, self.v, self.d_in,
                      self.d_out, self.b, self.tokens, self.code, self.workspace, stream)
        return self.y

    def backward(self, dy, x, W0, theta_P, theta_R, stream=None):
        poetx_backward(dy, x, W0, theta_P, theta_R, self.P_blocks, self.R_blocks, self.v,
                       self.dx, self.dtheta_P, self.dtheta_R, self.d_in, self.d_out, self.b,
                       self.k, self.tokens, self.code, self.workspace, stream)
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
    """Upload a LayerInputs (numpy) to torch tensors in the working dtype."""
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def act(a):
        return torch.from_numpy(a).to(device=device).to(tdt).contiguous()

    return dict(theta_P=torch.from_numpy(inp.theta_P).to(device).contiguous(),
                theta_R=torch.from_numpy(inp.theta_R).to(device).contiguous(),
                W0=act(inp.W0), x=act(inp.x), dy=act(inp.dy))


class PoetxPermutedLayer:
    """One projection with permuted block-diagonal factors,
    R = Pi_R^T B_R Pi_R and P = Pi_P^T B_P Pi_P.  The two inner permutations
    are folded into the weight once (fold()); each step applies the outer two
    to the activations as index maps around a plain PoetxLayer step."""

    def __init__(self, d_in, d_out, b, k, tokens, perm_P, perm_R, dtype="bf16", device="cuda"):
        import numpy as np
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
