"""Parity at the workloads' full sizes, run exactly as the benchmark runs
them (one PoetxLayer step per projection shape).  The oracle checks sampled
outputs it can compute one by one: y and dx rows of sampled tokens (each
row depends on its own token only), and dtheta of sampled blocks (each
block's gradient is a sum over all tokens of that block's features only).
Tolerance: 2e-2 relative Frobenius (bf16 with fp32 accumulation) over the
sampled rows and per sampled block, and 4e-2 on the worst single row."""

import numpy as np
import pytest

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import WORKLOADS, make_layer_inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_ROW = 4e-2  # largest single-row error: twice the Frobenius tolerance


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def max_row_rel(got, want):
    """Largest relative error of one sampled row."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    num = np.linalg.norm(got - want, axis=1)
    return float(np.max(num / np.maximum(np.linalg.norm(want, axis=1), 1e-300)))


def tile_rows(T, rng, tile=128):
    """One random token in every tile of `tile` tokens, plus the first and last."""
    starts = np.arange(0, T, tile)
    offs = rng.integers(0, tile, size=len(starts))
    rows = np.minimum(starts + offs, T - 1)
    return np.unique(np.concatenate([[0, T - 1], rows]))


def sampled_check(layer, inp, rng):
    b, k, T = inp.b, inp.k, inp.tokens
    P = oracle.build_blocks(inp.theta_P, b, k)
    R = oracle.build_blocks(inp.theta_R, b, k)
    # rows of sampled tokens: one at random in every 128-token tile (so every
    # output tile of every kernel holds a checked row, the last partial round
    # of GEMM tiles included), the first and the last
    rows = tile_rows(T, rng)
    y_ref, _, v_ref = oracle.forward(inp.x[rows], inp.W0, P, R)
    dx_ref, _, _ = oracle.backward(inp.dy[rows], inp.x[rows], inp.W0, P, R, v_ref)
    idx = torch.from_numpy(rows).cuda()
    y_got = layer.y.index_select(0, idx).float().cpu().numpy()
    dx_got = layer.dx.index_select(0, idx).float().cpu().numpy()
    errs = {"y": rel_fro(y_got, y_ref), "dx": rel_fro(dx_got, dx_ref),
            "y max row": max_row_rel(y_got, y_ref), "dx max row": max_row_rel(dx_got, dx_ref)}
    # dtheta of sampled blocks
    nP, nR = inp.d_in // b, inp.d_out // b
    QP = oracle.unpack(inp.theta_P, b)
    QR = oracle.unpack(inp.theta_R, b)
    dthR = layer.dtheta_R.view(nR, -1).cpu().numpy()
    dthP = layer.dtheta_P.view(nP, -1).cpu().numpy()
    for g in sorted({0, nR // 2, nR - 1}):
        sl = slice(g * b, (g + 1) * b)
        v_g = oracle.forward_v_rows(inp.x, inp.W0, P, sl)
        G = oracle.blockwise_outer(inp.dy[:, sl], v_g, b)
        want = oracle.pack_skew_grad(oracle.cnp_adjoint(QR[g:g + 1], G, k))[0]
        errs[f"dtheta_R[{g}]"] = rel_fro(dthR[g], want)
    for g in sorted({0, nP // 2, nP - 1}):
        sl = slice(g * b, (g + 1) * b)
        du_g = oracle.backward_du_cols(inp.dy, inp.W0, R, sl)
        G = oracle.blockwise_outer(du_g, inp.x[:, sl], b)
        want = oracle.pack_skew_grad(oracle.cnp_adjoint(QP[g:g + 1], G, k))[0]
        errs[f"dtheta_P[{g}]"] = rel_fro(dthP[g], want)
    bad = {n: e for n, e in errs.items() if not e <= (TOL_ROW if "max row" in n else TOL)}
    assert not bad, f"above tolerance: {bad} (all: {errs})"


# the distinct projection shapes of the workloads, full token counts
FULL = [
    ("bf16_2048x5632", dict(WORKLOADS["bf16_2048x5632"])),
    ("llama3_8b_qo", dict(WORKLOADS["llama3_8b_qo"])),
    ("llama3_8b_kv", dict(WORKLOADS["llama3_8b_kv"])),
    ("llama3_8b_gate_up", dict(WORKLOADS["llama3_8b_gate_up"])),
    ("llama3_8b_down", dict(WORKLOADS["llama3_8b_down"])),
    ("llama_1b3_qkvo", dict(d_in=2048, d_out=2048, b=256, k=3, tokens=16384, dtype="bf16")),
    ("llama_1b3_down", dict(d_in=5632, d_out=2048, b=256, k=3, tokens=16384, dtype="bf16")),
]


@pytest.mark.parametrize("name,cfg", FULL, ids=[n for n, _ in FULL])
def test_full_size_layer(px, name, cfg):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    inp = make_layer_inputs(**cfg, seed=0)
    dev = to_device(inp)
    layer = PoetxLayer(inp.d_in, inp.d_out, inp.b, inp.k, inp.tokens, dtype=inp.dtype)
    layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"])
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    sampled_check(layer, inp, np.random.default_rng(1))


SWEEP = [(b, k) for b in (32, 64, 128, 256, 512) for k in (1, 3, 5)]


@pytest.mark.parametrize("b,k", SWEEP)
def test_full_size_transform_sweep(px, b, k):
    d, T = 4096, 8192
    inp = make_layer_inputs(d, d, b, k, T, dtype="bf16", seed=100 + b + k)
    c = px.BF16
    theta = torch.from_numpy(inp.theta_P).cuda()
    blocks = torch.empty((d // b, b, b), dtype=torch.bfloat16, device="cuda")
    wsz = max(px.poetx_build_workspace_size(d, b, k, c),
              px.poetx_transform_workspace_size(d, b, k, T, c))
    ws = torch.empty((wsz,), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(inp.x).cuda().to(torch.bfloat16)
    dout = torch.from_numpy(inp.dy).cuda().to(torch.bfloat16)
    out = torch.empty_like(x)
    dx = torch.empty_like(x)
    dtheta = torch.empty((d // b, b * (b - 1) // 2), dtype=torch.float32, device="cuda")
    px.poetx_build_blocks(theta, d, b, k, c, blocks, ws)
    px.poetx_transform_forward(x, blocks, out, d, b, T, c, ws)
    px.poetx_transform_backward(dout, x, theta, blocks, dx, dtheta, d, b, k, T, c, ws)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    rng = np.random.default_rng(2)
    rows = tile_rows(T, rng)
    B = oracle.build_blocks(inp.theta_P, b, k)
    idx = torch.from_numpy(rows).cuda()
    z_got = out.index_select(0, idx).float().cpu().numpy()
    z_ref = oracle.apply_blockdiag(inp.x[rows], B)
    dx_got = dx.index_select(0, idx).float().cpu().numpy()
    dx_ref = oracle.apply_blockdiag_transposed(inp.dy[rows], B)
    errs = {"z": rel_fro(z_got, z_ref), "dx": rel_fro(dx_got, dx_ref),
            "z max row": max_row_rel(z_got, z_ref), "dx max row": max_row_rel(dx_got, dx_ref)}
    Q = oracle.unpack(inp.theta_P, b)
    n = d // b
    dth = dtheta.cpu().numpy()
    for g in sorted({0, n // 2, n - 1}):
        sl = slice(g * b, (g + 1) * b)
        G = oracle.blockwise_outer(inp.dy[:, sl], inp.x[:, sl], b)
        want = oracle.pack_skew_grad(oracle.cnp_adjoint(Q[g:g + 1], G, k))[0]
        errs[f"dtheta[{g}]"] = rel_fro(dth[g], want)
    bad = {n_: e for n_, e in errs.items() if not e <= (TOL_ROW if "max row" in n_ else TOL)}
    assert not bad, f"above tolerance: {bad} (all: {errs})"
