"""GPU parity: the CUDA library, called through its C ABI, against the
float64 oracle on the same seeded inputs.

Tolerances (relative Frobenius error unless stated):
  * packed-index / unpack mapping: bit-exact;
  * fp32 mode: 1e-4 on y, dx, dtheta; 1e-6 on the built blocks (fp32 FFMA
    over at most b = 512 terms per product, k <= 5 products);
  * bf16 mode (fp32 accumulate): 2e-2 on y, dx, dtheta; blocks are stored
    in bf16, so they are compared at 2^-8 (one bf16 rounding of a value
    plus the bf16 rounding of the intermediate E matrices).
"""

import numpy as np
import pytest

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import (bf16_bits, make_layer_inputs,
                                                            round_to_bf16)

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
TOL_BLOCKS = {"f32": 1e-6, "bf16": 2.0 ** -8}


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


def tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def code(px, dtype):
    return px.BF16 if dtype == "bf16" else px.F32


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def dev_act(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda().to(tdt(dtype)).contiguous()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def ws_tensor(nbytes):
    return torch.empty((max(int(nbytes), 16),), dtype=torch.uint8, device="cuda")


def check_status(px):
    torch.cuda.synchronize()
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)


def build(px, theta, d, b, k, dtype):
    c = code(px, dtype)
    blocks = torch.empty((d // b, b, b), dtype=tdt(dtype), device="cuda")
    ws = ws_tensor(px.poetx_build_workspace_size(d, b, k, c))
    px.poetx_build_blocks(dev_f32(theta), d, b, k, c, blocks, ws)
    return blocks


# ------------------------------------------------------------ unpack map

def _enumerated_q(theta, b):
    """Skew Q from packed theta by walking the strict upper triangle row by
    row (independent of both the oracle and the kernel's index formula)."""
    n = theta.shape[0]
    Q = np.zeros((n, b, b), dtype=np.float32)
    ii, jj = np.triu_indices(b, 1)  # row-major order of the strict upper triangle
    Q[:, ii, jj] = theta
    Q[:, jj, ii] = -theta
    return Q


@pytest.mark.parametrize("dtype,d,b", [("f32", 40, 2), ("f32", 15, 5), ("f32", 256, 32),
                                       ("f32", 512, 256), ("bf16", 512, 32),
                                       ("bf16", 512, 128), ("bf16", 512, 256),
                                       ("bf16", 1024, 512)])
def test_unpack_is_bit_exact(px, dtype, d, b):
    # k = 0 blocks are I + Q: every entry is a copy of a packed value (or
    # its negation, or 1 on the diagonal), so the map must be bit-exact.
    rng = np.random.default_rng(20)
    theta = (rng.standard_normal((d // b, b * (b - 1) // 2)) * 0.05).astype(np.float32)
    blocks = build(px, theta, d, b, 0, dtype)
    check_status(px)
    want = _enumerated_q(theta, b) + np.eye(b, dtype=np.float32)
    if dtype == "f32":
        got = blocks.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    else:
        got = blocks.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, bf16_bits(round_to_bf16(want)))


# --------------------------------------------------------------- builder

@pytest.mark.parametrize("dtype,d,b,k", [
    ("f32", 256, 32, 3), ("f32", 512, 256, 3), ("f32", 64, 8, 5), ("f32", 96, 3, 1),
    ("bf16", 512, 32, 5), ("bf16", 512, 64, 3), ("bf16", 512, 128, 1), ("bf16", 512, 128, 3),
    ("bf16", 1024, 256, 3), ("bf16", 1024, 256, 5), ("bf16", 1024, 512, 3),
    ("bf16", 1024, 512, 1), ("bf16", 512, 256, 10), ("bf16", 512, 128, 0),
    ("bf16", 512, 256, 16), ("f32", 64, 8, 16), ("bf16", 768, 256, 8),  # k = 16: the maximum
    # b <= 256: the CTA-pair builds (256 x 256 superblocks; k = 3 and any other k)
    ("bf16", 256, 32, 3), ("bf16", 768, 64, 3), ("bf16", 2048, 128, 3), ("bf16", 4096, 256, 3),
    ("bf16", 512, 64, 1), ("bf16", 256, 32, 2), ("bf16", 1024, 64, 5), ("bf16", 768, 128, 4),
    ("bf16", 4096, 256, 6)])
def test_build_blocks_matches_oracle(px, dtype, d, b, k):
    rng = np.random.default_rng(21)
    theta = (rng.standard_normal((d // b, b * (b - 1) // 2)) * 0.02).astype(np.float32)
    blocks = build(px, theta, d, b, k, dtype)
    check_status(px)
    want = oracle.build_blocks(theta, b, k)
    assert rel_fro(to_np(blocks), want) <= TOL_BLOCKS[dtype]


# --------------------------------------------- isolated block transform

TRANSFORM_CASES = [
    ("bf16", 1024, 32, 5, 300), ("bf16", 1024, 64, 3, 300), ("bf16", 1024, 128, 1, 300),
    ("bf16", 1024, 256, 3, 300), ("bf16", 1024, 512, 3, 300), ("bf16", 512, 256, 0, 129),
    ("bf16", 1536, 512, 1, 37), ("bf16", 2048, 512, 5, 513),  # 512-blocks on CTA pairs
    ("f32", 256, 32, 3, 300), ("f32", 96, 3, 2, 50),
    ("f32", 256, 32, 3, 37),  # fp32 token sums over one partial 64-token chunk
]


@pytest.mark.parametrize("dtype,d,b,k,T", TRANSFORM_CASES)
def test_transform_matches_oracle(px, dtype, d, b, k, T):
    inp = make_layer_inputs(d, d, b, k, T, dtype=dtype, seed=22)
    c = code(px, dtype)
    blocks = build(px, inp.theta_P, d, b, k, dtype)
    x = dev_act(inp.x, dtype)
    dout = dev_act(inp.dy, dtype)
    out = torch.empty_like(x)
    dx = torch.empty_like(x)
    dtheta = torch.empty((d // b, b * (b - 1) // 2), dtype=torch.float32, device="cuda")
    ws = ws_tensor(px.poetx_transform_workspace_size(d, b, k, T, c))
    px.poetx_transform_forward(x, blocks, out, d, b, T, c, ws)
    px.poetx_transform_backward(dout, x, dev_f32(inp.theta_P), blocks, dx, dtheta, d, b, k, T,
                                c, ws)
    check_status(px)
    ref = oracle.transform(inp.theta_P, inp.x, inp.dy, b, k)
    assert rel_fro(to_np(out), ref["z"]) <= TOL[dtype]
    assert rel_fro(to_np(dx), ref["dx"]) <= TOL[dtype]
    assert rel_fro(to_np(dtheta), ref["dtheta"]) <= TOL[dtype]


# ----------------------------------------------------------- whole layer

def run_layer(px, inp, recompute_v=False):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    dev = to_device(inp)
    layer = PoetxLayer(inp.d_in, inp.d_out, inp.b, inp.k, inp.tokens, dtype=inp.dtype,
                       recompute_v=recompute_v)
    layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"])
    check_status(px)
    return layer


def max_row_rel(got, want):
    """Largest relative error of one row (a token of y / dx, a block of
    dtheta): a fault confined to one tile cannot average away in it."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if want.shape[0] == 0:
        return 0.0
    num = np.linalg.norm(got - want, axis=1)
    den = np.maximum(np.linalg.norm(want, axis=1), 1e-300)
    return float(np.max(num / den))


# Per-row and per-block maximum: twice the Frobenius tolerance (a row of
# d >= 48 rounded values has almost the spread of the whole array).
TOL_ROW = {"f32": 2e-4, "bf16": 4e-2}


def compare_layer(layer, ref, dtype, rows=None):
    n_in = layer.d_in // layer.b
    n_out = layer.d_out // layer.b
    got = dict(y=to_np(layer.y), dx=to_np(layer.dx),
               dtheta_P=to_np(layer.dtheta_P).reshape(n_in, -1),
               dtheta_R=to_np(layer.dtheta_R).reshape(n_out, -1))
    errs = {}
    for name, g in got.items():
        errs[name] = rel_fro(g, ref[name])
    bad = {n: e for n, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"errors above {TOL[dtype]}: {bad} (all: {errs})"
    rows_err = {name: max_row_rel(g, ref[name]) for name, g in got.items()}
    bad = {n: e for n, e in rows_err.items() if not e <= TOL_ROW[dtype]}
    assert not bad, f"row / block errors above {TOL_ROW[dtype]}: {bad} (all: {rows_err})"


LAYER_CASES = [
    # (d_in, d_out, b, k, T, dtype)
    (256, 256, 32, 3, 512, "f32"),      # the single-layer fp32 workload, full size
    (96, 48, 3, 2, 37, "f32"),
    (512, 768, 256, 3, 333, "bf16"),
    (256, 512, 128, 2, 130, "bf16"),
    (1024, 512, 512, 1, 200, "bf16"),
    (512, 256, 64, 3, 257, "bf16"),
    (256, 256, 32, 0, 64, "bf16"),
    (256, 256, 256, 5, 1, "bf16"),
    (256, 256, 256, 3, 127, "bf16"),
    (256, 512, 128, 9, 64, "bf16"),      # k above the one-launch chain limit
    (512, 256, 256, 16, 40, "bf16"),     # the largest k
    (64, 32, 8, 16, 20, "f32"),
    (256, 256, 64, 3, 300, "f32"),      # fp32 token sums split over 4 CTAs, ragged ranges
    (96, 192, 32, 3, 200, "f32"),       # one token-sum launch over 3 P blocks and 6 R blocks
    # the fused fp32 W0 GEMM's other block sizes: ragged K step (48 = 1.5 steps),
    # ragged N tile, ragged token tile; a K slice boundary inside a 64-block
    (48, 80, 16, 3, 70, "f32"),
    (32, 64, 4, 2, 45, "f32"),
    (16, 8, 2, 1, 33, "f32"),
    (192, 64, 64, 2, 100, "f32"),
    (512, 256, 256, 0, 70, "bf16"),
    # the CTA-pair adjoint for k != 3 (Horner form), every block size
    (512, 256, 32, 5, 100, "bf16"),
    (256, 512, 64, 1, 70, "bf16"),
    (768, 512, 128, 4, 150, "bf16"),
    (512, 512, 256, 2, 96, "bf16"),
]


@pytest.mark.parametrize("d_in,d_out,b,k,T,dtype", LAYER_CASES)
def test_layer_matches_oracle(px, d_in, d_out, b, k, T, dtype):
    sigma = 0.01 if dtype == "f32" and b == 32 else 0.02
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, sigma_theta=sigma, seed=0)
    layer = run_layer(px, inp)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, b, k)
    compare_layer(layer, ref, dtype)


RECOMPUTE_CASES = [
    (256, 256, 32, 3, 512, "f32"),
    (48, 80, 16, 3, 70, "f32"),
    (512, 768, 256, 3, 333, "bf16"),
    (256, 512, 128, 2, 130, "bf16"),
    (512, 256, 64, 3, 257, "bf16"),
    (1024, 512, 512, 1, 200, "bf16"),
]


@pytest.mark.parametrize("d_in,d_out,b,k,T,dtype", RECOMPUTE_CASES)
def test_layer_recompute_v_matches_oracle(px, d_in, d_out, b, k, T, dtype):
    # POET-Xmem: the backward recomputes v = W0 P x instead of reading it
    sigma = 0.01 if dtype == "f32" and b == 32 else 0.02
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, sigma_theta=sigma, seed=8)
    layer = run_layer(px, inp, recompute_v=True)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, b, k)
    compare_layer(layer, ref, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_recompute_v_gives_identical_results(px, dtype):
    b = 256 if dtype == "bf16" else 32
    inp = make_layer_inputs(512, 256, b, 3, 200, dtype=dtype, seed=3)
    a = run_layer(px, inp, recompute_v=False)
    r = run_layer(px, inp, recompute_v=True)
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        assert torch.equal(getattr(a, name), getattr(r, name)), name


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_zero_tokens(px, dtype):
    b = 256 if dtype == "bf16" else 32
    inp = make_layer_inputs(256, 512, b, 3, 0, dtype=dtype, seed=4)
    layer = run_layer(px, inp)
    assert torch.count_nonzero(layer.dtheta_P) == 0
    assert torch.count_nonzero(layer.dtheta_R) == 0


def test_zero_theta_is_plain_linear(px):
    inp = make_layer_inputs(512, 256, 256, 3, 100, dtype="bf16", seed=5)
    inp.theta_P[:] = 0
    inp.theta_R[:] = 0
    layer = run_layer(px, inp)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, 256, 3)
    # blocks are exactly I in bf16
    eye = torch.eye(256, dtype=torch.bfloat16, device="cuda").expand(2, 256, 256)
    assert torch.equal(layer.P_blocks, eye)
    compare_layer(layer, ref, "bf16")


def test_deterministic(px):
    inp = make_layer_inputs(512, 512, 256, 3, 300, dtype="bf16", seed=6)
    a = run_layer(px, inp)
    b = run_layer(px, inp)
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("dtype,b", [("bf16", 256), ("bf16", 64), ("f32", 32)])
def test_one_call_build_equals_two_calls(px, dtype, b):
    # theta_P and theta_R back to back are built by one call over d_in + d_out
    # features; the blocks must be bitwise those of two separate calls.
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, adjacent, to_device
    inp = make_layer_inputs(512, 768, b, 3, 8, dtype=dtype, seed=7)
    dev = to_device(inp)
    assert adjacent(dev["theta_P"], dev["theta_R"]) is not None
    one = PoetxLayer(512, 768, b, 3, 8, dtype=dtype)
    one.build(dev["theta_P"], dev["theta_R"])
    two = PoetxLayer(512, 768, b, 3, 8, dtype=dtype)
    tP, tR = dev["theta_P"].clone(), dev["theta_R"].clone()
    assert adjacent(tP, tR) is None
    two.build(tP, tR)
    check_status(px)
    assert torch.equal(one.blocks, two.blocks)


@pytest.mark.parametrize("b,k", [(256, 3), (64, 5), (512, 3)])
def test_block_stack_builds_every_projection_in_one_call(px, b, k):
    # a model's factors built by one call equal each projection built alone
    from orthogonal_reparameterized_packed_gb300.layer import BlockStack, PoetxLayer
    shapes = [(512, 1024), (1024, 512), (512, 512)]
    stack = BlockStack(shapes, b, k, dtype="bf16")
    rng = np.random.default_rng(70 + b + k)
    stack.theta.copy_(torch.from_numpy(
        (rng.standard_normal(stack.theta.numel()) * 0.02).astype(np.float32)))
    stack.build()
    for i, (di, do) in enumerate(shapes):
        lay = PoetxLayer(di, do, b, k, 8, dtype="bf16")
        lay.build(*stack.theta_views(i))
        check_status(px)
        P, R = stack.block_views(i)
        assert torch.equal(P, lay.P_blocks) and torch.equal(R, lay.R_blocks), i
