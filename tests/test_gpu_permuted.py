"""Permuted block-diagonal factors (R = Pi_R^T B_R Pi_R, P = Pi_P^T B_P Pi_P)
through the C ABI: the weight fold, the activation index maps and a whole
permuted step against the dense-permutation-matrix oracle.  Index maps are
bit-exact; the step uses the layer tolerances (1e-4 fp32, 2e-2 bf16)."""

import numpy as np
import pytest

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_index_maps_are_exact(px, dtype):
    rng = np.random.default_rng(40)
    T, d = 37, 1024
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = px.BF16 if dtype == "bf16" else px.F32
    x = torch.randn((T, d), device="cuda").to(tdt)
    perm = rng.permutation(d).astype(np.int32)
    out = torch.empty_like(x)
    px.poetx_permute_features(x, torch.from_numpy(perm).cuda(), out, T, d, code)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    assert torch.equal(out, x[:, torch.from_numpy(perm).long().cuda()])
    # fold: W'[i][j] = W[perm_out[i]][perm_in[j]]
    W = torch.randn((512, d), device="cuda").to(tdt)
    po = rng.permutation(512).astype(np.int32)
    Wf = torch.empty_like(W)
    px.poetx_fold_permutations(W, torch.from_numpy(po).cuda(), torch.from_numpy(perm).cuda(), Wf,
                               d, 512, code)
    torch.cuda.synchronize()
    want = W[torch.from_numpy(po).long().cuda()][:, torch.from_numpy(perm).long().cuda()]
    assert torch.equal(Wf, want)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d,T", [(8, 5), (9552, 13), (9560, 7), (14336, 11), (14344, 6),
                                 (28672, 9)],
                         ids=["tiny", "bulk-max", "two-tables", "two-tables-max", "one-table",
                              "max"])
def test_index_maps_at_every_kernel_form(px, d, T, dtype):
    """Rows whose two staged groups and table fit shared memory (d <= 9556)
    move by bulk copies; wider rows are read straight into one or two
    tables by producer warps."""
    if dtype == "f32" and d % 4:
        pytest.skip("rows must be a multiple of 16 bytes")
    rng = np.random.default_rng(d + T)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = px.BF16 if dtype == "bf16" else px.F32
    x = torch.randn((T, d), device="cuda").to(tdt)
    perm = torch.from_numpy(rng.permutation(d).astype(np.int32)).cuda()
    out = torch.empty_like(x)
    px.poetx_permute_features(x, perm, out, T, d, code)
    # the fold: rows through a map too, fewer rows than a CTA's group at the end
    rows = 7
    W = torch.randn((rows, d), device="cuda").to(tdt)
    po = torch.from_numpy(rng.permutation(rows).astype(np.int32)).cuda()
    Wf = torch.empty_like(W)
    px.poetx_fold_permutations(W, po, perm, Wf, d, rows, code)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    assert torch.equal(out, x[:, perm.long()])
    assert torch.equal(Wf, W[po.long()][:, perm.long()])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1, 2, 3, 6])
def test_index_maps_over_fewer_rows_than_a_group(px, T, dtype):
    """A group is four bf16 (two fp32) rows; shorter and ragged row counts."""
    rng = np.random.default_rng(T)
    d = 4096
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = px.BF16 if dtype == "bf16" else px.F32
    x = torch.randn((T, d), device="cuda").to(tdt)
    perm = torch.from_numpy(rng.permutation(d).astype(np.int32)).cuda()
    out = torch.full_like(x, 7.0)
    px.poetx_permute_features(x, perm, out, T, d, code)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    assert torch.equal(out, x[:, perm.long()])


@pytest.mark.parametrize("d", [256, 14336], ids=["bulk", "two-tables"])
def test_out_of_range_row_map_entries_give_zero_rows(px, d):
    rows = 6
    W = torch.randn((rows, d), device="cuda").to(torch.bfloat16)
    po = np.array([3, -1, 0, 6, 5, 1], dtype=np.int32)  # -1 and 6: out of range
    perm = torch.arange(d, dtype=torch.int32, device="cuda").flip(0).contiguous()
    Wf = torch.full_like(W, 7.0)
    px.poetx_fold_permutations(W, torch.from_numpy(po).cuda(), perm, Wf, d, rows, px.BF16)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 1  # POETX_ERR_INVALID_ARG recorded
    for i, r in enumerate(po):
        want = W[r].flip(0) if 0 <= r < rows else torch.zeros_like(W[0])
        assert torch.equal(Wf[i], want), i


def test_out_of_range_map_entries_are_not_followed(px):
    x = torch.randn((4, 256), device="cuda").to(torch.bfloat16)
    perm = np.arange(256, dtype=np.int32)
    perm[5] = 999  # out of range
    out = torch.full_like(x, 7.0)
    px.poetx_permute_features(x, torch.from_numpy(perm).cuda(), out, 4, 256, px.BF16)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 1  # POETX_ERR_INVALID_ARG recorded
    assert torch.all(out[:, 5] == 0)
    assert torch.equal(out[:, :5], x[:, :5])


@pytest.mark.parametrize("d_in,d_out,b,k,T,dtype", [
    (512, 768, 256, 3, 200, "bf16"),
    (256, 512, 128, 2, 130, "bf16"),
    (256, 256, 32, 3, 96, "f32"),
])
def test_permuted_step_matches_oracle(px, d_in, d_out, b, k, T, dtype):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxPermutedLayer, to_device
    rng = np.random.default_rng(41)
    perm_P, perm_R = rng.permutation(d_in), rng.permutation(d_out)
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, seed=42)
    dev = to_device(inp)
    layer = PoetxPermutedLayer(d_in, d_out, b, k, T, perm_P, perm_R, dtype=dtype)
    layer.fold(dev["W0"])
    layer.step(dev["theta_P"], dev["theta_R"], dev["x"], dev["dy"])
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    ref = oracle.layer_permuted(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, b, k,
                                perm_P, perm_R)
    got = dict(y=layer.y, dx=layer.dx,
               dtheta_P=layer.dtheta_P.view(d_in // b, -1),
               dtheta_R=layer.dtheta_R.view(d_out // b, -1))
    errs = {n: rel_fro(t.float().cpu().numpy(), ref[n]) for n, t in got.items()}
    assert all(e <= TOL[dtype] for e in errs.values()), errs
