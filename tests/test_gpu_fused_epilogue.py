"""The W0 GEMMs with the block-diagonal factor in their epilogues (y = R v
in the forward GEMM, dx = du P in the dgrad GEMM), on CTA pairs and on the
one-SM cluster form: parity with the oracle at the layer tolerances, and
agreement with the unfused path.  v, and hence y and everything on the R
side, has the same bits: the block product runs on the same bf16-rounded
tile whether it comes from HBM or from the staging tile.  The P side's token
sums run apart from the transform when the dgrad GEMM applies P, with
another K split over tokens, so dtheta_P agrees to fp32 summation order
(carried through the bf16 operands of the block-build adjoint).  The
unfused GEMM's K split of its last round is off, so that both sum every
tile's K steps in the same order."""

import numpy as np
import pytest

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


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


def run(px, inp, fused, recompute_v=False, pair=True):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    dev = to_device(inp)
    layer = PoetxLayer(inp.d_in, inp.d_out, inp.b, inp.k, inp.tokens, dtype=inp.dtype,
                       recompute_v=recompute_v)
    prev = px.poetx_set_block_epilogue_fusion(fused)
    prev_split = px.poetx_set_w0_split_tail(False)
    prev_pair = px.poetx_set_w0_pair_mma(pair)
    try:
        layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"])
        torch.cuda.synchronize()
    finally:
        px.poetx_set_block_epilogue_fusion(prev)
        px.poetx_set_w0_split_tail(prev_split)
        px.poetx_set_w0_pair_mma(prev_pair)
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)
    return layer


CASES = [(512, 768, 256, 3, 333), (256, 512, 128, 2, 130), (512, 256, 64, 3, 257),
         (256, 256, 32, 3, 64), (256, 256, 256, 5, 1), (768, 512, 256, 3, 1000),
         (4096, 4096, 256, 3, 2048)]


def max_row_rel(got, want):
    num = np.linalg.norm(got - want, axis=1)
    return float(np.max(num / np.maximum(np.linalg.norm(want, axis=1), 1e-300)))


@pytest.mark.parametrize("pair", [True, False], ids=["pair", "cluster"])
@pytest.mark.parametrize("d_in,d_out,b,k,T", CASES)
def test_fused_epilogue_matches_oracle_and_unfused(px, d_in, d_out, b, k, T, pair):
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype="bf16", seed=60)
    fused = run(px, inp, True, pair=pair)
    plain = run(px, inp, False, pair=pair)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, b, k)
    n_in, n_out = d_in // b, d_out // b
    for name in ("y", "dtheta_R"):
        assert torch.equal(getattr(fused, name), getattr(plain, name)), name
    for name, bound in (("dx", 2e-3), ("dtheta_P", 1e-2)):
        g, h = getattr(fused, name).float(), getattr(plain, name).float()
        rel = float(torch.linalg.norm(g - h) / torch.linalg.norm(h))
        assert rel <= bound, (name, rel)
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        got = getattr(fused, name).float().cpu().numpy().astype(np.float64)
        want = ref[name]
        if name == "dtheta_P":
            got = got.reshape(n_in, -1)
        if name == "dtheta_R":
            got = got.reshape(n_out, -1)
        assert rel_fro(got, want) <= 2e-2, name
        assert max_row_rel(got, want) <= 4e-2, name


@pytest.mark.parametrize("pair", [True, False], ids=["pair", "cluster"])
def test_fused_forward_without_saved_v(px, pair):
    inp = make_layer_inputs(512, 512, 256, 3, 200, dtype="bf16", seed=61)
    fused = run(px, inp, True, recompute_v=True, pair=pair)
    plain = run(px, inp, False, recompute_v=False, pair=pair)
    for name in ("y", "dtheta_R"):
        assert torch.equal(getattr(fused, name), getattr(plain, name)), name
    for name, bound in (("dx", 2e-3), ("dtheta_P", 1e-2)):
        g, h = getattr(fused, name).float(), getattr(plain, name).float()
        assert float(torch.linalg.norm(g - h) / torch.linalg.norm(h)) <= bound, name


def test_switch_is_off_by_default_and_returns_previous(px):
    prev = px.poetx_set_block_epilogue_fusion(True)
    assert px.poetx_set_block_epilogue_fusion(prev) is True
    assert prev is False
