"""The W0 GEMM with the block-diagonal factor in its epilogue (opt-in):
parity with the oracle at the layer tolerances, and the same bits as the
unfused path (the block product runs the same MMA sequence on the same
bf16-rounded tile, whether it comes from HBM or from the staging tile).
The bit comparison runs with the unfused GEMM's K split of its last round
off, so that both sum every tile's K steps in the same order."""

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


def run(px, inp, fused, recompute_v=False):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    dev = to_device(inp)
    layer = PoetxLayer(inp.d_in, inp.d_out, inp.b, inp.k, inp.tokens, dtype=inp.dtype,
                       recompute_v=recompute_v)
    prev = px.poetx_set_block_epilogue_fusion(fused)
    prev_split = px.poetx_set_w0_split_tail(False)
    try:
        layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"])
        torch.cuda.synchronize()
    finally:
        px.poetx_set_block_epilogue_fusion(prev)
        px.poetx_set_w0_split_tail(prev_split)
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)
    return layer


CASES = [(512, 768, 256, 3, 333), (256, 512, 128, 2, 130), (512, 256, 64, 3, 257),
         (256, 256, 32, 3, 64), (256, 256, 256, 5, 1), (768, 512, 256, 3, 1000)]


@pytest.mark.parametrize("d_in,d_out,b,k,T", CASES)
def test_fused_epilogue_matches_oracle_and_unfused_bits(px, d_in, d_out, b, k, T):
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype="bf16", seed=60)
    fused = run(px, inp, True)
    plain = run(px, inp, False)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, b, k)
    n_in, n_out = d_in // b, d_out // b
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        g = getattr(fused, name)
        assert torch.equal(g, getattr(plain, name)), name
        want = ref[name]
        got = g.float().cpu().numpy()
        if name == "dtheta_P":
            got = got.reshape(n_in, -1)
        if name == "dtheta_R":
            got = got.reshape(n_out, -1)
        assert rel_fro(got, want) <= 2e-2, name


def test_fused_forward_without_saved_v(px):
    inp = make_layer_inputs(512, 512, 256, 3, 200, dtype="bf16", seed=61)
    fused = run(px, inp, True, recompute_v=True)
    plain = run(px, inp, False, recompute_v=False)
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        assert torch.equal(getattr(fused, name), getattr(plain, name)), name


def test_switch_is_off_by_default_and_returns_previous(px):
    prev = px.poetx_set_block_epilogue_fusion(True)
    assert px.poetx_set_block_epilogue_fusion(prev) is True
    assert prev is False
