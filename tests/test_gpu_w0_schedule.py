"""The W0 GEMMs' forms: CTA pairs with one 256-row MMA across two SMs (the
default, poetx_set_w0_pair_mma), or clusters of two one-SM MMAs whose last
partial round of tiles may be spread one per cluster with the K steps split
between the cluster's two CTAs (poetx_set_w0_split_tail).  Shapes are chosen so that, on a GPU with
about 70-80 clusters of two, every kind of schedule occurs: all tiles split
(few tiles), whole units plus a split last round, and no split (a last
round more than half full).  With theta = 0 the blocks are exactly I, so
y = x W0^T and dx = dy W0 (each rounded once to bf16), checked element by
element against the float64 oracle's layer; the split and unsplit schedules
agree to fp32 summation order."""

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


# the W0 GEMM forms: (pair MMA, split last round of the cluster form)
MODES = {"pair": (True, True), "split": (False, True), "unsplit": (False, False)}


def run(px, inp, mode):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    pair, split = MODES[mode]
    dev = to_device(inp)
    layer = PoetxLayer(inp.d_in, inp.d_out, inp.b, inp.k, inp.tokens, dtype=inp.dtype)
    prev = px.poetx_set_w0_split_tail(split)
    prev_pair = px.poetx_set_w0_pair_mma(pair)
    try:
        layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"])
        torch.cuda.synchronize()
    finally:
        px.poetx_set_w0_split_tail(prev)
        px.poetx_set_w0_pair_mma(prev_pair)
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)
    return layer, dev


def check_plain_linear(got, want):
    # one rounding of an fp32 sum to bf16: within 2^-8 relative, plus the
    # fp32 summation error (far below that)
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    bound = np.abs(want) * 2.0 ** -8 + 1e-5 * float(np.abs(want).max())
    assert bool((err <= bound).all()), float((err - bound).max())


# T, d_in, d_out: (128-row tiles, 256-wide N tiles, pairs of M tiles per cluster)
SHAPES = [
    (129, 512, 1024),     # 1 pair x 4 N tiles: every tile split
    (333, 768, 512),      # ragged: 3 M tiles (the second pair's second tile is empty)
    (1024, 4096, 4096),   # 64 units: one round, more than half full, no split
    (1280, 4096, 4096),   # 80 units: one round plus a split last round of 4
    (2560, 1024, 2048),   # forward 10 pairs x 8 N tiles = 80 units (split); dgrad 40 (none)
]


@pytest.mark.parametrize("T,d_in,d_out", SHAPES + [(1, 256, 256), (255, 256, 512),
                                                   (257, 512, 256)])
@pytest.mark.parametrize("mode", sorted(MODES))
def test_zero_theta_layer_is_the_plain_linear_map(px, T, d_in, d_out, mode):
    inp = make_layer_inputs(d_in, d_out, 256, 3, T, dtype="bf16", seed=80)
    inp.theta_P[:] = 0
    inp.theta_R[:] = 0
    layer, dev = run(px, inp, mode)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, 256, 3)
    check_plain_linear(layer.y, ref["y"])
    check_plain_linear(layer.dx, ref["dx"])


@pytest.mark.parametrize("T,d_in,d_out", [(129, 512, 1024), (1280, 4096, 4096),
                                          (16384, 4096, 4096)])
@pytest.mark.parametrize("mode", ["split", "pair"])
def test_schedules_agree(px, T, d_in, d_out, mode):
    inp = make_layer_inputs(d_in, d_out, 256, 3, T, dtype="bf16", seed=81)
    a, _ = run(px, inp, mode)
    b, _ = run(px, inp, "unsplit")
    # v and du (bf16 roundings of fp32 sums in two orders) differ in a few
    # elements by one bf16 step; y and dx carry that through a block product
    for name, bound in (("y", 2e-3), ("dx", 2e-3), ("dtheta_P", 1e-2), ("dtheta_R", 1e-2)):
        ga, gb = getattr(a, name).float(), getattr(b, name).float()
        rel = float(torch.linalg.norm(ga - gb) / torch.linalg.norm(gb))
        assert rel < bound, (name, rel)
