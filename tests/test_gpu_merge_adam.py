"""GPU parity of the two calls around the layer step: the merge
W0 <- R W0 P with the factor reset, and the Adam update of the packed
parameters, against the float64 oracle.

Tolerances: merge 1e-4 relative Frobenius in fp32; in bf16 the blocks, the
intermediate W0 P and the result are each rounded to bf16 once, so 1e-2.
Adam: fp32 arithmetic, 1e-5 relative per element plus 2e-7 of the array's
largest magnitude (the moment updates cancel, so their rounding error scales
with the terms rather than with the result).
"""

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


def check_status(px):
    torch.cuda.synchronize()
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)


MERGE_CASES = [
    # (d_in, d_out, b, k, dtype)
    (512, 768, 256, 3, "bf16"),
    (512, 256, 128, 2, "bf16"),
    (256, 512, 32, 5, "bf16"),
    (1024, 512, 512, 1, "bf16"),
    (256, 256, 32, 3, "f32"),
    (96, 48, 3, 2, "f32"),
]


@pytest.mark.parametrize("d_in,d_out,b,k,dtype", MERGE_CASES)
def test_merge_matches_oracle_and_resets_theta(px, d_in, d_out, b, k, dtype):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    inp = make_layer_inputs(d_in, d_out, b, k, 16, dtype=dtype, sigma_theta=0.03, seed=31)
    dev = to_device(inp)
    layer = PoetxLayer(d_in, d_out, b, k, 16, dtype=dtype)
    layer.build(dev["theta_P"], dev["theta_R"])
    W0 = dev["W0"].clone()
    layer.merge(W0, dev["theta_P"], dev["theta_R"])
    check_status(px)
    want = oracle.merge(inp.theta_P, inp.theta_R, inp.W0, b, k)
    tol = 1e-2 if dtype == "bf16" else 1e-4
    assert rel_fro(W0.float().cpu().numpy(), want) <= tol
    assert torch.count_nonzero(dev["theta_P"]) == 0
    assert torch.count_nonzero(dev["theta_R"]) == 0


def test_merge_into_a_separate_output_keeps_theta(px):
    inp = make_layer_inputs(512, 512, 256, 3, 16, dtype="bf16", sigma_theta=0.03, seed=32)
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    dev = to_device(inp)
    layer = PoetxLayer(512, 512, 256, 3, 16)
    layer.build(dev["theta_P"], dev["theta_R"])
    W0 = dev["W0"].clone()
    out = torch.empty_like(W0)
    px.poetx_merge(W0, layer.P_blocks, layer.R_blocks, out, None, None, 512, 512, 256, px.BF16,
                   layer.workspace)
    check_status(px)
    assert torch.equal(W0, dev["W0"])  # the input weight is untouched
    assert torch.count_nonzero(dev["theta_P"]) > 0
    want = oracle.merge(inp.theta_P, inp.theta_R, inp.W0, 256, 3)
    assert rel_fro(out.float().cpu().numpy(), want) <= 1e-2


def test_step_after_merge_matches_the_unmerged_layer(px):
    # After the merge the factors restart at I: the merged layer's output
    # equals the pre-merge layer's output (the method's invariant).
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    inp = make_layer_inputs(256, 256, 32, 4, 64, dtype="f32", sigma_theta=0.02, seed=33)
    dev = to_device(inp)
    layer = PoetxLayer(256, 256, 32, 4, 64, dtype="f32")
    layer.build(dev["theta_P"], dev["theta_R"])
    y_before = layer.forward(dev["x"], dev["W0"]).clone()
    layer.merge(dev["W0"], dev["theta_P"], dev["theta_R"])
    layer.build(dev["theta_P"], dev["theta_R"])
    y_after = layer.forward(dev["x"], dev["W0"])
    check_status(px)
    assert rel_fro(y_after.cpu().numpy(), y_before.cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("n,wd", [(1, 0.0), (1000, 0.0), (123457, 0.1)])
def test_adam_two_steps_match_oracle(px, n, wd):
    rng = np.random.default_rng(34)
    theta = rng.standard_normal(n) * 0.1
    g1 = rng.standard_normal(n)
    g2 = rng.standard_normal(n) * 0.5
    t = torch.from_numpy(theta.astype(np.float32)).cuda()
    m = torch.zeros_like(t)
    v = torch.zeros_like(t)
    want_t, want_m, want_v = theta.astype(np.float32), np.zeros(n), np.zeros(n)
    # the hyperparameters cross the C ABI as float32: give the oracle the same values
    f32 = lambda a: float(np.float32(a))  # noqa: E731
    lr, b1, b2, eps, wd32 = f32(1e-3), f32(0.9), f32(0.999), f32(1e-8), f32(wd)
    for step, g in ((1, g1), (2, g2)):
        gd = torch.from_numpy(g.astype(np.float32)).cuda()
        px.poetx_adam_update(t, gd, m, v, n, step, lr, b1, b2, eps, wd32)
        want_t, want_m, want_v = oracle.adam_update(want_t, g.astype(np.float32), want_m,
                                                    want_v, step, lr, beta1=b1, beta2=b2,
                                                    eps=eps, weight_decay=wd32)
    check_status(px)
    for got, want in ((t, want_t), (m, want_m), (v, want_v)):
        got = got.cpu().numpy().astype(np.float64)
        # m = b1 m + (1-b1) g cancels: its fp32 error scales with the terms, not the sum
        scale = np.max(np.abs(want))
        assert np.all(np.abs(got - want) <= 1e-5 * np.abs(want) + 2e-7 * scale)


def test_adam_rejects_bad_arguments(px):
    t = torch.zeros(4, device="cuda")
    with pytest.raises(px.PoetxError):
        px.poetx_adam_update(t, t, t, t, 4, 0, 1e-3)
    with pytest.raises(px.PoetxError):
        px.poetx_adam_update(t, t, t, t, 4, 1, 1e-3, beta1=1.0)
    px.poetx_adam_update(t, t, t, t, 0, 1, 1e-3)  # empty: nothing to do
