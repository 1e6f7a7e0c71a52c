"""GPU parity of the INT8 frozen weight (POET-XQ): codes, scales and the
dequantised weight are bit-exact against the oracle (both take the deciding
division and the dequantising product in float32); the layer step on the
dequantised weight is within the layer tolerances (fp32 1e-4, bf16 2e-2)."""

import numpy as np
import pytest

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import (bf16_bits, make_layer_inputs,
                                                            round_to_bf16)

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


def check_status(px):
    torch.cuda.synchronize()
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def weight(d_out, d_in, dtype, seed):
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((d_out, d_in)) / np.sqrt(d_in)
    W[1] = 0.0                        # a zero row: scale 0, codes 0
    W[2] = 0.0
    W[2, d_in // 2] = -3.0            # one entry carries the whole row
    W[3] *= 1e-30                     # tiny but normal scale
    W = round_to_bf16(W) if dtype == "bf16" else W.astype(np.float32)
    return W.astype(np.float32)


@pytest.mark.parametrize("dtype,d_out,d_in", [("bf16", 768, 512), ("bf16", 256, 4096),
                                              ("f32", 48, 96), ("f32", 10, 40),
                                              ("bf16", 7, 24)])
def test_quantize_and_dequantize_are_bit_exact(px, dtype, d_out, d_in):
    W = weight(d_out, d_in, dtype, 40)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = px.BF16 if dtype == "bf16" else px.F32
    Wd = torch.from_numpy(W).cuda().to(tdt)
    from orthogonal_reparameterized_packed_gb300.layer import quantize
    q, s = quantize(Wd, code)
    out = torch.empty_like(Wd)
    px.poetx_dequantize_w0(q, s, out, d_in, d_out, code)
    check_status(px)
    q_ref, s_ref = oracle.quantize_w0(W)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    deq = oracle.dequantize_w0(q_ref, s_ref)
    if dtype == "bf16":
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, bf16_bits(round_to_bf16(deq)))
    else:
        assert np.array_equal(out.cpu().numpy().view(np.uint32), deq.view(np.uint32))


def test_dequantize_unaligned_codes_take_the_scalar_path(px):
    W = weight(64, 256, "bf16", 41)
    q_ref, s_ref = oracle.quantize_w0(W)
    store = torch.empty(64 * 256 + 1, dtype=torch.int8, device="cuda")
    q = store[1:].view(64, 256)  # 1 byte off a 16-byte boundary
    q.copy_(torch.from_numpy(q_ref))
    s = torch.from_numpy(s_ref).cuda()
    out = torch.empty((64, 256), dtype=torch.bfloat16, device="cuda")
    px.poetx_dequantize_w0(q, s, out, 256, 64, px.BF16)
    check_status(px)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, bf16_bits(round_to_bf16(oracle.dequantize_w0(q_ref, s_ref))))


LAYER_CASES = [(512, 768, 256, 3, 300, "bf16"), (1024, 512, 128, 2, 129, "bf16"),
               (256, 256, 32, 3, 200, "f32")]


@pytest.mark.parametrize("d_in,d_out,b,k,T,dtype", LAYER_CASES)
def test_int8_layer_matches_oracle(px, d_in, d_out, b, k, T, dtype):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxQLayer, to_device
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, sigma_theta=0.02, seed=42)
    q_ref, s_ref = oracle.quantize_w0(inp.W0)
    dev = to_device(inp)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    layer = PoetxQLayer(d_in, d_out, b, k, T, dtype=dtype)
    layer.step(dev["theta_P"], dev["theta_R"], q, s, dev["x"], dev["dy"])
    check_status(px)
    W_deq = oracle.dequantize_w0(q_ref, s_ref)
    if dtype == "bf16":
        W_deq = round_to_bf16(W_deq)
    ref = oracle.layer(inp.theta_P, inp.theta_R, W_deq, inp.x, inp.dy, b, k)
    tol = 2e-2 if dtype == "bf16" else 1e-4
    n_in, n_out = d_in // b, d_out // b
    got = dict(y=layer.y, dx=layer.dx, dtheta_P=layer.dtheta_P.view(n_in, -1),
               dtheta_R=layer.dtheta_R.view(n_out, -1))
    for name, g in got.items():
        assert rel_fro(g.float().cpu().numpy(), ref[name]) <= tol, name


def test_merge_then_requantize(px):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxQLayer, to_device
    inp = make_layer_inputs(512, 256, 256, 3, 8, dtype="bf16", sigma_theta=0.03, seed=43)
    q_ref, s_ref = oracle.quantize_w0(inp.W0)
    dev = to_device(inp)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    layer = PoetxQLayer(512, 256, 256, 3, 8)
    layer.build(dev["theta_P"], dev["theta_R"])
    layer.merge_quantized(q, s, dev["theta_P"], dev["theta_R"])
    check_status(px)
    want = oracle.merge(inp.theta_P, inp.theta_R,
                        round_to_bf16(oracle.dequantize_w0(q_ref, s_ref)), 256, 3)
    got = oracle.dequantize_w0(q.cpu().numpy(), s.cpu().numpy())
    # one bf16 merge plus a re-quantisation (half a code step of each row)
    assert rel_fro(got, want) <= 1.5e-2
    assert torch.count_nonzero(dev["theta_P"]) == 0
