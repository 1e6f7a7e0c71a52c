"""Out-of-bounds writes: every output and workspace buffer of the C ABI is
placed between two guard bands filled with a byte pattern; after the calls
the bands must be unchanged (compute-sanitizer is not available, so this is
the check that no kernel stores past its buffers).  Ragged token counts and
every kernel family (tensor-core chains and transforms, the fused backward
kernel, the FFMA path, index maps, INT8 weight, merge) are covered."""

import numpy as np
import pytest

from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


class Guarded:
    """Device buffers carved from byte arrays with guard bands around them."""

    def __init__(self):
        self.bufs = []

    def tensor(self, shape, dtype):
        n = int(np.prod(shape)) if len(shape) else 1
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, nbytes))
        return raw[GUARD:GUARD + nbytes].view(dtype).view(*shape)

    def workspace(self, nbytes):
        return self.tensor((max(int(nbytes), 16),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, nbytes) in enumerate(self.bufs):
            head = raw[:GUARD]
            tail = raw[GUARD + nbytes:]
            assert bool((head == PATTERN).all()), f"buffer {i}: write before its start"
            assert bool((tail == PATTERN).all()), f"buffer {i}: write past its end"


def status_ok(px):
    torch.cuda.synchronize()
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)


def dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dtype)


LAYER_CASES = [
    # d_in, d_out, b, k, T, dtype   (chain k = 3 / other k, fused backward, b < 128, FFMA)
    (512, 768, 256, 3, 333, "bf16"),
    (256, 512, 128, 2, 130, "bf16"),
    (512, 256, 64, 3, 257, "bf16"),
    (1024, 512, 512, 3, 129, "bf16"),
    (96, 48, 3, 2, 37, "f32"),
]


@pytest.mark.parametrize("d_in,d_out,b,k,T,dtype", LAYER_CASES)
@pytest.mark.parametrize("recompute_v", [False, True])
def test_layer_calls_write_only_their_buffers(px, d_in, d_out, b, k, T, dtype, recompute_v):
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, seed=70)
    code = px.BF16 if dtype == "bf16" else px.F32
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = Guarded()
    tP, tR = dev(inp.theta_P, torch.float32), dev(inp.theta_R, torch.float32)
    W0, x, dy = dev(inp.W0, tdt), dev(inp.x, tdt), dev(inp.dy, tdt)
    Pb = g.tensor((d_in // b, b, b), tdt)
    Rb = g.tensor((d_out // b, b, b), tdt)
    y = g.tensor((T, d_out), tdt)
    v = None if recompute_v else g.tensor((T, d_out), tdt)
    dx = g.tensor((T, d_in), tdt)
    dP = g.tensor((px.poetx_packed_size(d_in, b),), torch.float32)
    dR = g.tensor((px.poetx_packed_size(d_out, b),), torch.float32)
    ws = g.workspace(max(px.poetx_build_workspace_size(d_in, b, k, code),
                         px.poetx_build_workspace_size(d_out, b, k, code),
                         px.poetx_forward_workspace_size(d_in, d_out, b, T, code),
                         px.poetx_backward_workspace_size(d_in, d_out, b, k, T, code,
                                                          recompute_v)))
    px.poetx_build_blocks(tP, d_in, b, k, code, Pb, ws)
    px.poetx_build_blocks(tR, d_out, b, k, code, Rb, ws)
    px.poetx_forward(x, W0, Pb, Rb, y, v, d_in, d_out, b, T, code, ws)
    px.poetx_backward(dy, x, W0, tP, tR, Pb, Rb, v, dx, dP, dR, d_in, d_out, b, k, T, code, ws)
    status_ok(px)
    g.check()
    assert bool(torch.isfinite(y.float()).all()) and bool(torch.isfinite(dP).all())


@pytest.mark.parametrize("d,b,k,T", [(1024, 256, 3, 300), (1024, 32, 5, 77), (512, 128, 1, 129)])
def test_transform_calls_write_only_their_buffers(px, d, b, k, T):
    inp = make_layer_inputs(d, d, b, k, T, dtype="bf16", seed=71)
    g = Guarded()
    th = dev(inp.theta_P, torch.float32)
    x, dout = dev(inp.x, torch.bfloat16), dev(inp.dy, torch.bfloat16)
    blocks = g.tensor((d // b, b, b), torch.bfloat16)
    out = g.tensor((T, d), torch.bfloat16)
    dx = g.tensor((T, d), torch.bfloat16)
    dth = g.tensor((d // b, b * (b - 1) // 2), torch.float32)
    ws = g.workspace(max(px.poetx_build_workspace_size(d, b, k, px.BF16),
                         px.poetx_transform_workspace_size(d, b, k, T, px.BF16)))
    px.poetx_build_blocks(th, d, b, k, px.BF16, blocks, ws)
    px.poetx_transform_forward(x, blocks, out, d, b, T, px.BF16, ws)
    px.poetx_transform_backward(dout, x, th, blocks, dx, dth, d, b, k, T, px.BF16, ws)
    status_ok(px)
    g.check()


def test_weight_calls_write_only_their_buffers(px):
    d_in, d_out, b = 512, 768, 256
    inp = make_layer_inputs(d_in, d_out, b, 3, 8, dtype="bf16", seed=72)
    g = Guarded()
    W0 = dev(inp.W0, torch.bfloat16)
    q = g.tensor((d_out, d_in), torch.int8)
    s = g.tensor((d_out,), torch.float32)
    Wd = g.tensor((d_out, d_in), torch.bfloat16)
    px.poetx_quantize_w0(W0, q, s, d_in, d_out, px.BF16)
    px.poetx_dequantize_w0(q, s, Wd, d_in, d_out, px.BF16)
    ws = g.workspace(max(px.poetx_build_workspace_size(d_in + d_out, b, 3, px.BF16),
                         px.poetx_merge_workspace_size(d_in, d_out, b, px.BF16)))
    blocks = g.tensor(((d_in + d_out) // b, b, b), torch.bfloat16)
    theta = dev(np.concatenate([inp.theta_P.ravel(), inp.theta_R.ravel()]), torch.float32)
    px.poetx_build_blocks(theta, d_in + d_out, b, 3, px.BF16, blocks, ws)
    Wm = g.tensor((d_out, d_in), torch.bfloat16)
    px.poetx_merge(W0, blocks[:d_in // b], blocks[d_in // b:], Wm, None, None, d_in, d_out, b,
                   px.BF16, ws)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(d_in).astype(np.int32)).cuda()
    xp = g.tensor((37, d_in), torch.bfloat16)
    px.poetx_permute_features(dev(inp.x[:8].repeat(5, axis=0)[:37], torch.bfloat16), perm, xp, 37,
                              d_in, px.BF16)
    status_ok(px)
    g.check()
