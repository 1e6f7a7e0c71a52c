"""poetx_build_blocks_noalloc: the block build for callers that cannot
allocate device memory (a static memory plan, or a framework that owns every
device buffer and has no workspace to hand over).  Called through the C ABI,
twice in a row with different parameters, its blocks must match those of
poetx_build_blocks (which uses a caller workspace) within the block
tolerances of the parity tests: 1e-6 (fp32) and 2^-8 (bf16) relative
Frobenius error.  Both run the same kernels, so the results are expected to
be identical; the second call also shows that what the first call left in
the shared scratch array does not leak into the next result.

This file is collected last on purpose."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_BLOCKS = {"f32": 1e-6, "bf16": 2.0 ** -8}


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


def rel_fro(a, b):
    a = a.double()
    b = b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


# the last two reach the scratch limit d * b = 2^20 on the fp32 path (three
# fp32 stacks of d * b elements: exactly 12 MiB)
@pytest.mark.parametrize("dtype,d,b,k", [("bf16", 4096, 256, 3), ("f32", 256, 32, 3),
                                         ("bf16", 1024, 64, 5), ("bf16", 2048, 512, 1),
                                         ("f32", 4096, 256, 3), ("f32", 2048, 512, 2)])
def test_noalloc_build_matches_workspace_build(px, dtype, d, b, k):
    code = px.BF16 if dtype == "bf16" else px.F32
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n, m = d // b, b * (b - 1) // 2
    ws = torch.empty((px.poetx_build_workspace_size(d, b, k, code),), dtype=torch.uint8,
                     device="cuda")
    for call, seed in enumerate((30, 31)):  # two calls in a row
        rng = np.random.default_rng(seed)
        theta = torch.from_numpy((rng.standard_normal((n, m)) * 0.02).astype(np.float32)).cuda()
        want = torch.empty((n, b, b), dtype=tdt, device="cuda")
        got = torch.full((n, b, b), float("nan"), dtype=tdt, device="cuda")
        px.poetx_build_blocks(theta, d, b, k, code, want, ws)
        px.poetx_build_blocks_noalloc(theta, d, b, k, code, got)
        torch.cuda.synchronize()
        assert px.poetx_device_status() == 0
        assert torch.isfinite(got.float()).all(), f"call {call}"
        err = rel_fro(got, want)
        assert err <= TOL_BLOCKS[dtype], f"call {call}: {err}"


def test_noalloc_rejects_builds_beyond_its_scratch(px):
    theta = torch.zeros((32, 256 * 255 // 2), dtype=torch.float32, device="cuda")
    blocks = torch.empty((32, 256, 256), dtype=torch.bfloat16, device="cuda")
    # d * b = 8192 * 256 = 2^21 > 2^20
    with pytest.raises(px.PoetxError) as e:
        px.poetx_build_blocks_noalloc(theta, 8192, 256, 3, px.BF16, blocks)
    assert e.value.status == 3  # POETX_ERR_WORKSPACE
