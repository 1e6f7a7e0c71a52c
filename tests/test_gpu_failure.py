"""Failure detection without a GPU fault: a barrier wait that nothing
satisfies runs out after its limit, the kernel records POETX_ERR_TIMEOUT in
the device status word and returns; the host reads the status once, and the
context keeps working (a block build afterwards succeeds with status OK)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


def test_wait_runs_out_and_context_survives(px):
    assert px.poetx_device_status() == 0
    px.poetx_selftest_wait_timeout(2000)  # 2 ms
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 5  # POETX_ERR_TIMEOUT
    assert px.poetx_device_status() == 0  # read once, then cleared
    # the context is still usable
    d, b, k = 512, 256, 3
    theta = torch.from_numpy((np.random.default_rng(0).standard_normal(
        (d // b, b * (b - 1) // 2)) * 0.02).astype(np.float32)).cuda()
    blocks = torch.empty((d // b, b, b), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty((px.poetx_build_workspace_size(d, b, k, px.BF16),), dtype=torch.uint8,
                     device="cuda")
    px.poetx_build_blocks(theta, d, b, k, px.BF16, blocks, ws)
    torch.cuda.synchronize()
    assert px.poetx_device_status() == 0
    assert torch.isfinite(blocks.float()).all()


def test_selftest_rejects_bad_limits(px):
    with pytest.raises(px.PoetxError):
        px.poetx_selftest_wait_timeout(0)
