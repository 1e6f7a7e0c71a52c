"""The device-side pull of pinned host memory: bit-exact copies of several
sizes, and pageable (not page-locked) memory rejected before anything is
enqueued."""

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


@pytest.mark.parametrize("nbytes", [16, 4096, (1 << 20) + 48, 64 << 20])
def test_pull_is_bit_exact(px, nbytes):
    g = torch.Generator().manual_seed(nbytes)
    host = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes + 32,), 7, dtype=torch.uint8, device="cuda")
    px.poetx_copy_from_host(host, dev[:nbytes])
    torch.cuda.synchronize()
    assert torch.equal(dev[:nbytes].cpu(), host)
    assert bool((dev[nbytes:] == 7).all())  # nothing written past the end
    assert px.poetx_device_status() == 0


def test_pull_on_a_side_stream_then_use(px):
    host = torch.arange(1 << 16, dtype=torch.float32).pin_memory()
    dev = torch.empty(1 << 16, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        px.poetx_copy_from_host(host, dev, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    assert float(dev.sum()) == float(host.sum())


def test_pageable_memory_is_rejected(px):
    host = torch.zeros(4096, dtype=torch.uint8)  # not page-locked
    dev = torch.empty(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(px.PoetxError):
        px.poetx_copy_from_host(host, dev)
