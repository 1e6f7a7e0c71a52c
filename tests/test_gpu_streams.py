"""Independent layers on concurrent streams.  The library keeps no state
between calls outside the caller's buffers (each layer has its own
workspace), so layer steps enqueued on separate streams at once must give
bitwise the results of running them one after the other.  The streams'
kernels overlap on the GPU: the cooperative chain launches, the clustered W0
GEMMs, the fused backward kernel and the FFMA path run beside each other."""

import pytest

from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

OUTPUTS = ("y", "dx", "dtheta_P", "dtheta_R")


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    poetx.load_library()
    return poetx


def make(case, seed):
    from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
    d_in, d_out, b, k, T, dtype = case
    inp = make_layer_inputs(d_in, d_out, b, k, T, dtype=dtype, seed=seed)
    dev = to_device(inp)
    layer = PoetxLayer(d_in, d_out, b, k, T, dtype=dtype)
    return layer, dev


def step(layer, dev, stream=None):
    layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"], stream=stream)


CASES = [
    (1024, 768, 256, 3, 1000, "bf16"),   # fused backward kernel, chains, split W0 GEMM tail
    (512, 1024, 128, 2, 700, "bf16"),    # b = 128: the general chain recursion
    (2048, 2048, 256, 3, 2304, "bf16"),  # more tiles than one round of clusters
    (256, 256, 32, 3, 512, "f32"),       # FFMA path
]


def test_concurrent_streams_match_sequential(px):
    layers = [make(c, 90 + i) for i, c in enumerate(CASES)]
    want = []
    for layer, dev in layers:
        step(layer, dev)
        torch.cuda.synchronize()
        want.append({n: getattr(layer, n).clone() for n in OUTPUTS})
    st = px.poetx_device_status()
    assert st == 0, px.poetx_status_string(st)

    streams = [torch.cuda.Stream() for _ in layers]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for (layer, dev), s in zip(layers, streams):
            for n in OUTPUTS:
                getattr(layer, n).zero_()
        torch.cuda.synchronize()
        for (layer, dev), s in zip(layers, streams):
            step(layer, dev, stream=s)  # enqueued back to back, the streams overlap
        torch.cuda.synchronize()
        st = px.poetx_device_status()
        assert st == 0, px.poetx_status_string(st)
        for i, (layer, _) in enumerate(layers):
            for n in OUTPUTS:
                assert torch.equal(getattr(layer, n), want[i][n]), (CASES[i], n, rep)


THREADED = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import orthogonal_reparameterized_packed_gb300 as poetx
from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs
from orthogonal_reparameterized_packed_gb300.layer import PoetxLayer, to_device
poetx.load_library()
cases = [(1024, 768, 256, 3, 1000, "bf16"), (512, 1024, 128, 2, 700, "bf16"),
         (2048, 2048, 256, 3, 2304, "bf16"), (256, 256, 32, 3, 512, "f32")]
jobs = []
for i, (d_in, d_out, b, k, T, dt) in enumerate(cases):
    dev = to_device(make_layer_inputs(d_in, d_out, b, k, T, dtype=dt, seed=95 + i))
    jobs.append((PoetxLayer(d_in, d_out, b, k, T, dtype=dt), dev, torch.cuda.Stream()))
torch.cuda.synchronize()
names = ("y", "dx", "dtheta_P", "dtheta_R")
errors = []
def run(layer, dev, s):
    try:
        layer.step(dev["theta_P"], dev["theta_R"], dev["W0"], dev["x"], dev["dy"], stream=s)
    except Exception as e:  # reported by the main thread
        errors.append(repr(e))
# first calls of the process, from four host threads at once
threads = [threading.Thread(target=run, args=j) for j in jobs]
for t in threads: t.start()
for t in threads: t.join()
torch.cuda.synchronize()
assert not errors, errors
assert poetx.poetx_device_status() == 0
got = [{n: getattr(l, n).clone() for n in names} for l, _, _ in jobs]
for l, dev, _ in jobs:
    run(l, dev, None)
    torch.cuda.synchronize()
assert not errors, errors
for i, (l, _, _) in enumerate(jobs):
    for n in names:
        assert torch.equal(getattr(l, n), got[i][n]), (cases[i], n)
print("threads ok")
"""


def test_first_calls_from_several_host_threads():
    # a fresh process, so that the library's per-device setup (function
    # attributes, cluster and occupancy queries) happens under the race
    import os
    import subprocess
    import sys
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", THREADED, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "threads ok" in r.stdout
