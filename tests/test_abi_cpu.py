"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, it exports every function include/poetx.h declares, the workspace
size queries agree with the documented buffer plan, and invalid arguments
are rejected before anything is enqueued."""

import ctypes
import os
import re

import pytest

import orthogonal_reparameterized_packed_gb300 as poetx
from orthogonal_reparameterized_packed_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "poetx.h")


@pytest.fixture(scope="module")
def lib():
    build_library()
    return poetx.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(poetx_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_declares_the_three_core_calls():
    names = _declared_functions()
    for core in ("poetx_build_blocks", "poetx_forward", "poetx_backward"):
        assert core in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names == set(poetx.EXPORTED_SYMBOLS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(6):
        s = poetx.poetx_status_string(code)
        assert s.startswith("POETX_")
    assert "unknown" in poetx.poetx_status_string(99)


@pytest.mark.parametrize("d,b", [(256, 32), (4096, 256), (96, 3), (1024, 512)])
def test_packed_size(lib, d, b):
    assert poetx.poetx_packed_size(d, b) == (d // b) * b * (b - 1) // 2


def test_packed_size_rejects_bad_dims(lib):
    assert poetx.poetx_packed_size(100, 32) == 0
    assert poetx.poetx_packed_size(0, 4) == 0


def test_workspace_sizes_are_positive_and_monotone(lib):
    F32, BF16 = poetx.F32, poetx.BF16
    # the bf16 builds on CTA pairs (b <= 256, 1 <= k <= 16) keep their
    # operands in shared memory; the chain (b = 512) and k = 0 need scratch
    assert poetx.poetx_build_workspace_size(4096, 256, 3, BF16) == 0
    assert poetx.poetx_build_workspace_size(4096, 256, 5, BF16) == 0
    assert poetx.poetx_build_workspace_size(4096, 64, 16, BF16) == 0
    assert poetx.poetx_build_workspace_size(4096, 512, 3, BF16) > 0
    assert poetx.poetx_build_workspace_size(4096, 256, 0, BF16) > 0
    assert poetx.poetx_build_workspace_size(256, 32, 3, F32) > 0
    a = poetx.poetx_forward_workspace_size(4096, 4096, 256, 1024, BF16)
    b = poetx.poetx_forward_workspace_size(4096, 4096, 256, 2048, BF16)
    assert 0 < a < b
    # the forward needs at least the intermediate u = P x
    assert a >= 1024 * 4096 * 2
    r0 = poetx.poetx_backward_workspace_size(4096, 4096, 256, 3, 1024, BF16, False)
    r1 = poetx.poetx_backward_workspace_size(4096, 4096, 256, 3, 1024, BF16, True)
    assert 0 < r0 < r1
    assert poetx.poetx_transform_workspace_size(4096, 32, 5, 8192, BF16) > 0


def test_unsupported_shapes_give_zero_workspace(lib):
    BF16 = poetx.BF16
    assert poetx.poetx_forward_workspace_size(4800, 4800, 48, 16, BF16) == 0  # b not a power of 2
    assert poetx.poetx_forward_workspace_size(384, 384, 128, 16, BF16) == 0   # d % 256
    assert poetx.poetx_build_workspace_size(100, 32, 3, poetx.F32) == 0       # d % b


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on these paths


def _raw():
    return poetx.load_library()


def test_build_rejects_invalid_arguments(lib):
    L = _raw()
    ws = poetx.poetx_build_workspace_size(256, 32, 3, poetx.F32)
    assert L.poetx_build_blocks(FAKE, 100, 32, 3, poetx.F32, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(None, 256, 32, 3, poetx.F32, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(FAKE + 4, 256, 32, 3, poetx.F32, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(FAKE, 256, 32, -1, poetx.F32, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(FAKE, 256, 32, 17, poetx.F32, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(FAKE, 256, 32, 3, 7, FAKE, FAKE, ws, None) == 1
    assert L.poetx_build_blocks(FAKE, 256, 32, 3, poetx.F32, FAKE, FAKE, ws - 1, None) == 3
    assert L.poetx_build_blocks(FAKE, 256, 32, 3, poetx.F32, FAKE, None, ws, None) == 3
    assert L.poetx_build_blocks(FAKE, 4800, 48, 3, poetx.BF16, FAKE, FAKE, ws, None) == 2


def test_forward_and_backward_reject_invalid_arguments(lib):
    L = _raw()
    B = poetx.BF16
    ws = poetx.poetx_forward_workspace_size(512, 512, 256, 64, B)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    assert L.poetx_forward(*args, 512, 512, 256, -1, B, FAKE, ws, None) == 1
    assert L.poetx_forward(*args, 512, 500, 256, 64, B, FAKE, ws, None) == 1
    assert L.poetx_forward(*args, 512, 640, 128, 64, B, FAKE, ws, None) == 2
    # v_saved = NULL: the workspace must also hold v
    assert L.poetx_forward(FAKE, FAKE, FAKE, FAKE, FAKE, None, 512, 512, 256, 64, B, FAKE,
                           ws - 256, None) == 3
    assert L.poetx_forward(FAKE, FAKE, None, FAKE, FAKE, None, 512, 512, 256, 64, B, FAKE, ws,
                           None) == 1
    assert L.poetx_forward(FAKE, FAKE, FAKE, FAKE, FAKE + 8, None, 512, 512, 256, 64, B, FAKE,
                           ws, None) == 1
    wb = poetx.poetx_backward_workspace_size(512, 512, 256, 3, 64, B, 0)
    bargs = [FAKE] * 7
    assert L.poetx_backward(*bargs, FAKE, FAKE, FAKE, FAKE, 512, 512, 256, 3, 64, B, FAKE,
                            wb - 1, None) == 3
    assert L.poetx_backward(*bargs, FAKE, None, FAKE, FAKE, 512, 512, 256, 3, 64, B, FAKE,
                            wb, None) == 1
    assert L.poetx_backward(*bargs, FAKE, FAKE, FAKE, FAKE, 512, 512, 256, 20, 64, B, FAKE,
                            wb, None) == 1


def test_merge_and_adam_reject_invalid_arguments(lib):
    L = _raw()
    B, F = poetx.BF16, poetx.F32
    ws = poetx.poetx_merge_workspace_size(512, 768, 256, B)
    # the merge needs W0 P (bf16) in the workspace
    assert ws >= 768 * 512 * 2
    assert poetx.poetx_merge_workspace_size(512, 768, 48, B) == 0
    assert poetx.poetx_merge_workspace_size(100, 64, 32, F) == 0
    p4 = [FAKE] * 4
    assert L.poetx_merge(*p4, None, None, 512, 700, 256, B, FAKE, ws, None) == 1
    assert L.poetx_merge(FAKE, None, FAKE, FAKE, None, None, 512, 768, 256, B, FAKE, ws,
                         None) == 1
    assert L.poetx_merge(*p4, FAKE + 4, None, 512, 768, 256, B, FAKE, ws, None) == 1
    assert L.poetx_merge(*p4, None, None, 512, 768, 256, B, FAKE, ws - 1, None) == 3
    assert L.poetx_merge(*p4, None, None, 512, 768, 256, B, None, ws, None) == 3
    assert L.poetx_merge(*p4, None, None, 512, 640, 128, B, FAKE, ws, None) == 2
    f = ctypes.c_float
    assert L.poetx_adam_update(FAKE, FAKE, FAKE, FAKE, 4, 0, f(1e-3), f(0.9), f(0.999), f(1e-8),
                               f(0.0), None) == 1
    assert L.poetx_adam_update(FAKE, FAKE, FAKE, FAKE, -1, 1, f(1e-3), f(0.9), f(0.999),
                               f(1e-8), f(0.0), None) == 1
    assert L.poetx_adam_update(FAKE, FAKE, FAKE, FAKE, 4, 1, f(1e-3), f(1.0), f(0.999), f(1e-8),
                               f(0.0), None) == 1
    assert L.poetx_adam_update(FAKE, FAKE, FAKE, FAKE, 4, 1, f(1e-3), f(0.9), f(0.999), f(0.0),
                               f(0.0), None) == 1
    assert L.poetx_adam_update(None, FAKE, FAKE, FAKE, 4, 1, f(1e-3), f(0.9), f(0.999), f(1e-8),
                               f(0.0), None) == 1
    assert L.poetx_adam_update(None, None, None, None, 0, 1, f(1e-3), f(0.9), f(0.999), f(1e-8),
                               f(0.0), None) == 0


def test_int8_weight_calls_reject_invalid_arguments(lib):
    L = _raw()
    for fn in (L.poetx_quantize_w0, L.poetx_dequantize_w0):
        assert fn(FAKE, FAKE, FAKE, 64, 64, 7, None) == 1
        assert fn(FAKE, FAKE, FAKE, -1, 64, poetx.BF16, None) == 1
        assert fn(None, FAKE, FAKE, 64, 64, poetx.BF16, None) == 1
        assert fn(FAKE, None, FAKE, 64, 64, poetx.F32, None) == 1
        assert fn(FAKE, FAKE, None, 64, 64, poetx.F32, None) == 1
        assert fn(None, None, None, 0, 64, poetx.BF16, None) == 0  # empty: nothing to do


def test_index_map_calls_reject_invalid_arguments(lib):
    L = _raw()
    B, F = poetx.BF16, poetx.F32
    # d beyond the shared-memory entry table, d * element size not a multiple of 16
    assert L.poetx_permute_features(FAKE, FAKE, FAKE + 4096, 8, 28672 + 8, B, None) == 1
    assert L.poetx_permute_features(FAKE, FAKE, FAKE + 4096, 8, 12, B, None) == 1
    # the column map is read as 16-byte vectors
    assert L.poetx_permute_features(FAKE, FAKE + 4, FAKE + 4096, 8, 64, B, None) == 1
    assert L.poetx_permute_features(FAKE, FAKE, FAKE, 8, 64, B, None) == 1  # in == out
    assert L.poetx_permute_features(None, None, None, 0, 64, F, None) == 0  # no rows
    assert L.poetx_fold_permutations(FAKE, FAKE, FAKE + 4, FAKE + 4096, 64, 64, B, None) == 1
    assert L.poetx_fold_permutations(FAKE, FAKE, FAKE, FAKE + 4096, 28680, 64, B, None) == 1


def test_process_wide_switches_return_the_previous_setting(lib):
    # host-only state: block-epilogue fusion off and the W0 tail split on by default
    assert poetx.poetx_set_block_epilogue_fusion(False) is False
    assert poetx.poetx_set_w0_split_tail(False) is True
    assert poetx.poetx_set_w0_split_tail(True) is False
    assert poetx.poetx_set_w0_split_tail(True) is True
    # the W0 GEMMs on CTA pairs by default
    assert poetx.poetx_set_w0_pair_mma(False) is True
    assert poetx.poetx_set_w0_pair_mma(True) is False
    assert poetx.poetx_set_w0_pair_mma(True) is True
