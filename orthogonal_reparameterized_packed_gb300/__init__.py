"""POET-X layer hot path on one GB300: Python binding of libpoetx.so.

The binding only marshals arguments (tensor data pointers, sizes, the
current CUDA stream) into the C ABI declared in include/poetx.h; every step
of the computation runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing or cannot be loaded, every call raises.
PyTorch is used for device memory and streams only.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "PoetxError", "load_library", "F32", "BF16",
    "poetx_packed_size", "poetx_build_workspace_size", "poetx_build_blocks",
    "poetx_build_blocks_noalloc",
    "poetx_forward_workspace_size", "poetx_forward",
    "poetx_backward_workspace_size", "poetx_backward",
    "poetx_transform_workspace_size", "poetx_transform_forward", "poetx_transform_backward",
    "poetx_permute_features", "poetx_fold_permutations", "poetx_merge_workspace_size",
    "poetx_merge", "poetx_adam_update", "poetx_quantize_w0", "poetx_dequantize_w0",
    "poetx_set_block_epilogue_fusion",
    "poetx_set_w0_split_tail",
    "poetx_set_w0_pair_mma",
    "poetx_device_status", "poetx_selftest_wait_timeout", "poetx_launch_count", "poetx_profile_start", "poetx_profile_stop",
    "poetx_profile_query", "poetx_status_string", "EXPORTED_SYMBOLS",
]

F32 = 0
BF16 = 1

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpoetx.so")

_c_size = ctypes.c_size_t
_c_int = ctypes.c_int
_c_i64 = ctypes.c_int64
_c_ptr = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/poetx.h
_SIGNATURES = {
    "poetx_status_string": (ctypes.c_char_p, [_c_int]),
    "poetx_packed_size": (_c_size, [_c_int, _c_int]),
    "poetx_build_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "poetx_build_blocks": (_c_int, [_c_ptr, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_ptr,
                                    _c_size, _c_ptr]),
    "poetx_build_blocks_noalloc": (_c_int, [_c_ptr, _c_int, _c_int, _c_int, _c_int, _c_ptr,
                                            _c_ptr]),
    "poetx_forward_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_i64, _c_int]),
    "poetx_forward": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int,
                               _c_int, _c_i64, _c_int, _c_ptr, _c_size, _c_ptr]),
    "poetx_backward_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int,
                                                _c_int]),
    "poetx_backward": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_i64,
                                _c_int, _c_ptr, _c_size, _c_ptr]),
    "poetx_transform_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_i64, _c_int]),
    "poetx_transform_forward": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_i64, _c_int,
                                         _c_ptr, _c_size, _c_ptr]),
    "poetx_transform_backward": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int,
                                          _c_int, _c_int, _c_i64, _c_int, _c_ptr, _c_size,
                                          _c_ptr]),
    "poetx_permute_features": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_int, _c_int, _c_ptr]),
    "poetx_fold_permutations": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int,
                                         _c_ptr]),
    "poetx_merge_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "poetx_merge": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int,
                             _c_int, _c_ptr, _c_size, _c_ptr]),
    "poetx_adam_update": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_int,
                                   ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                   ctypes.c_float, _c_ptr]),
    "poetx_quantize_w0": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_ptr]),
    "poetx_dequantize_w0": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_ptr]),
    "poetx_set_block_epilogue_fusion": (_c_int, [_c_int]),
    "poetx_set_w0_split_tail": (_c_int, [_c_int]),
    "poetx_set_w0_pair_mma": (_c_int, [_c_int]),
    "poetx_device_status": (_c_int, []),
    "poetx_selftest_wait_timeout": (_c_int, [ctypes.c_uint, _c_ptr]),
    "poetx_launch_count": (ctypes.c_longlong, []),
    "poetx_profile_start": (_c_int, [_c_int]),
    "poetx_profile_stop": (None, []),
    "poetx_profile_query": (_c_int, [ctypes.c_char_p, ctypes.POINTER(_c_int),
                                     ctypes.POINTER(ctypes.c_double)]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


class PoetxError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {poetx_status_string(status)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpoetx.so (built by build()).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(fn, status):
    if status != 0:
        raise PoetxError(fn, status)


def poetx_status_string(status: int) -> str:
    return load_library().poetx_status_string(status).decode()


def poetx_packed_size(d: int, b: int) -> int:
    return load_library().poetx_packed_size(d, b)


def poetx_build_workspace_size(d, b, k, dtype) -> int:
    return load_library().poetx_build_workspace_size(d, b, k, dtype)


def poetx_build_blocks(theta, d, b, k, dtype, blocks, workspace, stream=None):
    _check("poetx_build_blocks", load_library().poetx_build_blocks(
        _ptr(theta), d, b, k, dtype, _ptr(blocks), _ptr(workspace), _nbytes(workspace),
        _stream(stream)))


def poetx_build_blocks_noalloc(theta, d, b, k, dtype, blocks, stream=None):
    """Block build without a workspace, for callers that cannot allocate
    device memory (scratch is the library's fixed device array; d * b must be
    at most 2^20; calls that overlap on the GPU race on that array)."""
    _check("poetx_build_blocks_noalloc", load_library().poetx_build_blocks_noalloc(
        _ptr(theta), d, b, k, dtype, _ptr(blocks), _stream(stream)))


def poetx_forward_workspace_size(d_in, d_out, b, tokens, dtype) -> int:
    return load_library().poetx_forward_workspace_size(d_in, d_out, b, tokens, dtype)


def poetx_forward(x, W0, P_blocks, R_blocks, y, v_saved, d_in, d_out, b, tokens, dtype,
                  workspace, stream=None):
    _check("poetx_forward", load_library().poetx_forward(
        _ptr(x), _ptr(W0), _ptr(P_blocks), _ptr(R_blocks), _ptr(y), _ptr(v_saved), d_in, d_out,
        b, tokens, dtype, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def poetx_backward_workspace_size(d_in, d_out, b, k, tokens, dtype, recompute_v=False) -> int:
    return load_library().poetx_backward_workspace_size(d_in, d_out, b, k, tokens, dtype,
                                                        int(bool(recompute_v)))


def poetx_backward(dy, x, W0, theta_P, theta_R, P_blocks, R_blocks, v_saved, dx, dtheta_P,
                   dtheta_R, d_in, d_out, b, k, tokens, dtype, workspace, stream=None):
    _check("poetx_backward", load_library().poetx_backward(
        _ptr(dy), _ptr(x), _ptr(W0), _ptr(theta_P), _ptr(theta_R), _ptr(P_blocks),
        _ptr(R_blocks), _ptr(v_saved), _ptr(dx), _ptr(dtheta_P), _ptr(dtheta_R), d_in, d_out, b,
        k, tokens, dtype, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def poetx_transform_workspace_size(d, b, k, tokens, dtype) -> int:
    return load_library().poetx_transform_workspace_size(d, b, k, tokens, dtype)


def poetx_transform_forward(x, blocks, out, d, b, tokens, dtype, workspace, stream=None):
    _check("poetx_transform_forward", load_library().poetx_transform_forward(
        _ptr(x), _ptr(blocks), _ptr(out), d, b, tokens, dtype, _ptr(workspace),
        _nbytes(workspace), _stream(stream)))


def poetx_transform_backward(dout, x, theta, blocks, dx, dtheta, d, b, k, tokens, dtype,
                             workspace, stream=None):
    _check("poetx_transform_backward", load_library().poetx_transform_backward(
        _ptr(dout), _ptr(x), _ptr(theta), _ptr(blocks), _ptr(dx), _ptr(dtheta), d, b, k, tokens,
        dtype, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def poetx_permute_features(inp, perm, out, rows, d, dtype, stream=None):
    _check("poetx_permute_features", load_library().poetx_permute_features(
        _ptr(inp), _ptr(perm), _ptr(out), rows, d, dtype, _stream(stream)))


def poetx_fold_permutations(W0, perm_out, perm_in, W0_folded, d_in, d_out, dtype, stream=None):
    _check("poetx_fold_permutations", load_library().poetx_fold_permutations(
        _ptr(W0), _ptr(perm_out), _ptr(perm_in), _ptr(W0_folded), d_in, d_out, dtype,
        _stream(stream)))


def poetx_merge_workspace_size(d_in, d_out, b, dtype) -> int:
    return load_library().poetx_merge_workspace_size(d_in, d_out, b, dtype)


def poetx_merge(W0, P_blocks, R_blocks, W0_out, theta_P, theta_R, d_in, d_out, b, dtype,
                workspace, stream=None):
    _check("poetx_merge", load_library().poetx_merge(
        _ptr(W0), _ptr(P_blocks), _ptr(R_blocks), _ptr(W0_out), _ptr(theta_P), _ptr(theta_R),
        d_in, d_out, b, dtype, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def poetx_adam_update(theta, grad, m, v, n, step, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                      weight_decay=0.0, stream=None):
    _check("poetx_adam_update", load_library().poetx_adam_update(
        _ptr(theta), _ptr(grad), _ptr(m), _ptr(v), n, step, lr, beta1, beta2, eps, weight_decay,
        _stream(stream)))


def poetx_quantize_w0(W0, W0_q, scales, d_in, d_out, dtype, stream=None):
    _check("poetx_quantize_w0", load_library().poetx_quantize_w0(
        _ptr(W0), _ptr(W0_q), _ptr(scales), d_in, d_out, dtype, _stream(stream)))


def poetx_dequantize_w0(W0_q, scales, W0, d_in, d_out, dtype, stream=None):
    _check("poetx_dequantize_w0", load_library().poetx_dequantize_w0(
        _ptr(W0_q), _ptr(scales), _ptr(W0), d_in, d_out, dtype, _stream(stream)))


def poetx_set_block_epilogue_fusion(enable: bool) -> bool:
    """Turn the W0 GEMM's block-diagonal epilogue on or off (process-wide);
    returns the previous setting."""
    return bool(load_library().poetx_set_block_epilogue_fusion(1 if enable else 0))


def poetx_set_w0_split_tail(enable: bool) -> bool:
    """Turn the K split of the W0 GEMMs' last partial round of tiles on or
    off (process-wide); returns the previous setting."""
    return bool(load_library().poetx_set_w0_split_tail(1 if enable else 0))


def poetx_set_w0_pair_mma(enable: bool) -> bool:
    """Run the W0 GEMMs on CTA pairs (256-row MMAs across two SMs) or on
    clusters of one-SM MMAs (process-wide); returns the previous setting."""
    return bool(load_library().poetx_set_w0_pair_mma(1 if enable else 0))


def poetx_device_status() -> int:
    return load_library().poetx_device_status()


def poetx_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Enqueue the self-check kernel whose barrier wait must time out."""
    _check("poetx_selftest_wait_timeout",
           load_library().poetx_selftest_wait_timeout(limit_us, _stream(stream)))


def poetx_launch_count() -> int:
    return load_library().poetx_launch_count()


def poetx_profile_start(capacity: int) -> None:
    if load_library().poetx_profile_start(capacity) != 0:
        raise RuntimeError("poetx_profile_start: could not create CUDA events")


def poetx_profile_stop() -> None:
    load_library().poetx_profile_stop()


def poetx_profile_query(tag=None):
    """(count, total_ms) over the recorded launches with this tag."""
    n = _c_int(0)
    ms = ctypes.c_double(0.0)
    r = load_library().poetx_profile_query(None if tag is None else tag.encode(),
                                           ctypes.byref(n), ctypes.byref(ms))
    if r != 0:
        raise RuntimeError("poetx_profile_query failed")
    return n.value, ms.value
