"""weight_only_bit_gb300 -- fused 4-bit weight-only dequant-GEMV (W4A16) for GB300.

Python binding of libw4 (include/w4.h).  Each function has the C name and argument order,
accepts device buffers as torch tensors (or raw integer addresses), and returns the C status
code; `check(status)` turns a non-zero status into W4Error.  All arithmetic runs in libw4's CUDA
kernels; this module only marshals arguments.  `stream=None` means torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes

from ._lib import (GemvDesc, GemvPlan, W4Error, lib, SYMBOLS, W4_OK, W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_ALIGN,
                   W4_ERR_BLOCKSIZE, W4_ERR_CUDA, W4_ERR_TIMEOUT, W4_ERR_UNSUPPORTED, W4_FMT_NF4,
                   W4_FMT_INT4, W4_FMT_FP4, W4_MAX_BATCH, W4_MAX_K, W4_KERNEL_SMALL_BATCH, W4_KERNEL_TCGEN05)

__all__ = [
    "w4_nf4_codebook", "w4_quantize_nf4", "w4_quantize_int4", "w4_dequantize_nf4", "w4_dequantize_int4",
    "w4_gemv_nf4", "w4_gemv_int4", "w4_gemv_sequence", "w4_step_workspace_bytes", "w4_step_create",
    "w4_step_launch",
    "w4_step_destroy", "w4_status_str", "w4_last_cuda_error", "w4_device_check", "w4_launch_count",
    "w4_inject_timeout_once", "w4_gemv_levels_noalloc", "w4_gemv_plan",
    "w4_quantize_fp4", "w4_dequantize_fp4", "w4_gemv_fp4", "w4_step_run_host",
    "check", "W4Error", "GemvDesc", "GemvPlan", "W4_FMT_NF4", "W4_FMT_INT4", "W4_FMT_FP4", "W4_MAX_BATCH",
    "W4_MAX_K",
    "W4_KERNEL_SMALL_BATCH", "W4_KERNEL_TCGEN05",
]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(status: int, what: str = "") -> int:
    if status != W4_OK:
        raise W4Error(status, what)
    return status


def w4_nf4_codebook():
    """Host function: returns (status, list of 16 floats)."""
    out = (ctypes.c_float * 16)()
    st = lib().w4_nf4_codebook(out)
    return st, list(out)


def w4_quantize_nf4(W, packed, absmax, codebook, N, K, blocksize=64, stream=None):
    return lib().w4_quantize_nf4(_ptr(W), _ptr(packed), _ptr(absmax), _ptr(codebook), N, K, blocksize,
                                 _stream(stream))


def w4_quantize_int4(W, packed, scale, N, K, group=128, stream=None):
    return lib().w4_quantize_int4(_ptr(W), _ptr(packed), _ptr(scale), N, K, group, _stream(stream))


def w4_quantize_fp4(W, packed, scale, N, K, group=32, stream=None):
    return lib().w4_quantize_fp4(_ptr(W), _ptr(packed), _ptr(scale), N, K, group, _stream(stream))


def w4_dequantize_nf4(packed, absmax, codebook, W_out, N, K, blocksize=64, stream=None):
    return lib().w4_dequantize_nf4(_ptr(packed), _ptr(absmax), _ptr(codebook), _ptr(W_out), N, K, blocksize,
                                   _stream(stream))


def w4_dequantize_int4(packed, scale, W_out, N, K, group=128, stream=None):
    return lib().w4_dequantize_int4(_ptr(packed), _ptr(scale), _ptr(W_out), N, K, group, _stream(stream))


def w4_dequantize_fp4(packed, scale, W_out, N, K, group=32, stream=None):
    return lib().w4_dequantize_fp4(_ptr(packed), _ptr(scale), _ptr(W_out), N, K, group, _stream(stream))


def w4_gemv_nf4(packed, absmax, codebook, x, y, M, N, K, blocksize=64, stream=None):
    return lib().w4_gemv_nf4(_ptr(packed), _ptr(absmax), _ptr(codebook), _ptr(x), _ptr(y), M, N, K, blocksize,
                             _stream(stream))


def w4_gemv_int4(packed, scale, x, y, M, N, K, group=128, stream=None):
    return lib().w4_gemv_int4(_ptr(packed), _ptr(scale), _ptr(x), _ptr(y), M, N, K, group, _stream(stream))


def w4_gemv_fp4(packed, scale, x, y, M, N, K, group=32, stream=None):
    return lib().w4_gemv_fp4(_ptr(packed), _ptr(scale), _ptr(x), _ptr(y), M, N, K, group, _stream(stream))


def _descs(descs):
    arr = (GemvDesc * len(descs))()
    for i, d in enumerate(descs):
        arr[i] = GemvDesc(d["format"], _ptr(d["packed"]), _ptr(d["scales"]), _ptr(d.get("codebook")),
                          _ptr(d["x"]), _ptr(d["y"]), d["M"], d["N"], d["K"], d["blocksize"], d.get("level", i))
    return arr


def w4_gemv_sequence(descs, stream=None):
    """descs: sequence of dicts with keys format, packed, scales, codebook, x, y, M, N, K, blocksize and
    optionally level (default: the descriptor's index, i.e. every GEMV waits for the one before)."""
    arr = _descs(descs)
    return lib().w4_gemv_sequence(arr, len(descs), _stream(stream))


def w4_step_workspace_bytes(count: int) -> int:
    return lib().w4_step_workspace_bytes(count)


def w4_step_create(descs, workspace):
    """Returns (status, handle).  workspace: device buffer of w4_step_workspace_bytes(len(descs))."""
    arr = _descs(descs)
    h = ctypes.c_void_p()
    st = lib().w4_step_create(arr, len(descs), _ptr(workspace), ctypes.byref(h))
    return st, h.value


def w4_step_launch(step, stream=None):
    return lib().w4_step_launch(step, _stream(stream))


def w4_step_run_host(step, x_host, x_dev, x_bytes, y_host, y_dev, y_bytes, stream=None):
    """x_host / y_host: pinned host tensors (or raw addresses); x_dev / y_dev: the step's device
    input and output buffers."""
    return lib().w4_step_run_host(step, _ptr(x_host), _ptr(x_dev), x_bytes, _ptr(y_host), _ptr(y_dev), y_bytes,
                                  _stream(stream))


def w4_step_destroy(step):
    return lib().w4_step_destroy(step)


def w4_status_str(status: int) -> str:
    return lib().w4_status_str(status).decode()


def w4_last_cuda_error() -> int:
    return lib().w4_last_cuda_error()


def w4_device_check(stream=None) -> int:
    return lib().w4_device_check(_stream(stream))


def w4_gemv_plan(format: int, M: int, N: int, K: int, blocksize: int, sm_count: int = 152):
    """Host function: returns (status, dict of w4_gemv_plan_t's fields); no device call."""
    out = GemvPlan()
    st = lib().w4_gemv_plan(format, M, N, K, blocksize, sm_count, ctypes.byref(out))
    return st, {name: getattr(out, name) for name, _ in GemvPlan._fields_}


def w4_launch_count() -> int:
    return lib().w4_launch_count()


def w4_inject_timeout_once() -> int:
    return lib().w4_inject_timeout_once()


def w4_gemv_levels_noalloc(descs, stream=None) -> int:
    """One persistent launch of the descriptors with the level counters inside libw4, for callers
    that cannot allocate device memory; see include/w4.h for its limits and its one-time set-up."""
    arr = _descs(descs)
    return lib().w4_gemv_levels_noalloc(arr, len(descs), _stream(stream))
