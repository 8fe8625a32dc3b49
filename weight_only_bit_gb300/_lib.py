"""ctypes loader for libw4.so (the C ABI in include/w4.h).

Loading never touches the GPU.  If the library has not been built, every call raises W4Error:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libw4.so")

W4_OK = 0
W4_ERR_NULL = -1
W4_ERR_SHAPE = -2
W4_ERR_ALIGN = -3
W4_ERR_BLOCKSIZE = -4
W4_ERR_CUDA = -5
W4_ERR_TIMEOUT = -6
W4_ERR_UNSUPPORTED = -7
W4_ERR_LIMIT = -8
W4_NOALLOC_MAX_LEVELS = 256
W4_NOALLOC_MAX_GEMVS = 256
W4_FMT_NF4 = 0
W4_FMT_INT4 = 1
W4_FMT_FP4 = 2
W4_KERNEL_SMALL_BATCH = 1
W4_KERNEL_TCGEN05 = 2
W4_MAX_BATCH = 4096
W4_MAX_K = 10240

# Every symbol include/w4.h declares.
SYMBOLS = (
    "w4_nf4_codebook", "w4_quantize_nf4", "w4_quantize_int4", "w4_dequantize_nf4",
    "w4_dequantize_int4", "w4_gemv_nf4", "w4_gemv_int4", "w4_gemv_sequence", "w4_step_workspace_bytes", "w4_step_create",
    "w4_step_launch", "w4_step_destroy", "w4_status_str", "w4_last_cuda_error", "w4_device_check",
    "w4_launch_count", "w4_inject_timeout_once", "w4_gemv_levels_noalloc", "w4_gemv_plan",
    "w4_quantize_fp4", "w4_dequantize_fp4", "w4_gemv_fp4", "w4_step_run_host",
)


class W4Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{what}: " if what else ""
        try:
            msg += lib().w4_status_str(status).decode()
        except Exception:  # the library itself may be what is missing
            msg += f"status {status}"
        if status == W4_ERR_CUDA:
            try:
                msg += f" (cudaError {lib().w4_last_cuda_error()})"
            except Exception:
                pass
        super().__init__(msg)


class GemvDesc(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int),
        ("packed", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("codebook", ctypes.c_void_p),
        ("x", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
        ("M", ctypes.c_int),
        ("N", ctypes.c_int),
        ("K", ctypes.c_int),
        ("blocksize", ctypes.c_int),
        ("level", ctypes.c_int),
    ]


class GemvPlan(ctypes.Structure):
    """w4_gemv_plan_t of include/w4.h."""
    _fields_ = [(name, ctypes.c_int) for name in
                ("kernel", "launches", "batch_tile", "threads", "smem_bytes", "stages", "grid", "cluster")]


_lib = None


def _declare(L):
    P, I, V = ctypes.c_void_p, ctypes.c_int, None
    sig = {
        "w4_nf4_codebook": (I, [P]),
        "w4_quantize_nf4": (I, [P, P, P, P, I, I, I, P]),
        "w4_quantize_int4": (I, [P, P, P, I, I, I, P]),
        "w4_dequantize_nf4": (I, [P, P, P, P, I, I, I, P]),
        "w4_dequantize_int4": (I, [P, P, P, I, I, I, P]),
        "w4_gemv_nf4": (I, [P, P, P, P, P, I, I, I, I, P]),
        "w4_gemv_int4": (I, [P, P, P, P, I, I, I, I, P]),
        "w4_quantize_fp4": (I, [P, P, P, I, I, I, P]),
        "w4_dequantize_fp4": (I, [P, P, P, I, I, I, P]),
        "w4_gemv_fp4": (I, [P, P, P, P, I, I, I, I, P]),
        "w4_gemv_sequence": (I, [ctypes.POINTER(GemvDesc), I, P]),
        "w4_step_workspace_bytes": (ctypes.c_int64, [I]),
        "w4_step_create": (I, [ctypes.POINTER(GemvDesc), I, P, ctypes.POINTER(P)]),
        "w4_step_launch": (I, [P, P]),
        "w4_step_destroy": (I, [P]),
        "w4_step_run_host": (I, [P, P, P, ctypes.c_int64, P, P, ctypes.c_int64, P]),
        "w4_status_str": (ctypes.c_char_p, [I]),
        "w4_last_cuda_error": (I, []),
        "w4_device_check": (I, [P]),
        "w4_launch_count": (ctypes.c_longlong, []),
        "w4_inject_timeout_once": (I, []),
        "w4_gemv_levels_noalloc": (I, [ctypes.POINTER(GemvDesc), I, P]),
        "w4_gemv_plan": (I, [I, I, I, I, I, I, ctypes.POINTER(GemvPlan)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded libw4 (raises W4Error if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise W4Error(W4_ERR_UNSUPPORTED, f"{LIB_PATH} is missing; build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib
