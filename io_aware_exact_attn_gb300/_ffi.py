"""ctypes declarations of the C ABI in ``include/attn.h``.

Loading fails loudly if ``libattn.so`` has not been built: there is no
fallback implementation of any entry point.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

c_void_p, c_int, c_float, c_int64, c_size_t = C.c_void_p, C.c_int, C.c_float, C.c_int64, C.c_size_t


class attn_trace_record_t(C.Structure):
    _fields_ = [("kernel", C.c_int32), ("ms", C.c_float)]


KERNEL_NAMES = {1: "fwd", 2: "partial_fwd", 3: "merge", 4: "bwd_preprocess", 5: "bwd_dkdv", 6: "bwd_dq",
                7: "selftest", 8: "decode", 9: "varlen_fwd", 10: "fp8_transpose_v", 11: "fwd_fp8"}


class attn_mask_t(C.Structure):
    _fields_ = [("kind", C.c_int32), ("causal_in_blocks", C.c_int32), ("block_mask", C.c_void_p),
                ("window", C.c_int32)]


MASK_NONE, MASK_CAUSAL, MASK_BLOCK_SPARSE, MASK_SLIDING_WINDOW = 0, 1, 2, 3
DTYPE_BF16, DTYPE_F32 = 0, 1
STATUS = {0: "ATTN_OK", -1: "ATTN_ERR_INVALID_ARG", -2: "ATTN_ERR_UNSUPPORTED", -3: "ATTN_ERR_MISALIGNED",
          -4: "ATTN_ERR_CUDA", -5: "ATTN_ERR_DEVICE_TIMEOUT", -6: "ATTN_ERR_WORKSPACE",
          -7: "ATTN_ERR_NO_DEVICE", -8: "ATTN_ERR_DEVICE_BOUNDS"}

# name -> (restype, argtypes); the full exported surface of attn.h
SIGNATURES = {
    "attn_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                         c_float, C.POINTER(attn_mask_t), c_void_p]),
    "attn_partial_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_float, C.POINTER(attn_mask_t), c_int64, c_int64, c_int64,
                                 c_int64, c_void_p]),
    "attn_merge_lse": (c_int, [C.POINTER(c_void_p), C.POINTER(c_void_p), c_int, c_void_p, c_int, c_void_p, c_int,
                               c_int, c_int, c_int, c_int64, c_void_p]),
    "attn_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         c_void_p, c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_int, c_float,
                         C.POINTER(attn_mask_t), c_void_p]),
    "attn_bwd_static_scratch": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                                        C.POINTER(attn_mask_t), c_void_p]),
    "attn_bwd_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_bwd_preprocess": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int64, c_void_p,
                                    c_size_t, c_void_p]),
    "attn_partial_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p,
                                 c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                 C.POINTER(attn_mask_t), c_int64, c_int64, c_int64, c_int64, c_int, c_void_p]),
    "attn_varlen_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int64,
                                c_int, c_int, c_int, c_float, C.POINTER(attn_mask_t), c_void_p]),
    "attn_varlen_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_int, c_int, c_int64, c_int, c_int, c_int, c_float,
                                C.POINTER(attn_mask_t), c_void_p, c_size_t, c_void_p]),
    "attn_varlen_bwd_workspace_bytes": (c_size_t, [c_int, c_int64, c_int]),
    "attn_fwd_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_float, c_float, c_float, c_void_p, c_void_p, c_int,
                             c_int, c_int, c_int, c_int, c_float, C.POINTER(attn_mask_t), c_void_p, c_size_t,
                             c_void_p]),
    "attn_fwd_fp8_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int]),
    "attn_decode_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                c_int, c_int, c_int, c_float, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "attn_decode_splits": (c_int, [c_int, c_int, c_int]),
    "attn_decode_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int, c_int]),
    "attn_build_schedule": (c_int, [c_int, c_int, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                    c_int64, c_int64, C.POINTER(C.c_int32), c_size_t, C.POINTER(c_size_t)]),
    "attn_build_chunk_schedule": (c_int, [c_int, c_int, C.POINTER(C.c_int32), c_size_t, C.POINTER(c_size_t)]),
    "attn_get_status": (c_int, [c_void_p]),
    "attn_set_wait_limit_ns": (None, [c_int64]),
    "attn_debug_set_tile_counts": (c_int, [c_void_p, c_int64]),
    "attn_selftest_wait_timeout": (c_int, [c_int64, c_void_p]),
    "attn_trace_enable": (c_int, [c_int]),
    "attn_trace_disable": (c_int, []),
    "attn_trace_read": (c_int, [C.POINTER(attn_trace_record_t), c_int, C.POINTER(c_int)]),
    "attn_status_string": (C.c_char_p, [c_int]),
    "attn_last_error_message": (C.c_char_p, []),
    "attn_version": (c_int, []),
}

_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            h = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
        return _lib


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().attn_last_error_message().decode(errors="replace")
        super().__init__(f"{where}: {STATUS.get(code, code)}: {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != 0:
        raise AttnError(code, where)
