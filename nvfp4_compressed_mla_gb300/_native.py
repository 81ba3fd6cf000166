"""ctypes declarations of the C ABI in include/nvfp4_mla.h (no logic here)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
F32 = ctypes.c_float
SZ = ctypes.c_size_t

SIGNATURES = {
    "nvfp4_mla_row_bytes": (I32, [I32]),
    "nvfp4_mla_status_string": (ctypes.c_char_p, [I32]),
    "nvfp4_mla_append": (I32, [P, P, P, P, I32, P, I32, I32, I32, P, I64, I64, I32, F32, F32,
                               P, P]),
    "sparse_mla_decode_num_splits": (I32, [I32, I32, I32]),
    "nvfp4_mla_set_wait_limit": (I32, [I64]),
    "sparse_mla_decode_workspace_size": (SZ, [I32, I32, I32, I32]),
    "sparse_mla_decode": (I32, [P, P, P, P, I32, I32, I32, P, I32, I32, P, I32, P, I64, I64, I32,
                                F32, F32, F32, P, I32, P, P, SZ, I32, P, P]),
    "sparse_mla_decode_noalloc": (I32, [P, P, P, P, I32, I32, I32, P, I32, I32, P, I32, P, I64,
                                        I64, I32, F32, F32, F32, P, I32, P, I32, P, P]),
    "sparse_mla_merge_states": (I32, [P, P, I32, I32, I32, P, I32, P, P]),
    "nvfp4_mla_staged_rows_per_q": (I64, [I32, I32]),
    "nvfp4_mla_stage_fp8": (I32, [P, P, I32, I32, P, I32, I32, P, I32, P, I64, I64, F32, P, P,
                                  P, P]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the CUDA library; build it first if it is missing or stale.

    Raises if it cannot be built or loaded: there is no fallback path.
    """
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise ImportError(f"CUDA library not built: {path}")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
