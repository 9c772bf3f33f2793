"""ctypes loader for libgb300attn.so and the raw C-ABI signatures (include/attn.h).

The library is required: importing the bindings on a machine without the
built shared object raises immediately; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

ATTN_STATUS = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_WORKSPACE",
    5: "ATTN_ERR_CUDA",
    6: "ATTN_ERR_TIMEOUT",
}

# Every symbol include/attn.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_workspace_size": (ctypes.c_size_t, [_I]),
    "attn_fwd_ws": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, ctypes.c_size_t, _P]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, ctypes.c_size_t, _P]),
    "attn_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "attn_decode_default_splits": (_I, [_I, _I, _I]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t, _P]),
    "attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_kv_quantize_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "attn_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t,
                             _P]),
    "rmsnorm_fwd": (_I, [_P, _P, _P, _I, _I, _F, _P]),
    "rmsnorm_residual_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _F, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_last_device_error": (_I, [_P]),
    "attn_kernel_launches": (ctypes.c_ulonglong, []),
    "attn_selftest_wait_timeout": (_I, [_I, _P]),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {ATTN_STATUS.get(status, status)}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and type the shared library; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m exact_tiled_attention_attn_gb300.build` "
            "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise AttnError(fn, status)
