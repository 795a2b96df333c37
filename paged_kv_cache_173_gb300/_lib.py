"""ctypes loader for ``libpagedattn.so`` (the C ABI in include/pagedattn.h).

The library is built in-tree (``python -m paged_kv_cache_173_gb300.build`` or
``__graft_entry__.build()``).  There is no fallback: if the library is
missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedattn.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_FP16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2

# Every function the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "pa_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pa_copy_blocks": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pa_decode": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "pa_splitk_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "pa_decode_splitk": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I,
                              _P, _SZ, _P]),
    "pa_splitk_reduce": (_I, [_P, _P, _SZ, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "pa_decode_splitk_static": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                                     _P]),
    "pa_reshape_and_cache_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _P]),
    "pa_decode_fp8": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _F, _F, _P]),
    "pa_decode_splitk_fp8": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _F, _F, _I,
                                  _I, _P, _SZ, _P]),
    "pa_decode_prefix_splitk": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _F, _F,
                                     _I, _P, _I, _I, _P, _SZ, _P]),
    "pa_append_and_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _F, _F,
                                  _P]),
    "pa_append_and_decode_splitk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _F,
                                         _F, _I, _I, _P, _SZ, _P]),
    "pa_prefill": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "pa_selftest_wait": (_I, [_P, ctypes.c_uint, _P]),
    "pa_status_string": (ctypes.c_char_p, [_I]),
    "pa_last_error": (ctypes.c_char_p, []),
}

_lib: Optional[ctypes.CDLL] = None
_lock = threading.Lock()


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} failed: {status_name(status)} ({status}): {detail}")
        self.status = status


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build the CUDA library first "
                        "(python -m paged_kv_cache_173_gb300.build)")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    f = getattr(L, name)
                    f.restype = res
                    f.argtypes = args
                _lib = L
    return _lib


def status_name(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def last_error() -> str:
    return lib().pa_last_error().decode()


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(fn, status, last_error())
