"""ctypes front end of the C oracle (``pa_oracle.c``).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
CPU-baseline leg may call it.  Inputs are numpy arrays; nothing here touches
a GPU.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from .build import LIB, build_oracle

_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build_oracle()
        L = ctypes.CDLL(LIB)
        L.pa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.pa_oracle_half_to_double.restype = ctypes.c_double
        L.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.pa_oracle_bf16_to_double.restype = ctypes.c_double
        L.pa_oracle_locate_kv.argtypes = [_I64, _P, _I, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]
        L.pa_oracle_locate_kv.restype = _I
        L.pa_oracle_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I]
        L.pa_oracle_reshape_and_cache.restype = _I
        L.pa_oracle_decode.argtypes = [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I64,
                                       ctypes.c_double, _I, _I, _I, ctypes.c_double, ctypes.c_double]
        L.pa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.pa_oracle_e4m3_to_double.restype = ctypes.c_double
        L.pa_oracle_quantize_e4m3.argtypes = [ctypes.c_float, ctypes.c_float]
        L.pa_oracle_quantize_e4m3.restype = ctypes.c_uint8
        L.pa_oracle_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I,
                                                      ctypes.c_float, ctypes.c_float]
        L.pa_oracle_reshape_and_cache_fp8.restype = _I
        L.pa_oracle_decode.restype = _I
        L.pa_oracle_prefill.argtypes = [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I64,
                                        ctypes.c_double, _I, _I, _I, ctypes.c_double, ctypes.c_double]
        L.pa_oracle_prefill.restype = _I
        L.pa_oracle_copy_blocks.argtypes = [_P, _P, _P, _I64, _I64, _I, _I, _I]
        L.pa_oracle_copy_blocks.restype = _I
        L.pa_oracle_max_threads.argtypes = []
        L.pa_oracle_max_threads.restype = _I
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def half_to_double(bits: int) -> float:
    return lib().pa_oracle_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return lib().pa_oracle_bf16_to_double(int(bits) & 0xFFFF)


DTYPES = {"fp16": 0, "bf16": 1, "fp8": 2}


def e4m3_to_double(bits: int) -> float:
    return lib().pa_oracle_e4m3_to_double(int(bits) & 0xFF)


def quantize_e4m3(x: float, scale: float) -> int:
    return int(lib().pa_oracle_quantize_e4m3(float(x), float(scale)))


def reshape_and_cache_fp8(key: np.ndarray, value: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                          slot_mapping: np.ndarray, k_scale: float, v_scale: float,
                          dtype: str = "fp16", inplace: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Return the E4M3 pools (uint8) after quantising and writing the new
    tokens (key/value: float16, or bfloat16 bit patterns): copies, or with
    inplace=True the given (contiguous) pools themselves."""
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    if inplace:
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        kc, vc = k_cache, v_cache
    else:
        kc = np.ascontiguousarray(k_cache).copy()
        vc = np.ascontiguousarray(v_cache).copy()
    N, B, Hk, d = kc.shape
    key = np.ascontiguousarray(key)
    value = np.ascontiguousarray(value)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = lib().pa_oracle_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc), _ptr(sm),
                                               int(sm.size), N, B, Hk, d, DTYPES[dtype], float(k_scale),
                                               float(v_scale))
    if rc:
        raise OracleError(f"reshape_and_cache_fp8 precondition failed ({rc})")
    return kc, vc


def locate_kv(logical_token_idx: int, block_table, block_size: int) -> Tuple[int, int]:
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    phys = ctypes.c_int32()
    off = ctypes.c_int32()
    rc = lib().pa_oracle_locate_kv(int(logical_token_idx), _ptr(bt), int(block_size),
                                   ctypes.byref(phys), ctypes.byref(off))
    if rc:
        raise OracleError(f"locate_kv failed ({rc})")
    return int(phys.value), int(off.value)


def reshape_and_cache(key: np.ndarray, value: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: np.ndarray, inplace: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Return the pools after the write: updated copies (inputs untouched), or
    the given pools themselves, written in place, with ``inplace=True``."""
    assert key.itemsize == 2 and value.itemsize == 2  # float16, or bfloat16 bit patterns
    if inplace:
        assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
        kc, vc = k_cache, v_cache
    else:
        kc = np.ascontiguousarray(k_cache).copy()
        vc = np.ascontiguousarray(v_cache).copy()
    N, B, Hk, d = kc.shape
    key = np.ascontiguousarray(key)
    value = np.ascontiguousarray(value)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = lib().pa_oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc), _ptr(sm),
                                           int(sm.size), N, B, Hk, d)
    if rc:
        raise OracleError(f"reshape_and_cache precondition failed ({rc})")
    return kc, vc


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_mapping) -> Tuple[np.ndarray, np.ndarray]:
    """Return copies of the pools after copying the (src, dst) blocks.  The
    copy moves whole blocks of bytes, so one-byte (E4M3) pools go through as
    16-bit elements, two codes to an element."""
    kc = np.ascontiguousarray(k_cache).copy()
    vc = np.ascontiguousarray(v_cache).copy()
    N, B, Hk, d = kc.shape
    if kc.itemsize == 1:
        assert d % 2 == 0
        d //= 2
    bm = np.ascontiguousarray(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2))
    rc = lib().pa_oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(bm), int(bm.shape[0]), N, B, Hk, d)
    if rc:
        raise OracleError(f"copy_blocks precondition failed ({rc})")
    return kc, vc


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
           context_lens: np.ndarray, scale: float, num_threads: int = 0, dtype: str = "fp16",
           k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """float64 attention output [S, H, d].  q and the caches are float16
    arrays, or (dtype="bf16") uint16 arrays of bfloat16 bit patterns; uint8
    caches are E4M3 codes whose values are multiplied by k_scale / v_scale."""
    cache_dtype = "fp8" if k_cache.dtype == np.uint8 else dtype
    assert q.itemsize == 2 and k_cache.dtype == v_cache.dtype
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, H, d = q.shape
    N, B, Hk, d2 = k_cache.shape
    assert d == d2 and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, H, d), dtype=np.float64)
    rc = lib().pa_oracle_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                int(bt.shape[1]), _ptr(cl), S, H, Hk, d, B, N, float(scale),
                                int(num_threads), DTYPES[dtype], DTYPES[cache_dtype], float(k_scale),
                                float(v_scale))
    if rc:
        raise OracleError(f"decode precondition failed ({rc})")
    return out


def prefill(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
            context_lens: np.ndarray, query_start_loc: np.ndarray, scale: float, num_threads: int = 0,
            dtype: str = "fp16", k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """float64 prefill output [rows, H, d]: row i of sequence s (rows
    query_start_loc[s] .. query_start_loc[s+1]) attends causally up to its
    position ctx - qlen + i.  Element types as decode()."""
    cache_dtype = "fp8" if k_cache.dtype == np.uint8 else dtype
    assert q.itemsize == 2 and k_cache.dtype == v_cache.dtype
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    R, H, d = q.shape
    N, B, Hk, _ = k_cache.shape
    S = int(cl.size)
    assert qsl.size == S + 1 and int(qsl[-1]) == R
    out = np.zeros((R, H, d), dtype=np.float64)
    rc = lib().pa_oracle_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), int(bt.shape[1]),
                                 _ptr(cl), _ptr(qsl), S, H, Hk, d, B, N, float(scale), int(num_threads),
                                 DTYPES[dtype], DTYPES[cache_dtype], float(k_scale), float(v_scale))
    if rc:
        raise OracleError(f"prefill precondition failed ({rc})")
    return out


def max_threads() -> int:
    return int(lib().pa_oracle_max_threads())
