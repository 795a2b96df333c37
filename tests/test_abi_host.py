"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host (no kernel is launched, so no GPU is needed)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from paged_kv_cache_173_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_173_gb300.build import build_library
    build_library()
    return _lib.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert {"pa_reshape_and_cache", "pa_decode", "pa_decode_splitk", "pa_splitk_reduce",
            "pa_splitk_workspace_bytes", "pa_status_string", "pa_last_error"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
        assert n in _lib.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(L):
    assert _lib.status_name(0) == "PA_OK"
    assert _lib.status_name(-1) == "PA_ERR_INVALID_ARG"
    assert _lib.status_name(-2) == "PA_ERR_UNSUPPORTED"
    assert _lib.status_name(-3) == "PA_ERR_CUDA"
    assert _lib.status_name(7) == "PA_UNKNOWN_STATUS"


def test_workspace_size(L):
    assert L.pa_splitk_workspace_bytes(4, 32, 128, 256) == 4 * 32 * 256 * (128 + 2) * 4
    assert L.pa_splitk_workspace_bytes(0, 32, 128, 256) == 0
    assert L.pa_splitk_workspace_bytes(4, 32, 128, -1) == 0


A = 1 << 20  # a fake, 16-byte aligned "device" address: never dereferenced on these paths


def _decode(L, **kw):
    args = dict(out=A, q=A, k=A, v=A, bt=A, M=8, cl=A, S=2, H=8, Hk=2, d=128, B=16, N=32,
                scale=0.1, dtype=0, stream=None)
    args.update(kw)
    return L.pa_decode(args["out"], args["q"], args["k"], args["v"], args["bt"], args["M"], args["cl"],
                       args["S"], args["H"], args["Hk"], args["d"], args["B"], args["N"], args["scale"],
                       args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(dtype=2), _lib.PA_ERR_UNSUPPORTED),
    (dict(d=256, H=32, Hk=2), _lib.PA_ERR_UNSUPPORTED),  # head_dim 256: query groups up to 8
    (dict(H=6, Hk=4), _lib.PA_ERR_UNSUPPORTED),
    (dict(H=64, Hk=2), _lib.PA_ERR_UNSUPPORTED),
    (dict(B=8), _lib.PA_ERR_UNSUPPORTED),
    (dict(B=24), _lib.PA_ERR_UNSUPPORTED),
    (dict(B=48), _lib.PA_ERR_UNSUPPORTED),
    (dict(B=512), _lib.PA_ERR_UNSUPPORTED),
    (dict(S=-1), _lib.PA_ERR_INVALID_ARG),
    (dict(S=70000), _lib.PA_ERR_UNSUPPORTED),
    (dict(M=0), _lib.PA_ERR_INVALID_ARG),
    (dict(N=0), _lib.PA_ERR_INVALID_ARG),
    (dict(q=None), _lib.PA_ERR_INVALID_ARG),
    (dict(bt=None), _lib.PA_ERR_INVALID_ARG),
    (dict(out=A + 2), _lib.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _lib.PA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments(L, kw, status):
    assert _decode(L, **kw) == status
    assert _lib.last_error() != ""


def test_empty_batch_is_a_no_op(L):
    assert _decode(L, S=0, q=None, out=None) == _lib.PA_OK
    assert L.pa_reshape_and_cache(A, A, A, A, A, 0, 8, 16, 2, 128, 0, None) == _lib.PA_OK


def _splitk(L, **kw):
    args = dict(ps=64, P=2, ws=A, wsb=10 ** 9, B=16, M=8)
    args.update(kw)
    return L.pa_decode_splitk(A, A, A, A, A, args["M"], A, 2, 8, 2, 128, args["B"], 32, 0.1, 0,
                              args["ps"], args["P"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw", [dict(ps=40), dict(ps=0), dict(P=1), dict(ws=None), dict(wsb=100),
                                dict(ws=A + 4), dict(P=70000)])
def test_splitk_rejects_bad_arguments(L, kw):
    assert _splitk(L, **kw) in (_lib.PA_ERR_INVALID_ARG, _lib.PA_ERR_UNSUPPORTED)


def test_reduce_rejects_bad_arguments(L):
    bad_ps = L.pa_splitk_reduce(A, A, 10 ** 9, A, 8, 16, 2, 8, 128, 40, 8, 0, None)
    assert bad_ps == _lib.PA_ERR_INVALID_ARG
    small_ws = L.pa_splitk_reduce(A, A, 16, A, 8, 16, 2, 8, 128, 64, 2, 0, None)
    assert small_ws == _lib.PA_ERR_INVALID_ARG
    assert "workspace" in _lib.last_error()


@pytest.mark.parametrize("args,status", [
    ((A, A, A, A, A, 4, 8, 16, 2, 100, 0, None), _lib.PA_ERR_UNSUPPORTED),   # head_dim % 8
    ((A, A, A, A, A, -1, 8, 16, 2, 128, 0, None), _lib.PA_ERR_INVALID_ARG),  # negative T
    ((A, A, A, A, None, 4, 8, 16, 2, 128, 0, None), _lib.PA_ERR_INVALID_ARG),
    ((A, A, A + 8, A, A, 4, 8, 16, 2, 128, 0, None), _lib.PA_ERR_INVALID_ARG),
    ((A, A, A, A, A, 4, 8, 16, 2, 128, 3, None), _lib.PA_ERR_UNSUPPORTED),
])
def test_reshape_rejects_bad_arguments(L, args, status):
    assert L.pa_reshape_and_cache(*args) == status


def _decode_fp8(L, splitk=False, **kw):
    args = dict(S=2, H=8, Hk=2, d=128, B=16, dtype=0, ks=0.03125, vs=0.03125, q=A)
    args.update(kw)
    head = (A, args["q"], A, A, A, 8, A, args["S"], args["H"], args["Hk"], args["d"], args["B"], 32, 0.1,
            args["dtype"], args["ks"], args["vs"])
    if splitk:
        return L.pa_decode_splitk_fp8(*head, 64, 2, A, 10 ** 9, None)
    return L.pa_decode_fp8(*head, None)


@pytest.mark.parametrize("splitk", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(dtype=1), _lib.PA_ERR_UNSUPPORTED),          # E4M3 caches take float16 queries
    (dict(dtype=2), _lib.PA_ERR_UNSUPPORTED),
    (dict(ks=0.0), _lib.PA_ERR_INVALID_ARG),
    (dict(vs=-1.0), _lib.PA_ERR_INVALID_ARG),
    (dict(ks=float("inf")), _lib.PA_ERR_INVALID_ARG),
    (dict(vs=float("nan")), _lib.PA_ERR_INVALID_ARG),
    (dict(d=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(B=8), _lib.PA_ERR_UNSUPPORTED),
    (dict(q=None), _lib.PA_ERR_INVALID_ARG),
    (dict(S=0, q=None), _lib.PA_OK),
])
def test_fp8_decode_checks_arguments(L, splitk, kw, status):
    assert _decode_fp8(L, splitk=splitk, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((A, A, A, A, A, 4, 8, 16, 2, 40, 0, 1.0, 1.0, None), _lib.PA_ERR_UNSUPPORTED),   # head_dim % 16
    ((A, A, A, A, A, 4, 8, 16, 2, 128, 2, 1.0, 1.0, None), _lib.PA_ERR_UNSUPPORTED),  # key dtype
    ((A, A, A, A, A, 4, 8, 16, 2, 128, 0, 0.0, 1.0, None), _lib.PA_ERR_INVALID_ARG),
    ((A, A, A, A, A, 4, 8, 16, 2, 128, 0, 1.0, float("inf"), None), _lib.PA_ERR_INVALID_ARG),
    ((A, A, A + 8, A, A, 4, 8, 16, 2, 128, 0, 1.0, 1.0, None), _lib.PA_ERR_INVALID_ARG),
    ((A, A, A, A, A, 0, 8, 16, 2, 128, 1, 1.0, 1.0, None), _lib.PA_OK),              # empty
])
def test_fp8_reshape_checks_arguments(L, args, status):
    assert L.pa_reshape_and_cache_fp8(*args) == status


def test_copy_blocks_accepts_one_byte_caches(L):
    assert L.pa_copy_blocks(A, A, A, 0, 8, 16, 2, 128, _lib.PA_FP8_E4M3, None) == _lib.PA_OK
    assert L.pa_copy_blocks(A, A, A, 0, 8, 16, 2, 128, 3, None) == _lib.PA_ERR_UNSUPPORTED
    # 1-byte elements: 16 * 1 * 8 = 128 bytes per block, a multiple of 16
    assert L.pa_copy_blocks(A, A, A, 0, 8, 16, 1, 8, _lib.PA_FP8_E4M3, None) == _lib.PA_OK


def _prefill(L, **kw):
    a = dict(S=2, maxq=64, H=8, Hk=2, d=128, B=16, qsl=A, dtype=0)
    a.update(kw)
    return L.pa_prefill(A, A, A, A, A, 8, A, a["qsl"], a["S"], 100, a["maxq"], a["H"], a["Hk"], a["d"], a["B"], 32,
                        0.1, a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=256), _lib.PA_ERR_UNSUPPORTED),          # prefill: head_dim 64 or 128
    (dict(H=6, Hk=2), _lib.PA_ERR_UNSUPPORTED),      # a query group of 3 does not divide 128
    (dict(dtype=2), _lib.PA_ERR_UNSUPPORTED),
    (dict(qsl=None), _lib.PA_ERR_INVALID_ARG),
    (dict(qsl=A + 2), _lib.PA_ERR_INVALID_ARG),
    (dict(maxq=-1), _lib.PA_ERR_INVALID_ARG),
    (dict(B=8), _lib.PA_ERR_UNSUPPORTED),
    (dict(S=0, qsl=None), _lib.PA_OK),
    (dict(maxq=0, qsl=None), _lib.PA_OK),
])
def test_prefill_checks_arguments(L, kw, status):
    assert _prefill(L, **kw) == status


@pytest.mark.parametrize("args", [(None, 1000), (A, 0), (A, 10_000_001), (A + 2, 1000)])
def test_wait_selftest_checks_arguments(L, args):
    assert L.pa_selftest_wait(args[0], args[1], None) == _lib.PA_ERR_INVALID_ARG


def _append(L, splitk=False, **kw):
    args = dict(out=A, q=A, key=A, value=A, k=A, v=A, S=2, H=8, Hk=2, d=128, dtype=0, kv=0, ks=1.0, vs=1.0,
                ps=64, P=2, ws=A, wsb=10 ** 9)
    args.update(kw)
    head = (args["out"], args["q"], args["key"], args["value"], args["k"], args["v"], A, 8, A, args["S"],
            args["H"], args["Hk"], args["d"], 16, 32, 0.1, args["dtype"], args["kv"], args["ks"], args["vs"])
    if splitk:
        return L.pa_append_and_decode_splitk(*head, args["ps"], args["P"], args["ws"], args["wsb"], None)
    return L.pa_append_and_decode(*head, None)


@pytest.mark.parametrize("splitk", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(key=None), _lib.PA_ERR_INVALID_ARG),
    (dict(value=A + 8), _lib.PA_ERR_INVALID_ARG),
    (dict(kv=1), _lib.PA_ERR_UNSUPPORTED),                 # 16-bit pools of another type than q
    (dict(dtype=1, kv=2), _lib.PA_ERR_UNSUPPORTED),        # E4M3 pools take fp16 queries
    (dict(kv=2, ks=0.0), _lib.PA_ERR_INVALID_ARG),
    (dict(kv=2, vs=float("nan")), _lib.PA_ERR_INVALID_ARG),
    (dict(d=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(k=None), _lib.PA_ERR_INVALID_ARG),
])
def test_append_rejects_bad_arguments(L, splitk, kw, status):
    assert _append(L, splitk, **kw) == status
    assert _lib.last_error() != ""


@pytest.mark.parametrize("kw", [dict(ps=40), dict(P=1), dict(ws=None), dict(wsb=100)])
def test_append_splitk_rejects_bad_workspace(L, kw):
    assert _append(L, True, **kw) == _lib.PA_ERR_INVALID_ARG


def test_append_empty_batch_is_a_no_op(L):
    assert _append(L, S=0, key=None, value=None, q=None, out=None) == _lib.PA_OK
    assert _append(L, True, S=0, key=None, value=None, ws=None) == _lib.PA_OK
