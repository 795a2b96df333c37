"""Python binding of the C ABI, one function per entry point, same names.

Argument marshalling only: shapes are read from the tensors, pointers and the
current CUDA stream are passed to ``libpagedattn.so``, and a non-zero status
raises ``PagedAttnError``.  Every step of the computation runs in the
library's kernels; PyTorch provides device memory and streams.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib
from ._lib import PA_BF16, PA_FP16, PA_FP8_E4M3, PagedAttnError  # noqa: F401  (re-exported)

_DTYPES = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16}
# E4M3 pools: uint8 codes, or torch's float8_e4m3fn (the same bytes)
_CODE_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}: float16 or bfloat16")
    return _DTYPES[t.dtype]


def _stream_ptr(t: torch.Tensor, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return int(t.data_ptr())


def _need_codes(t: torch.Tensor, name: str, device: torch.device) -> int:
    """Pointer of an E4M3 pool (uint8 or float8_e4m3fn, contiguous, on `device`)."""
    if not isinstance(t, torch.Tensor) or t.dtype not in _CODE_DTYPES:
        raise TypeError(f"{name} must be a uint8 or float8_e4m3fn tensor of E4M3 codes")
    return _need(t, name, t.dtype, device)


def _cuda_device(t: torch.Tensor) -> torch.device:
    if not t.is_cuda:
        raise ValueError("paged attention tensors must live on a CUDA device")
    return t.device


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write key/value [T, Hk, d] into the pools [N, B, Hk, d] at slot_mapping [T] (int64)."""
    dev = _cuda_device(k_cache)
    N, B, Hk, d = k_cache.shape
    T = key.shape[0]
    if key.shape != (T, Hk, d) or value.shape != (T, Hk, d) or v_cache.shape != k_cache.shape:
        raise ValueError("key/value must be [T, Hk, d] matching the pools [N, B, Hk, d]")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    dt = k_cache.dtype
    st = _lib.lib().pa_reshape_and_cache(
        _need(key, "key", dt, dev), _need(value, "value", dt, dev),
        _need(k_cache, "k_cache", dt, dev), _need(v_cache, "v_cache", dt, dev),
        _need(slot_mapping, "slot_mapping", torch.int64, dev), T, N, B, Hk, d, _dtype_code(k_cache),
        _stream_ptr(k_cache, stream))
    _lib.check("pa_reshape_and_cache", st)


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor,
                   stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy whole blocks: for each row (src, dst) of block_mapping [n, 2] (int64),
    k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src]."""
    dev = _cuda_device(k_cache)
    N, B, Hk, d = k_cache.shape
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be [n, 2]")
    dt = k_cache.dtype
    code = PA_FP8_E4M3 if dt in _CODE_DTYPES else _dtype_code(k_cache)
    st = _lib.lib().pa_copy_blocks(
        _need(k_cache, "k_cache", dt, dev), _need(v_cache, "v_cache", dt, dev),
        _need(block_mapping, "block_mapping", torch.int64, dev), int(block_mapping.shape[0]), N, B, Hk, d,
        code, _stream_ptr(k_cache, stream))
    _lib.check("pa_copy_blocks", st)


def _decode_common(out, q, k_cache, v_cache, block_tables, context_lens, codes: bool = False):
    dev = _cuda_device(q)
    S, H, d = q.shape
    N, B, Hk, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("q/out [S, H, d] must match the pools [N, B, Hk, d]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, M] and context_lens [S]")
    dt = q.dtype
    _dtype_code(q)
    if codes:
        pk, pv = _need_codes(k_cache, "k_cache", dev), _need_codes(v_cache, "v_cache", dev)
    else:
        pk, pv = _need(k_cache, "k_cache", dt, dev), _need(v_cache, "v_cache", dt, dev)
    ptrs = (_need(out, "out", dt, dev), _need(q, "q", dt, dev), pk, pv,
            _need(block_tables, "block_tables", torch.int32, dev))
    cl = _need(context_lens, "context_lens", torch.int32, dev)
    return dev, S, H, d, N, B, Hk, int(block_tables.shape[1]), ptrs, cl


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
              stream: Optional[torch.cuda.Stream] = None) -> None:
    """Single-pass paged decode: out[S, H, d] = attention of q over each sequence's paged KV."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens)
    st = _lib.lib().pa_decode(po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale), _dtype_code(q),
                              _stream_ptr(q, stream))
    _lib.check("pa_decode", st)


def pa_splitk_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int,
                              max_num_partitions: int) -> int:
    return int(_lib.lib().pa_splitk_workspace_bytes(num_seqs, num_heads, head_dim, max_num_partitions))


def max_num_partitions_for(max_blocks_per_seq: int, block_size: int, partition_size: int) -> int:
    return -(-(max_blocks_per_seq * block_size) // partition_size)


def pa_decode_splitk(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                     partition_size: int, workspace: torch.Tensor,
                     max_num_partitions: Optional[int] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> None:
    """Split-K paged decode; follow with pa_splitk_reduce on the same stream."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens)
    P = max_num_partitions or max_num_partitions_for(M, B, partition_size)
    ws = _need(workspace, "workspace", workspace.dtype, dev)
    st = _lib.lib().pa_decode_splitk(po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale),
                                     _dtype_code(q), int(partition_size), int(P), ws,
                                     workspace.numel() * workspace.element_size(),
                                     _stream_ptr(q, stream))
    _lib.check("pa_decode_splitk", st)


def pa_splitk_reduce(out: torch.Tensor, workspace: torch.Tensor, context_lens: torch.Tensor,
                     max_blocks_per_seq: int, block_size: int, partition_size: int,
                     max_num_partitions: Optional[int] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> None:
    """Merge the partitions of pa_decode_splitk into out[S, H, d]."""
    dev = _cuda_device(out)
    S, H, d = out.shape
    P = max_num_partitions or max_num_partitions_for(max_blocks_per_seq, block_size, partition_size)
    st = _lib.lib().pa_splitk_reduce(
        _need(out, "out", out.dtype, dev), _need(workspace, "workspace", workspace.dtype, dev),
        workspace.numel() * workspace.element_size(), _need(context_lens, "context_lens", torch.int32, dev),
        int(max_blocks_per_seq), int(block_size), S, H, d, int(partition_size), int(P), _dtype_code(out),
        _stream_ptr(out, stream))
    _lib.check("pa_splitk_reduce", st)


def pa_decode_splitk_static(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, scale: float, partition_size: int,
                            stream: Optional[torch.cuda.Stream] = None) -> None:
    """Split-K decode + reduce for callers that cannot allocate device memory:
    the partials go to a fixed array inside the library (at most
    PA_STATIC_SCRATCH_BYTES, 32 MiB).  Calls that overlap on the GPU race on
    that array; the first call on a device should precede any stream capture."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens)
    st = _lib.lib().pa_decode_splitk_static(po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N,
                                            float(scale), _dtype_code(q), int(partition_size),
                                            _stream_ptr(q, stream))
    _lib.check("pa_decode_splitk_static", st)


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                             v_scale: float, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Quantise key/value [T, Hk, d] (float16 or bfloat16) into the E4M3 pools
    [N, B, Hk, d] (uint8 codes) at slot_mapping [T]: code = E4M3(x / scale)."""
    dev = _cuda_device(k_cache)
    N, B, Hk, d = k_cache.shape
    T = key.shape[0]
    if key.shape != (T, Hk, d) or value.shape != (T, Hk, d) or v_cache.shape != k_cache.shape:
        raise ValueError("key/value must be [T, Hk, d] matching the pools [N, B, Hk, d]")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    dt = key.dtype
    st = _lib.lib().pa_reshape_and_cache_fp8(
        _need(key, "key", dt, dev), _need(value, "value", dt, dev),
        _need_codes(k_cache, "k_cache", dev), _need_codes(v_cache, "v_cache", dev),
        _need(slot_mapping, "slot_mapping", torch.int64, dev), T, N, B, Hk, d, _dtype_code(key),
        float(k_scale), float(v_scale), _stream_ptr(k_cache, stream))
    _lib.check("pa_reshape_and_cache_fp8", st)


def pa_decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, k_scale: float,
                  v_scale: float, stream: Optional[torch.cuda.Stream] = None) -> None:
    """pa_decode over E4M3 pools whose values are code * k_scale (K) and code * v_scale (V)."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens, codes=True)
    st = _lib.lib().pa_decode_fp8(po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale),
                                  _dtype_code(q), float(k_scale), float(v_scale), _stream_ptr(q, stream))
    _lib.check("pa_decode_fp8", st)


def pa_decode_splitk_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                         k_scale: float, v_scale: float, partition_size: int, workspace: torch.Tensor,
                         max_num_partitions: Optional[int] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Split-K decode over E4M3 pools; follow with pa_splitk_reduce on the same stream."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens, codes=True)
    P = max_num_partitions or max_num_partitions_for(M, B, partition_size)
    ws = _need(workspace, "workspace", workspace.dtype, dev)
    st = _lib.lib().pa_decode_splitk_fp8(po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale),
                                         _dtype_code(q), float(k_scale), float(v_scale), int(partition_size),
                                         int(P), ws, workspace.numel() * workspace.element_size(),
                                         _stream_ptr(q, stream))
    _lib.check("pa_decode_splitk_fp8", st)


def pa_decode_prefix_splitk(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                            seqs_per_group: int, prefix_lens: torch.Tensor, partition_size: int,
                            workspace: torch.Tensor, max_num_partitions: Optional[int] = None,
                            k_scale: float = 1.0, v_scale: float = 1.0,
                            stream: Optional[torch.cuda.Stream] = None) -> None:
    """Split-K decode that reads each group's shared prompt blocks once: sequences
    [j*seqs_per_group, (j+1)*seqs_per_group) share their first prefix_lens[j] tokens
    (int32 [ceil(S / seqs_per_group)], multiples of partition_size).  E4M3 pools
    (uint8 / float8_e4m3fn) take k_scale and v_scale.  Follow with pa_splitk_reduce."""
    codes = k_cache.dtype in _CODE_DTYPES
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl = _decode_common(
        out, q, k_cache, v_cache, block_tables, context_lens, codes=codes)
    ngroups = -(-S // int(seqs_per_group)) if seqs_per_group > 0 else 0
    if prefix_lens.shape != (ngroups,):
        raise ValueError(f"prefix_lens must be [{ngroups}] (one entry per group)")
    P = max_num_partitions or max_num_partitions_for(M, B, partition_size)
    ws = _need(workspace, "workspace", workspace.dtype, dev)
    dt = _dtype_code(q)
    kv = PA_FP8_E4M3 if codes else dt
    st = _lib.lib().pa_decode_prefix_splitk(
        po, pq, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale), dt, kv, float(k_scale), float(v_scale),
        int(seqs_per_group), _need(prefix_lens, "prefix_lens", torch.int32, dev), int(partition_size), int(P), ws,
        workspace.numel() * workspace.element_size(), _stream_ptr(q, stream))
    _lib.check("pa_decode_prefix_splitk", st)


def _append_common(out, q, key, value, k_cache, v_cache, block_tables, context_lens):
    codes = k_cache.dtype in _CODE_DTYPES
    dev, S, H, d, N, B, Hk, M, ptrs, pcl = _decode_common(out, q, k_cache, v_cache, block_tables, context_lens,
                                                          codes=codes)
    if key.shape != (S, Hk, d) or value.shape != (S, Hk, d):
        raise ValueError("key/value must be [S, Hk, d]: one new token per sequence")
    pkey, pval = _need(key, "key", q.dtype, dev), _need(value, "value", q.dtype, dev)
    dt = _dtype_code(q)
    return dev, S, H, d, N, B, Hk, M, ptrs, pcl, pkey, pval, dt, (PA_FP8_E4M3 if codes else dt)


def pa_append_and_decode(out: torch.Tensor, q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                         k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """One decode step in one launch: key/value [S, Hk, d] (one new token per sequence) go
    into the pools at position context_lens[s] - 1, then out = pa_decode over the whole
    context.  E4M3 pools (uint8 / float8_e4m3fn) take k_scale and v_scale."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl, pkey, pval, dt, kv = _append_common(
        out, q, key, value, k_cache, v_cache, block_tables, context_lens)
    st = _lib.lib().pa_append_and_decode(po, pq, pkey, pval, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale),
                                         dt, kv, float(k_scale), float(v_scale), _stream_ptr(q, stream))
    _lib.check("pa_append_and_decode", st)


def pa_append_and_decode_splitk(out: torch.Tensor, q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, scale: float, partition_size: int,
                                workspace: torch.Tensor, max_num_partitions: Optional[int] = None,
                                k_scale: float = 1.0, v_scale: float = 1.0,
                                stream: Optional[torch.cuda.Stream] = None) -> None:
    """pa_append_and_decode with the split-K partitions; follow with pa_splitk_reduce."""
    dev, S, H, d, N, B, Hk, M, (po, pq, pk, pv, pbt), pcl, pkey, pval, dt, kv = _append_common(
        out, q, key, value, k_cache, v_cache, block_tables, context_lens)
    P = max_num_partitions or max_num_partitions_for(M, B, partition_size)
    ws = _need(workspace, "workspace", workspace.dtype, dev)
    st = _lib.lib().pa_append_and_decode_splitk(
        po, pq, pkey, pval, pk, pv, pbt, M, pcl, S, H, Hk, d, B, N, float(scale), dt, kv, float(k_scale),
        float(v_scale), int(partition_size), int(P), ws, workspace.numel() * workspace.element_size(),
        _stream_ptr(q, stream))
    _lib.check("pa_append_and_decode_splitk", st)


def pa_prefill(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               block_tables: torch.Tensor, context_lens: torch.Tensor, query_start_loc: torch.Tensor,
               max_query_len: int, scale: float, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Paged prefill: q/out [rows, H, d]; sequence s owns rows query_start_loc[s] ..
    query_start_loc[s+1] (its last positions) and each row attends causally."""
    dev = _cuda_device(q)
    R, H, d = q.shape
    N, B, Hk, d2 = k_cache.shape
    S = int(context_lens.shape[0])
    if d2 != d or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("q/out [rows, H, d] must match the pools [N, B, Hk, d]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start_loc.shape != (S + 1,):
        raise ValueError("block_tables must be [S, M] and query_start_loc [S + 1]")
    dt = q.dtype
    st = _lib.lib().pa_prefill(
        _need(out, "out", dt, dev), _need(q, "q", dt, dev), _need(k_cache, "k_cache", dt, dev),
        _need(v_cache, "v_cache", dt, dev), _need(block_tables, "block_tables", torch.int32, dev),
        int(block_tables.shape[1]), _need(context_lens, "context_lens", torch.int32, dev),
        _need(query_start_loc, "query_start_loc", torch.int32, dev), S, R, int(max_query_len), H, Hk, d, B, N,
        float(scale), _dtype_code(q), _stream_ptr(q, stream))
    _lib.check("pa_prefill", st)


def pa_selftest_wait(device=None, limit_us: int = 20000,
                     stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Run the library's bounded-wait self-test on `device` (default: the current CUDA
    device) and return {"gave_up", "completed", "waited_us"} once it has finished."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.type != "cuda":
        raise ValueError("the self-test runs on a CUDA device")
    res = torch.full((3,), -1, dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    st = _lib.lib().pa_selftest_wait(int(res.data_ptr()), int(limit_us), int(s.cuda_stream))
    _lib.check("pa_selftest_wait", st)
    s.synchronize()
    r = res.cpu().tolist()
    return {"gave_up": r[0] == 1, "completed": r[1] == 1, "waited_us": r[2]}


def pa_status_string(status: int) -> str:
    return _lib.status_name(status)


def pa_last_error() -> str:
    return _lib.last_error()


def alloc_splitk_workspace(num_seqs: int, num_heads: int, head_dim: int, max_num_partitions: int,
                           device) -> torch.Tensor:
    """A float32 device buffer of the size pa_splitk_workspace_bytes states."""
    nbytes = pa_splitk_workspace_bytes(num_seqs, num_heads, head_dim, max_num_partitions)
    return torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=device)
