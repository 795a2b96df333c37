"""Seeded synthetic batches for paged decode attention.

This module only draws inputs: random values, context lengths, block tables
built from a shuffled free list, and the slot each new token is written to.
It holds none of the attention arithmetic, and both the CUDA path and the
CPU oracle consume what it returns.

Recipe (every batch):

* ``rng = numpy.random.default_rng(seed)`` (PCG64); draws happen in a fixed
  order: context lengths, the physical-id permutation, ``q``, the K pool, the
  V pool, the new tokens' K and V.
* values are standard normal drawn as float32 and rounded (to nearest even)
  to float16, or to bfloat16 with ``dtype="bf16"``; bfloat16 arrays are kept
  as uint16 bit patterns, since numpy has no bfloat16 type.
* the KV pools have the layout ``[num_blocks, block_size, num_kv_heads,
  head_dim]``, one pool for K and one for V.
* a sequence of ``ctx`` tokens owns ``ceil(ctx / block_size)`` blocks.  The
  block ids are taken in order from a random permutation of the pool, so the
  table is a scatter of physical blocks ("PagedAttention: when the KV cache
  meets OS paging", section 3.1, step 2: logical blocks map to arbitrary
  physical blocks).  The pool holds 1.25x the blocks the batch needs, rounded
  up, unless a batch states otherwise.
* ``context_lens[s]`` counts the token being decoded: that token sits at
  position ``ctx - 1`` and is written by ``reshape_and_cache`` through
  ``slot_mapping`` before decode ("Efficient Memory Management for LLM
  Serving with PagedAttention — in-depth reading", section 3.4, steps 1 and
  3: the new KV goes into its slot, then attention reads every valid slot).
* ``poison=True`` fills every slot that decode must not read (free blocks,
  the tail of each last block, the new token's slot before the write) with
  float16 NaN, and unused block-table entries with -1, so that a read past
  the context shows up as NaN.  ``poison=False`` leaves the standard-normal
  draws there (used for timing).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

FP16_NAN_BITS = np.uint16(0x7E00)
BF16_NAN_BITS = np.uint16(0x7FC0)
E4M3_NAN_BITS = np.uint8(0x7F)
FP8_SCALE = 2.0 ** -5  # FP8 pools hold N(0,1) / FP8_SCALE as E4M3 codes (an exact power of two)


def f32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of float32 values, through torch's float8 conversion."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bfloat16 (ties to even) and
    return the 16-bit patterns: the upper half of the float32 after adding
    0x7FFF plus the lowest kept bit."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


@dataclasses.dataclass
class PagedBatch:
    """One decode step's inputs for one layer (all arrays are numpy)."""

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float  # a float32 value, stored as a Python float
    q: np.ndarray  # [S, H, d] float16
    k_cache: np.ndarray  # [N, B, Hk, d] float16, state before the write
    v_cache: np.ndarray  # [N, B, Hk, d] float16, state before the write
    block_tables: np.ndarray  # [S, M] int32, -1 where unused
    context_lens: np.ndarray  # [S] int32, includes the new token
    key: np.ndarray  # [T, Hk, d] float16, new tokens
    value: np.ndarray  # [T, Hk, d] float16, new tokens
    slot_mapping: np.ndarray  # [T] int64, flat slot id, -1 = skip
    partition_size: int  # split-K partition length (tokens) for this workload
    unique_blocks: int  # distinct physical blocks referenced by the tables
    dtype: str = "fp16"  # "fp16": float16 arrays; "bf16": uint16 bfloat16 bit patterns
    kv_dtype: str = ""  # "": the caches have `dtype`; "fp8": uint8 E4M3 codes scaled by k/v_scale
    seqs_per_group: int = 1  # sequences [j*g, (j+1)*g) form group j ...
    prefix_lens: Optional[np.ndarray] = None  # ... sharing their first prefix_lens[j] tokens (int32)
    k_scale: float = 1.0
    v_scale: float = 1.0
    # prefill batches: q is [T, H, d], rows query_start_loc[s] .. query_start_loc[s+1]
    # belong to sequence s (its last qlen positions); None for decode batches
    query_start_loc: Optional[np.ndarray] = None

    @property
    def group_size(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def num_tokens(self) -> int:
        return int(self.key.shape[0])


def _normal_f16(rng: np.random.Generator, shape, chunk_elems: int = 1 << 26, dtype: str = "fp16") -> np.ndarray:
    """Standard normal float32 draws rounded to float16 (or bfloat16 bit
    patterns), drawn in chunks."""
    out = np.empty(int(np.prod(shape)), dtype=np.float16 if dtype == "fp16" else np.uint16)
    pos = 0
    total = out.size
    while pos < total:
        n = min(chunk_elems, total - pos)
        x = rng.standard_normal(n, dtype=np.float32)
        out[pos:pos + n] = x.astype(np.float16) if dtype == "fp16" else f32_to_bf16_bits(x)
        pos += n
    return out.reshape(shape)


def build_batch(
    *,
    name: str,
    seed: int,
    context_lens: Sequence[int],
    num_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    max_blocks_per_seq: Optional[int] = None,
    pool_factor: float = 1.25,
    num_blocks: Optional[int] = None,
    share_groups: Optional[Sequence[Sequence[int]]] = None,
    shared_prefix_len: int = 0,
    new_token: bool = True,
    poison: bool = True,
    partition_size: int = 512,
    rng: Optional[np.random.Generator] = None,
    q_scale: float = 1.0,
    dtype: str = "fp16",
    kv_dtype: str = "",
    draw_pools: bool = True,
) -> PagedBatch:
    """Build one batch.

    ``draw_pools=False`` leaves the K and V pools undrawn (allocated, not
    filled, and not taken from ``rng``, so the new tokens' draws move up):
    for timing runs that fill the pools on the device themselves.  It needs
    ``poison=False``.

    ``share_groups``: lists of sequence indices whose first
    ``shared_prefix_len`` tokens (a whole number of blocks) live in the same
    physical blocks (parallel sampling from one prompt).  The first sequence of
    a group draws the prefix blocks; the others point at them.  When the groups
    are consecutive runs of one size g, the batch records g and the shared
    length per group (``seqs_per_group``, ``prefix_lens``).
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = int(ctx.size)
    B = int(block_size)
    Hk = int(num_kv_heads)
    H = int(num_heads)
    d = int(head_dim)
    assert H % Hk == 0
    assert shared_prefix_len % B == 0
    nblk = [(int(c) + B - 1) // B for c in ctx]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(nblk) if nblk else 1)
    M = int(max_blocks_per_seq)
    assert all(n <= M for n in nblk)

    # Which sequence owns the prefix blocks of each sharing group.
    prefix_owner = list(range(S))
    if share_groups:
        for grp in share_groups:
            for s in grp:
                prefix_owner[s] = grp[0]
                assert ctx[s] > shared_prefix_len, "a sharing sequence must extend past the prefix"
    npre = shared_prefix_len // B

    needed = 0
    for s in range(S):
        if share_groups and prefix_owner[s] != s:
            needed += nblk[s] - npre
        else:
            needed += nblk[s]
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * needed)))
    N = int(num_blocks)
    assert N >= needed

    perm = rng.permutation(N).astype(np.int32)
    tables = np.full((S, M), -1, dtype=np.int32)
    nxt = 0
    for s in range(S):
        if share_groups and prefix_owner[s] != s:
            tables[s, :npre] = tables[prefix_owner[s], :npre]
            cnt = nblk[s] - npre
            tables[s, npre:nblk[s]] = perm[nxt:nxt + cnt]
            nxt += cnt
        else:
            tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
            nxt += nblk[s]
    unique_blocks = nxt

    assert dtype in ("fp16", "bf16")
    assert q_scale == 1.0 or dtype == "fp16"
    q = _normal_f16(rng, (S, H, d), dtype=dtype)
    if q_scale != 1.0:
        q = (q.astype(np.float32) * np.float32(q_scale)).astype(np.float16)
    if not draw_pools:
        assert not poison, "undrawn pools cannot be poisoned"
        k_cache = np.empty((N, B, Hk, d), dtype=np.uint8 if kv_dtype == "fp8" else
                           (np.float16 if dtype == "fp16" else np.uint16))
        v_cache = np.empty_like(k_cache)
    elif kv_dtype == "fp8":
        assert dtype == "fp16", "FP8 caches take float16 queries and new tokens"
        k_cache = f32_to_e4m3_codes(_normal_f16(rng, (N, B, Hk, d)).astype(np.float32) / np.float32(FP8_SCALE))
        v_cache = f32_to_e4m3_codes(_normal_f16(rng, (N, B, Hk, d)).astype(np.float32) / np.float32(FP8_SCALE))
    else:
        assert kv_dtype == ""
        k_cache = _normal_f16(rng, (N, B, Hk, d), dtype=dtype)
        v_cache = _normal_f16(rng, (N, B, Hk, d), dtype=dtype)

    T = S if new_token else 0
    key = _normal_f16(rng, (T, Hk, d), dtype=dtype)
    value = _normal_f16(rng, (T, Hk, d), dtype=dtype)
    slot_mapping = np.full((T,), -1, dtype=np.int64)
    if new_token:
        for s in range(S):
            pos = int(ctx[s]) - 1
            slot_mapping[s] = int(tables[s, pos // B]) * B + pos % B

    if poison:
        valid = np.zeros((N, B), dtype=bool)
        for s in range(S):
            for i in range(nblk[s]):
                lo = i * B
                hi = min(int(ctx[s]), lo + B)
                valid[tables[s, i], : hi - lo] = True
        if new_token:
            for s in range(S):
                sl = int(slot_mapping[s])
                valid[sl // B, sl % B] = False
        if kv_dtype == "fp8":
            kb, vb, nan = k_cache, v_cache, E4M3_NAN_BITS
        else:
            kb = k_cache.view(np.uint16)
            vb = v_cache.view(np.uint16)
            nan = FP16_NAN_BITS if dtype == "fp16" else BF16_NAN_BITS
        kb[~valid] = nan
        vb[~valid] = nan

    seqs_per_group, prefix_lens = 1, None
    if share_groups:
        g = len(share_groups[0])
        if all(list(grp) == list(range(i * g, i * g + len(grp))) for i, grp in enumerate(share_groups)) and \
                all(len(grp) == g for grp in share_groups[:-1]) and len(share_groups) == -(-S // g):
            seqs_per_group = g
            prefix_lens = np.full(len(share_groups), shared_prefix_len, dtype=np.int32)

    return PagedBatch(
        name=name, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_dim=d, block_size=B,
        num_blocks=N, max_blocks_per_seq=M, scale=float(np.float32(1.0 / math.sqrt(d))),
        q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
        context_lens=ctx.astype(np.int32), key=key, value=value, slot_mapping=slot_mapping,
        partition_size=int(partition_size), unique_blocks=int(unique_blocks), dtype=dtype,
        kv_dtype=kv_dtype, k_scale=FP8_SCALE if kv_dtype == "fp8" else 1.0,
        v_scale=FP8_SCALE if kv_dtype == "fp8" else 1.0, seqs_per_group=seqs_per_group, prefix_lens=prefix_lens,
    )


def build_prefill_batch(
    *,
    name: str,
    seed: int,
    context_lens: Sequence[int],
    query_lens: Sequence[int],
    num_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    max_blocks_per_seq: Optional[int] = None,
    pool_factor: float = 1.25,
    poison: bool = True,
    rng: Optional[np.random.Generator] = None,
    dtype: str = "fp16",
    kv_dtype: str = "",
) -> PagedBatch:
    """One prefill step: sequence s has context_lens[s] tokens, of which the
    last query_lens[s] are new (a whole prompt when they are equal, a chunk of
    one otherwise).  Draw order: a permutation of the physical ids, q [T, H, d]
    (T = sum of query_lens), the K pool, the V pool, the new tokens' K and V.
    The new tokens' slots (and every slot past a context) hold NaN until the
    cache write fills them."""
    rng = rng or np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    S = int(ctx.size)
    assert ql.size == S and (ql >= 0).all() and (ql <= ctx).all()
    B, Hk, H, d = int(block_size), int(num_kv_heads), int(num_heads), int(head_dim)
    assert H % Hk == 0 and dtype in ("fp16", "bf16") and kv_dtype in ("", "fp8")
    assert kv_dtype == "" or dtype == "fp16"
    nblk = [(int(c) + B - 1) // B for c in ctx]
    M = int(max_blocks_per_seq or max(1, max(nblk)))
    assert all(n <= M for n in nblk)
    need = sum(nblk)
    N = max(need + 1, int(math.ceil(need * pool_factor)))
    perm = rng.permutation(N).astype(np.int32)
    tables = np.full((S, M), -1, dtype=np.int32)
    nxt = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
        nxt += nblk[s]
    T = int(ql.sum())
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(ql)
    q = _normal_f16(rng, (T, H, d), dtype=dtype)
    if kv_dtype == "fp8":
        k_cache = f32_to_e4m3_codes(_normal_f16(rng, (N, B, Hk, d)).astype(np.float32) / np.float32(FP8_SCALE))
        v_cache = f32_to_e4m3_codes(_normal_f16(rng, (N, B, Hk, d)).astype(np.float32) / np.float32(FP8_SCALE))
    else:
        k_cache = _normal_f16(rng, (N, B, Hk, d), dtype=dtype)
        v_cache = _normal_f16(rng, (N, B, Hk, d), dtype=dtype)
    key = _normal_f16(rng, (T, Hk, d), dtype=dtype)
    value = _normal_f16(rng, (T, Hk, d), dtype=dtype)
    slot_mapping = np.empty(T, dtype=np.int64)
    for s in range(S):
        for i in range(int(ql[s])):
            pos = int(ctx[s] - ql[s]) + i
            slot_mapping[qsl[s] + i] = int(tables[s, pos // B]) * B + pos % B
    if poison:
        valid = np.zeros((N, B), dtype=bool)
        for s in range(S):
            for pos in range(int(ctx[s] - ql[s])):  # the cached part
                valid[tables[s, pos // B], pos % B] = True
        if kv_dtype == "fp8":
            kb, vb, nan = k_cache, v_cache, E4M3_NAN_BITS
        else:
            kb, vb = k_cache.view(np.uint16), v_cache.view(np.uint16)
            nan = FP16_NAN_BITS if dtype == "fp16" else BF16_NAN_BITS
        kb[~valid] = nan
        vb[~valid] = nan
    return PagedBatch(
        name=name, num_seqs=S, num_heads=H, num_kv_heads=Hk, head_dim=d, block_size=B, num_blocks=N,
        max_blocks_per_seq=M, scale=float(np.float32(1.0 / math.sqrt(d))), q=q, k_cache=k_cache,
        v_cache=v_cache, block_tables=tables, context_lens=ctx.astype(np.int32), key=key, value=value,
        slot_mapping=slot_mapping, partition_size=0, unique_blocks=int(need), dtype=dtype, kv_dtype=kv_dtype,
        k_scale=FP8_SCALE if kv_dtype == "fp8" else 1.0, v_scale=FP8_SCALE if kv_dtype == "fp8" else 1.0,
        query_start_loc=qsl)


def prefill_flops(batch: PagedBatch) -> int:
    """Multiply-adds of QK^T and PV, times 2: each query row at position p
    scores p + 1 keys and sums p + 1 values, per head, over d dims."""
    ctx = batch.context_lens.astype(np.int64)
    ql = np.diff(batch.query_start_loc.astype(np.int64))
    keys = 0
    for c, n in zip(ctx, ql):  # rows at positions c-n .. c-1 see c-n+1 .. c keys
        keys += n * (c - n) + n * (n + 1) // 2
    return int(4 * batch.head_dim * batch.num_heads * keys)


# ---------------------------------------------------------------------------
# The five workloads.  Sizes in the names are those of the full workloads; the
# ``num_seqs`` / ``ctx`` overrides give the scaled-down parity cases.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, poison: bool = True) -> PagedBatch:
    """4 sequences with contexts {1, 15, 16, 37}: one token, a partial block,
    an exactly full block, and three blocks with 5 valid slots in the last;
    H = Hk = 4, d = 64, B = 16, a pool of 16 blocks; the tables take the first
    six ids of a seeded permutation of 0..15, in order; scale = 1/8."""
    return build_batch(name="tiny", seed=seed, context_lens=[1, 15, 16, 37], num_heads=4,
                       num_kv_heads=4, head_dim=64, block_size=16, num_blocks=16,
                       max_blocks_per_seq=3, poison=poison, partition_size=16)


def llama3_8b(seed: int = 0, num_seqs: int = 64, poison: bool = True,
              min_ctx: int = 128, max_ctx: int = 2048, partition_size: int = 512,
              dtype: str = "fp16", kv_dtype: str = "") -> PagedBatch:
    """Llama-3-8B-shaped decode layer: 32 q heads, 8 KV heads (GQA 4), d = 128,
    B = 16; contexts uniform in [min_ctx, max_ctx]; 1.25x pool, shuffled ids."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(min_ctx, max_ctx + 1, size=num_seqs)
    return build_batch(name="llama3-8b", seed=seed, rng=rng, context_lens=ctx, num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16,
                       max_blocks_per_seq=(max_ctx + 15) // 16, poison=poison,
                       partition_size=partition_size, dtype=dtype, kv_dtype=kv_dtype)


def llama2_70b(seed: int = 0, block_size: int = 16, num_seqs: int = 32, ctx: int = 8192,
               poison: bool = True, partition_size: int = 512, dtype: str = "fp16", kv_dtype: str = "",
               draw_pools: bool = True) -> PagedBatch:
    """Llama-2-70B-shaped GQA decode: 64 q heads, 8 KV heads (GQA 8), d = 128;
    every context ``ctx`` tokens; one new token per sequence at position
    ctx - 1; 1.25x pool, shuffled ids."""
    return build_batch(name=f"llama2-70b-b{block_size}", seed=seed, context_lens=[ctx] * num_seqs,
                       num_heads=64, num_kv_heads=8, head_dim=128, block_size=block_size,
                       poison=poison, partition_size=partition_size, dtype=dtype, kv_dtype=kv_dtype,
                       draw_pools=draw_pools)


def long_context(seed: int = 0, ctxs: Sequence[int] = (32768, 65536, 98304, 131072),
                 poison: bool = True, partition_size: int = 512, dtype: str = "fp16", kv_dtype: str = "",
                 draw_pools: bool = True) -> PagedBatch:
    """Long-context split-K decode: 32 q heads, 8 KV heads, d = 128, B = 16;
    4 sequences of 32K..128K tokens; 512-token partitions."""
    return build_batch(name="long-context", seed=seed, context_lens=list(ctxs), num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, poison=poison,
                       partition_size=partition_size, dtype=dtype, kv_dtype=kv_dtype, draw_pools=draw_pools)


def shared_prefix(seed: int = 0, num_prompts: int = 16, samples: int = 8, prompt_len: int = 1024,
                  max_suffix: int = 512, poison: bool = True, partition_size: int = 512,
                  dtype: str = "fp16", kv_dtype: str = "") -> PagedBatch:
    """Parallel sampling: ``num_prompts`` prompts of ``prompt_len`` tokens, each
    sampled ``samples`` times.  The samples' tables point at the same prompt
    blocks (reference count ``samples``) and then diverge with suffixes
    uniform in [0, max_suffix]; plus one new token per sample, so
    ctx = prompt_len + suffix + 1.  MHA with 40 heads, d = 128, B = 16."""
    rng = np.random.default_rng(seed)
    S = num_prompts * samples
    suffix = rng.integers(0, max_suffix + 1, size=S)
    ctx = prompt_len + suffix + 1
    groups: List[List[int]] = [list(range(p * samples, (p + 1) * samples)) for p in range(num_prompts)]
    M = (prompt_len + max_suffix + 1 + 15) // 16
    return build_batch(name="shared-prefix", seed=seed, rng=rng, context_lens=ctx, num_heads=40,
                       num_kv_heads=40, head_dim=128, block_size=16, max_blocks_per_seq=M,
                       share_groups=groups, shared_prefix_len=prompt_len, poison=poison,
                       partition_size=partition_size, dtype=dtype, kv_dtype=kv_dtype)


WORKLOADS = {
    "tiny": tiny,
    "llama3-8b": llama3_8b,
    "llama2-70b": llama2_70b,
    "long-context": long_context,
    "shared-prefix": shared_prefix,
}


# ---------------------------------------------------------------------------
# Byte accounting for the measurement (what one decode must read at least).
# ---------------------------------------------------------------------------

def kv_elem_bytes(batch: PagedBatch) -> int:
    """Bytes of one cache element: 1 for E4M3 caches, else 2."""
    return 1 if batch.kv_dtype == "fp8" else 2


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K plus V bytes of one token of one layer."""
    return 2 * num_kv_heads * head_dim * elem_bytes


def algorithmic_kv_bytes(batch: PagedBatch, elem_bytes: int = 0) -> int:
    """Sum over sequences of ctx * (K + V bytes per token): the valid slots
    only, counted once per sequence that reads them (logical bytes)."""
    return int(np.sum(batch.context_lens.astype(np.int64))) * kv_bytes_per_token(
        batch.num_kv_heads, batch.head_dim, elem_bytes or kv_elem_bytes(batch))


def unique_kv_bytes(batch: PagedBatch, elem_bytes: int = 0) -> int:
    """Bytes of the distinct valid slots (shared prefix blocks counted once)."""
    seen = set()
    B = batch.block_size
    total_slots = 0
    for s in range(batch.num_seqs):
        c = int(batch.context_lens[s])
        for i in range((c + B - 1) // B):
            blk = int(batch.block_tables[s, i])
            valid = min(B, c - i * B)
            if blk in seen:
                continue
            seen.add(blk)
            total_slots += valid
    return total_slots * kv_bytes_per_token(batch.num_kv_heads, batch.head_dim,
                                            elem_bytes or kv_elem_bytes(batch))
