"""A second, pure-Python/numpy statement of the same oracle, for tiny cases.

TEST INFRASTRUCTURE.  It is written independently of ``pa_oracle.c`` and in a
different style: no gather into contiguous arrays; every score is taken token
by token, each token found through ``locate_kv`` ("Unveiling the NVIDIA
driver stack: GPU page tables and vLLM PagedAttention", section 6).  The
softmax is the two-pass textbook form ("vLLM PagedAttention source
walk-through", section 3.4).  Python loops: use it only on small batches.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def locate_kv(logical_token_idx: int, block_table: Sequence[int], block_size: int) -> Tuple[int, int]:
    logical_block = logical_token_idx // block_size
    offset_in_block = logical_token_idx % block_size
    return int(block_table[logical_block]), int(offset_in_block)


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping):
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    B = kc.shape[1]
    used = set()
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        assert slot not in used, "slots must be distinct"
        used.add(slot)
        kc[slot // B, slot % B] = key[t]
        vc[slot // B, slot % B] = value[t]
    return kc, vc


def decode_bruteforce(q, k_cache, v_cache, block_tables, context_lens, scale) -> np.ndarray:
    q = np.asarray(q)
    S, H, d = q.shape
    B = k_cache.shape[1]
    Hk = k_cache.shape[2]
    G = H // Hk
    out = np.zeros((S, H, d), dtype=np.float64)
    for s in range(S):
        n = int(context_lens[s])
        table = [int(x) for x in block_tables[s]]
        for h in range(H):
            kvh = h // G
            qv = q[s, h].astype(np.float64)
            scores: List[float] = []
            for t in range(n):
                blk, off = locate_kv(t, table, B)
                kt = k_cache[blk, off, kvh].astype(np.float64)
                scores.append(float(scale) * float(np.dot(qv, kt)))
            if n == 0:
                continue
            m = max(scores)
            w = [math.exp(x - m) for x in scores]
            z = sum(w)
            acc = np.zeros(d, dtype=np.float64)
            for t in range(n):
                blk, off = locate_kv(t, table, B)
                acc += (w[t] / z) * v_cache[blk, off, kvh].astype(np.float64)
            out[s, h] = acc
    return out


def copy_blocks(k_cache, v_cache, block_mapping):
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for src, dst in np.asarray(block_mapping).reshape(-1, 2).tolist():
        if 0 <= src < kc.shape[0] and 0 <= dst < kc.shape[0] and src != dst:
            kc[dst] = kc[src]
            vc[dst] = vc[src]
    return kc, vc


def prefill_bruteforce(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale) -> np.ndarray:
    """Prefill, row by row: row i of sequence s sits at position
    ctx - qlen + i and is decode attention over positions 0..that position."""
    q = np.asarray(q)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(len(context_lens)):
        r0, r1 = int(query_start_loc[s]), int(query_start_loc[s + 1])
        ctx = int(context_lens[s])
        for i, r in enumerate(range(r0, r1)):
            pos = ctx - (r1 - r0) + i
            out[r] = decode_bruteforce(q[r:r + 1], k_cache, v_cache, np.asarray(block_tables)[s:s + 1],
                                       [pos + 1], scale)[0]
    return out
