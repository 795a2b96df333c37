"""The seeded input generators produce the stated shapes, sharing and poison."""
from __future__ import annotations

import numpy as np
import pytest

from paged_kv_cache_173_gb300 import workloads


def _check_common(b: workloads.PagedBatch):
    S, B = b.num_seqs, b.block_size
    assert b.q.shape == (S, b.num_heads, b.head_dim) and b.q.dtype == np.float16
    assert b.k_cache.shape == (b.num_blocks, B, b.num_kv_heads, b.head_dim)
    assert b.v_cache.shape == b.k_cache.shape
    assert b.block_tables.shape == (S, b.max_blocks_per_seq) and b.block_tables.dtype == np.int32
    assert b.context_lens.dtype == np.int32
    assert b.slot_mapping.dtype == np.int64
    for s in range(S):
        c = int(b.context_lens[s])
        nb = (c + B - 1) // B
        assert 1 <= c <= b.max_blocks_per_seq * B
        assert np.all(b.block_tables[s, :nb] >= 0) and np.all(b.block_tables[s, :nb] < b.num_blocks)
        assert np.all(b.block_tables[s, nb:] == -1)
        assert nb * B - c <= B - 1  # waste bound of the last block
        pos = c - 1
        assert b.slot_mapping[s] == b.block_tables[s, pos // B] * B + pos % B


def test_tiny_batch_matches_its_recipe():
    b = workloads.tiny()
    _check_common(b)
    assert list(b.context_lens) == [1, 15, 16, 37]
    assert b.num_blocks == 16 and b.block_size == 16 and b.head_dim == 64
    perm = np.random.default_rng(0).permutation(16)
    used = [b.block_tables[0, 0], b.block_tables[1, 0], b.block_tables[2, 0], *b.block_tables[3, :3]]
    assert used == list(perm[:6])
    assert b.scale == np.float32(0.125)


def test_llama3_8b_batch():
    b = workloads.llama3_8b()
    _check_common(b)
    assert b.num_seqs == 64 and b.num_heads == 32 and b.num_kv_heads == 8
    assert b.context_lens.min() >= 128 and b.context_lens.max() <= 2048
    needed = int(sum((int(c) + 15) // 16 for c in b.context_lens))
    assert b.num_blocks == int(np.ceil(1.25 * needed))
    used = b.block_tables[b.block_tables >= 0]
    assert len(np.unique(used)) == used.size  # no sharing
    assert b.max_blocks_per_seq == 128


def test_shared_prefix_batch_shares_prompt_blocks():
    b = workloads.shared_prefix(num_prompts=3, samples=4, prompt_len=64, max_suffix=40)
    _check_common(b)
    for p in range(3):
        rows = b.block_tables[p * 4:(p + 1) * 4, :4]
        assert np.all(rows == rows[0])
    other = b.block_tables[:, 4:]
    other = other[other >= 0]
    assert len(np.unique(other)) == other.size
    assert np.all(b.context_lens >= 65) and np.all(b.context_lens <= 64 + 40 + 1)
    assert workloads.unique_kv_bytes(b) < workloads.algorithmic_kv_bytes(b)


def test_poison_marks_exactly_the_unread_slots():
    b = workloads.llama3_8b(num_seqs=6, min_ctx=17, max_ctx=90)
    B = b.block_size
    valid = np.zeros((b.num_blocks, B), bool)
    for s in range(b.num_seqs):
        for t in range(int(b.context_lens[s]) - 1):  # the new token's slot stays poisoned
            valid[b.block_tables[s, t // B], t % B] = True
    nan = np.isnan(b.k_cache.astype(np.float32)).all(axis=(2, 3))
    assert np.array_equal(nan, ~valid)
    assert np.array_equal(np.isnan(b.v_cache.astype(np.float32)).all(axis=(2, 3)), ~valid)
    clean = workloads.llama3_8b(num_seqs=6, min_ctx=17, max_ctx=90, poison=False)
    assert np.isfinite(clean.k_cache.astype(np.float32)).all()


def test_generators_are_deterministic():
    a = workloads.llama2_70b(num_seqs=2, ctx=300, block_size=32)
    b = workloads.llama2_70b(num_seqs=2, ctx=300, block_size=32)
    for f in ("q", "k_cache", "v_cache", "block_tables", "key", "value", "slot_mapping"):
        assert np.array_equal(getattr(a, f).view(np.uint8), getattr(b, f).view(np.uint8))


@pytest.mark.parametrize("bs", [16, 32])
def test_llama2_70b_batch(bs):
    b = workloads.llama2_70b(num_seqs=2, ctx=1000, block_size=bs)
    _check_common(b)
    assert b.group_size == 8 and b.block_size == bs


def test_prefill_batch_layout_and_poison():
    b = workloads.build_prefill_batch(name="pf", seed=3, context_lens=[20, 50, 16], query_lens=[20, 7, 1],
                                      num_heads=4, num_kv_heads=2, head_dim=64, block_size=16)
    assert list(b.query_start_loc) == [0, 20, 27, 28]
    assert b.q.shape == (28, 4, 64) and b.key.shape == (28, 2, 64)
    # each new token's slot is its position in its sequence's table, and holds NaN before the write
    for s, (c, n) in enumerate([(20, 20), (50, 7), (16, 1)]):
        for i in range(n):
            pos = c - n + i
            slot = b.slot_mapping[b.query_start_loc[s] + i]
            assert slot == b.block_tables[s, pos // 16] * 16 + pos % 16
            assert np.isnan(b.k_cache.reshape(-1, 2, 64)[slot]).all()
        for pos in range(c - n):  # the cached part is finite
            blk = b.block_tables[s, pos // 16]
            assert np.isfinite(b.k_cache[blk, pos % 16]).all()
