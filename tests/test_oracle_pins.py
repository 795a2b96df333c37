"""Pins of the CPU oracle against facts that do not come from the oracle.

Every check here runs on the CPU.  Sources are the pages' worked example and
byte sizes (stored under tests/golden/ with their citations), closed forms,
invariants that paged attention must keep, and an independent library
attention (torch's scaled_dot_product_attention in float64).  The last test
plants mistakes in a copy of the oracle and shows that the pins catch them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import c_oracle, numpy_oracle
from paged_kv_cache_173_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _written(batch):
    """Pools after the new tokens are written (oracle write path)."""
    return c_oracle.reshape_and_cache(batch.key, batch.value, batch.k_cache, batch.v_cache,
                                      batch.slot_mapping)


def _sdpa_contiguous(q, K, V, scale, group):
    """Library attention of one sequence: q [H, d], K/V [n, Hk, d] (float64)."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, :, None, :]
    kt = torch.from_numpy(np.asarray(K, dtype=np.float64)).permute(1, 0, 2)
    vt = torch.from_numpy(np.asarray(V, dtype=np.float64)).permute(1, 0, 2)
    kt = kt.repeat_interleave(group, dim=0)[None]
    vt = vt.repeat_interleave(group, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(scale))
    return o[0, :, 0, :].numpy()


# --------------------------------------------------------------------------
# float16 decoding
# --------------------------------------------------------------------------

def test_half_decoding_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([c_oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------
# the pages' worked numbers
# --------------------------------------------------------------------------

def test_locate_kv_worked_example():
    g = _golden("locate_kv_example.json")
    want = (g["expected_physical_block"], g["expected_offset"])
    assert c_oracle.locate_kv(g["logical_token_idx"], g["block_table"], g["block_size"]) == want
    assert numpy_oracle.locate_kv(g["logical_token_idx"], g["block_table"], g["block_size"]) == want


def test_locate_kv_walks_every_slot_once():
    table = [7, 42, 9, 103]
    seen = [c_oracle.locate_kv(t, table, 16) for t in range(64)]
    assert len(set(seen)) == 64
    assert [b for b, _ in seen[::16]] == table
    assert all(off == t % 16 for t, (_, off) in enumerate(seen))


def test_byte_accounting_matches_the_pages():
    g = _golden("kv_byte_sizes.json")
    t = g["per_token_per_layer"]
    per_tok = workloads.kv_bytes_per_token(t["num_kv_heads"], t["head_dim"], t["elem_bytes"])
    assert per_tok == t["bytes_per_token_per_layer"]
    assert per_tok * t["num_layers"] == t["kib_per_token_all_layers"] * 1024
    unit = g["per_request_table"]["unit_bytes"]
    for row in g["per_request_table"]["rows"]:
        req = row["seq_len"] * per_tok * t["num_layers"] / unit
        assert abs(req - row["per_request"]) <= 0.05 * row["per_request"]
        assert abs(8 * req - row["batch8"]) <= 0.05 * row["batch8"]
        assert abs(32 * req - row["batch32"]) <= 0.05 * row["batch32"]
    b = g["per_block"]
    half = b["block_size"] * workloads.kv_bytes_per_token(b["num_kv_heads"], b["head_dim"], b["elem_bytes"]) // 2
    assert half == b["k_bytes"] == b["v_bytes"]
    assert 2 * half == b["kv_bytes"]
    bt = g["block_table_size"]
    entries = bt["seq_len"] // bt["block_size"]
    assert entries == bt["entries"]
    assert entries * bt["entry_bytes"] == bt["bytes_per_request"]
    assert abs(bt["requests"] * entries * bt["entry_bytes"] / 1e6 - bt["mb_100_requests"]) < 0.05
    assert abs(bt["requests"] * 2 * entries * bt["entry_bytes"] / 1e6 - bt["mb_100_requests_block8"]) < 0.1
    w = g["waste_bound"]
    B = w["block_size"]
    wastes = [(-n) % B for n in range(1, 10 * B + 1)]
    assert max(wastes) == w["max_waste_tokens"] == B - 1
    assert abs(np.mean(wastes) - (B - 1) / 2) < 1e-12
    assert abs((B - 1) / 2 - w["mean_waste_tokens"]) <= 0.5
    assert w["mean_waste_tokens"] * per_tok // 1024 == w["mean_waste_kib_at_4kib_per_token"]


def test_algorithmic_bytes_of_the_tiny_batch():
    b = workloads.tiny()
    # 69 valid tokens x 4 KV heads x 64 dims x (K + V) x 2 bytes
    assert workloads.algorithmic_kv_bytes(b) == 69 * 4 * 64 * 2 * 2


# --------------------------------------------------------------------------
# decode against an independent attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("group", [1, 4, 8])
def test_identity_table_equals_library_attention(group):
    rng = np.random.default_rng(11)
    B, Hk, d = 16, 2, 64
    H = Hk * group
    ctx = [1, 15, 16, 17, 40]
    nblk = [(c + B - 1) // B for c in ctx]
    N = sum(nblk)
    tables = np.full((len(ctx), max(nblk)), -1, np.int32)
    start = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = np.arange(start, start + n)
        start += n
    kc = rng.standard_normal((N, B, Hk, d), dtype=np.float32).astype(np.float16)
    vc = rng.standard_normal((N, B, Hk, d), dtype=np.float32).astype(np.float16)
    q = rng.standard_normal((len(ctx), H, d), dtype=np.float32).astype(np.float16)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    got = c_oracle.decode(q, kc, vc, tables, np.array(ctx, np.int32), scale)
    # identity table: a sequence's tokens are a contiguous run of the pool
    flatk = kc.reshape(N * B, Hk, d).astype(np.float64)
    flatv = vc.reshape(N * B, Hk, d).astype(np.float64)
    start = 0
    for s, c in enumerate(ctx):
        ref = _sdpa_contiguous(q[s], flatk[start * B:start * B + c], flatv[start * B:start * B + c],
                               scale, group)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)
        start += nblk[s]


def test_scattered_table_equals_library_attention_on_tiny_batch():
    b = workloads.tiny()
    kc, vc = _written(b)
    got = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    for s in range(b.num_seqs):
        c = int(b.context_lens[s])
        rows_k = []
        rows_v = []
        for t in range(c):
            blk = b.block_tables[s, t // b.block_size]
            rows_k.append(kc[blk, t % b.block_size])
            rows_v.append(vc[blk, t % b.block_size])
        ref = _sdpa_contiguous(b.q[s], np.stack(rows_k).astype(np.float64),
                               np.stack(rows_v).astype(np.float64), b.scale, b.group_size)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)


def test_c_oracle_equals_bruteforce_on_tiny_batch():
    b = workloads.tiny()
    kc, vc = _written(b)
    a = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    r = numpy_oracle.decode_bruteforce(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    assert np.isfinite(a).all()
    np.testing.assert_allclose(a, r, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def _single_seq(K, V, q, B=16, scale=1.0, perm_seed=None):
    """Place one sequence's [n, Hk, d] K/V into a scattered pool."""
    n, Hk, d = K.shape
    nb = (n + B - 1) // B
    N = nb + 3
    rng = np.random.default_rng(perm_seed if perm_seed is not None else 5)
    ids = rng.permutation(N)[:nb].astype(np.int32)
    kc = np.full((N, B, Hk, d), np.float16(np.nan), np.float16)
    vc = np.full((N, B, Hk, d), np.float16(np.nan), np.float16)
    for t in range(n):
        kc[ids[t // B], t % B] = K[t]
        vc[ids[t // B], t % B] = V[t]
    return dict(q=q[None], k_cache=kc, v_cache=vc, block_tables=ids[None],
                context_lens=np.array([n], np.int32), scale=scale)


def test_single_token_returns_its_value_exactly():
    b = workloads.tiny()
    kc, vc = _written(b)
    out = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    s = 0
    assert b.context_lens[s] == 1
    blk = b.block_tables[s, 0]
    for h in range(b.num_heads):
        np.testing.assert_array_equal(out[s, h], vc[blk, 0, h // b.group_size].astype(np.float64))


def test_two_tokens_with_a_log3_score_gap_weigh_one_quarter_three_quarters():
    d = 64
    K = np.zeros((2, 1, d), np.float16)
    K[1, 0, 0] = 1.0
    V = np.zeros((2, 1, d), np.float16)
    V[0, 0, 1] = 1.0
    V[1, 0, 2] = 1.0
    q = np.zeros((1, d), np.float16)
    q[0, 0] = 1.0
    scale = float(np.float32(math.log(3.0)))  # score gap ln 3 -> weights 1:3
    case = _single_seq(K, V, q, scale=scale)
    out = c_oracle.decode(**case)[0, 0]
    assert abs(out[1] - 0.25) < 1e-7 and abs(out[2] - 0.75) < 1e-7
    assert np.all(out[3:] == 0) and out[0] == 0
    # the scale multiplies the score: with scale 0 both tokens weigh one half
    case["scale"] = 0.0
    out0 = c_oracle.decode(**case)[0, 0]
    assert out0[1] == 0.5 and out0[2] == 0.5


def test_query_heads_read_consecutive_kv_head_groups():
    rng = np.random.default_rng(3)
    Hk, G, d, n = 3, 4, 64, 37
    K = rng.standard_normal((n, Hk, d), dtype=np.float32).astype(np.float16)
    V = np.empty((n, Hk, d), np.float16)
    for kvh in range(Hk):
        V[:, kvh, :] = kvh + 1  # each KV head's values are the constant kvh + 1
    q = rng.standard_normal((Hk * G, d), dtype=np.float32).astype(np.float16)
    out = c_oracle.decode(**_single_seq(K, V, q, scale=0.125))[0]
    for h in range(Hk * G):
        np.testing.assert_allclose(out[h], h // G + 1, rtol=0, atol=1e-13)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 33, 48])
def test_equal_keys_give_the_mean_of_the_values(n):
    rng = np.random.default_rng(n)
    d = 64
    krow = rng.standard_normal(d, dtype=np.float32).astype(np.float16)
    K = np.broadcast_to(krow, (n, 1, d)).copy()
    V = rng.standard_normal((n, 1, d), dtype=np.float32).astype(np.float16)
    q = rng.standard_normal((1, d), dtype=np.float32).astype(np.float16)
    out = c_oracle.decode(**_single_seq(K, V, q, scale=0.125))[0, 0]
    np.testing.assert_allclose(out, V[:, 0].astype(np.float64).mean(axis=0), rtol=0, atol=1e-13)


def test_a_dominant_score_selects_its_value():
    rng = np.random.default_rng(9)
    n, d, j = 40, 64, 23
    K = rng.standard_normal((n, 1, d), dtype=np.float32).astype(np.float16) * np.float16(0.01)
    q = np.ones((1, d), np.float16)
    K[j, 0, :] = 4.0  # score of token j exceeds the others by > 250 logits at scale 1
    V = rng.standard_normal((n, 1, d), dtype=np.float32).astype(np.float16)
    out = c_oracle.decode(**_single_seq(K, V, q, scale=1.0))[0, 0]
    np.testing.assert_allclose(out, V[j, 0].astype(np.float64), rtol=0, atol=1e-15)


def test_empty_sequence_gives_zeros():
    b = workloads.tiny()
    kc, vc = _written(b)
    cl = b.context_lens.copy()
    cl[2] = 0
    out = c_oracle.decode(b.q, kc, vc, b.block_tables, cl, b.scale)
    assert np.all(out[2] == 0)


# --------------------------------------------------------------------------
# invariants of the paged layout
# --------------------------------------------------------------------------

def test_relabelling_physical_blocks_leaves_the_output_bit_identical():
    b = workloads.llama3_8b(num_seqs=3, max_ctx=300, min_ctx=100)
    kc, vc = _written(b)
    base = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    pi = np.random.default_rng(1).permutation(b.num_blocks)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = np.where(b.block_tables >= 0, pi[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out = c_oracle.decode(b.q, kc2, vc2, bt2, b.context_lens, b.scale)
    assert np.array_equal(out, base)


def test_shared_prefix_equals_duplicated_blocks():
    b = workloads.shared_prefix(num_prompts=2, samples=3, prompt_len=32, max_suffix=20)
    kc, vc = _written(b)
    shared = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    # give every sample its own copy of the prompt blocks
    bt = b.block_tables.copy()
    extra_k, extra_v = [], []
    nxt = b.num_blocks
    for s in range(b.num_seqs):
        for i in range(32 // b.block_size):
            extra_k.append(kc[bt[s, i]])
            extra_v.append(vc[bt[s, i]])
            bt[s, i] = nxt
            nxt += 1
    kc2 = np.concatenate([kc, np.stack(extra_k)])
    vc2 = np.concatenate([vc, np.stack(extra_v)])
    dup = c_oracle.decode(b.q, kc2, vc2, bt, b.context_lens, b.scale)
    assert np.array_equal(shared, dup)
    assert len(np.unique(bt[:, :2])) == bt.shape[0] * 2


def test_poisoned_slots_never_reach_the_output():
    for b in (workloads.tiny(), workloads.llama3_8b(num_seqs=4, max_ctx=200, min_ctx=130)):
        kc, vc = _written(b)
        out = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
        assert np.isfinite(out).all()
        # without the write, the new token's slot still holds NaN and leaks in
        stale = c_oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, b.scale)
        assert np.isnan(stale).all(axis=-1).any()


# --------------------------------------------------------------------------
# reshape_and_cache
# --------------------------------------------------------------------------

def test_reshape_and_cache_c_and_numpy_agree_bitwise():
    b = workloads.llama3_8b(num_seqs=5, max_ctx=100, min_ctx=20)
    ck, cv = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    nk, nv = numpy_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    assert np.array_equal(ck.view(np.uint16), nk.view(np.uint16))
    assert np.array_equal(cv.view(np.uint16), nv.view(np.uint16))


def test_reshape_and_cache_writes_only_the_mapped_slots():
    b = workloads.tiny()
    sm = b.slot_mapping.copy()
    sm[1] = -1  # padding token: skipped
    ck, cv = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, sm)
    B = b.block_size
    changed = np.any(ck.view(np.uint16) != b.k_cache.view(np.uint16), axis=(2, 3))
    expect = np.zeros_like(changed)
    for t, slot in enumerate(sm):
        if slot >= 0:
            expect[slot // B, slot % B] = True
            assert np.array_equal(ck[slot // B, slot % B].view(np.uint16), b.key[t].view(np.uint16))
            assert np.array_equal(cv[slot // B, slot % B].view(np.uint16), b.value[t].view(np.uint16))
    assert np.array_equal(changed, expect)


def test_reshape_and_cache_rejects_duplicate_and_out_of_range_slots():
    b = workloads.tiny()
    dup = b.slot_mapping.copy()
    dup[1] = dup[0]
    with pytest.raises(c_oracle.OracleError):
        c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, dup)
    bad = b.slot_mapping.copy()
    bad[0] = b.num_blocks * b.block_size
    with pytest.raises(c_oracle.OracleError):
        c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, bad)


def test_new_token_lands_at_the_last_context_position():
    b = workloads.llama3_8b(num_seqs=4, max_ctx=100, min_ctx=20)
    kc, vc = _written(b)
    for s in range(b.num_seqs):
        pos = int(b.context_lens[s]) - 1
        blk, off = c_oracle.locate_kv(pos, b.block_tables[s], b.block_size)
        assert np.array_equal(kc[blk, off].view(np.uint16), b.key[s].view(np.uint16))


# --------------------------------------------------------------------------
# planted mistakes: each mutant of the loop-by-token oracle fails a pin
# --------------------------------------------------------------------------

def _run_pins(decode_fn):
    """Return the names of the pins that the given decode function fails."""
    failed = []
    b = workloads.tiny()
    kc, vc = numpy_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    out = decode_fn(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    for s in range(b.num_seqs):
        c = int(b.context_lens[s])
        ks = np.stack([kc[b.block_tables[s, t // 16], t % 16] for t in range(c)]).astype(np.float64)
        vs = np.stack([vc[b.block_tables[s, t // 16], t % 16] for t in range(c)]).astype(np.float64)
        ref = _sdpa_contiguous(b.q[s], ks, vs, b.scale, b.group_size)
        if not (np.isfinite(out[s]).all() and np.allclose(out[s], ref, rtol=0, atol=1e-9)):
            failed.append("library-attention")
            break
    # GQA mapping
    rng = np.random.default_rng(3)
    K = rng.standard_normal((20, 2, 16), dtype=np.float32).astype(np.float16)
    V = np.empty((20, 2, 16), np.float16)
    V[:, 0] = 1
    V[:, 1] = 2
    q = rng.standard_normal((4, 16), dtype=np.float32).astype(np.float16)
    case = _single_seq(K, V, q, scale=0.25)
    o = decode_fn(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                  case["context_lens"], case["scale"])[0]
    if not all(np.allclose(o[h], h // 2 + 1) for h in range(4)):
        failed.append("gqa-mapping")
    return failed


def test_pins_pass_on_the_oracle_itself():
    assert _run_pins(numpy_oracle.decode_bruteforce) == []


@pytest.mark.parametrize("mutant", ["swap_block_and_offset", "drop_scale", "modulo_heads",
                                    "context_off_by_one", "divide_scale"])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    orig_locate = numpy_oracle.locate_kv
    decode = numpy_oracle.decode_bruteforce
    if mutant == "swap_block_and_offset":
        monkeypatch.setattr(numpy_oracle, "locate_kv",
                            lambda t, table, B: (int(table[t % len(table)]), t // len(table) % B))
    elif mutant == "drop_scale":
        def decode(q, kc, vc, bt, cl, scale):
            return numpy_oracle.decode_bruteforce(q, kc, vc, bt, cl, 1.0)
    elif mutant == "divide_scale":
        def decode(q, kc, vc, bt, cl, scale):
            return numpy_oracle.decode_bruteforce(q, kc, vc, bt, cl, 1.0 / scale)
    elif mutant == "context_off_by_one":
        def decode(q, kc, vc, bt, cl, scale):
            return numpy_oracle.decode_bruteforce(q, kc, vc, bt, np.maximum(cl - 1, 1), scale)
    elif mutant == "modulo_heads":
        def decode(q, kc, vc, bt, cl, scale):
            S, H, d = q.shape
            Hk = kc.shape[2]
            G = H // Hk
            # read KV head h % Hk instead of h // G: query head h is moved to
            # slot perm[h], which the correct mapping sends to KV head h % Hk
            perm = [(h % Hk) * G + (h // Hk) for h in range(H)]
            qn = np.empty_like(q)
            qn[:, perm] = q
            out = numpy_oracle.decode_bruteforce(qn, kc, vc, bt, cl, scale)
            return out[:, perm]
    assert orig_locate(37, [7, 42, 9, 103], 16) == (9, 5)
    assert _run_pins(decode) != []


# --------------------------------------------------------------------------
# bfloat16 inputs
# --------------------------------------------------------------------------

def _bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).double().numpy()


def test_bf16_decoding_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = _bf16_to_f64(bits)
    got = np.array([c_oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_generator_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(200_000, dtype=np.float32) * np.float32(3.0)
    x[:4] = [1.00390625, 1.01171875, -2.0078125, 0.0]  # exact ties round to even
    ours = workloads.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_bf16_batch_equals_library_attention():
    b = workloads.build_batch(name="bf16", seed=21, context_lens=[1, 17, 40], num_heads=8, num_kv_heads=2,
                              head_dim=64, block_size=16, dtype="bf16")
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    got = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale, dtype="bf16")
    assert np.isfinite(got).all()
    kf, vf, qf = _bf16_to_f64(kc), _bf16_to_f64(vc), _bf16_to_f64(b.q)
    for s in range(b.num_seqs):
        c = int(b.context_lens[s])
        ks = np.stack([kf[b.block_tables[s, t // 16], t % 16] for t in range(c)])
        vs = np.stack([vf[b.block_tables[s, t // 16], t % 16] for t in range(c)])
        ref = _sdpa_contiguous(qf[s], ks, vs, b.scale, b.group_size)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)
    # ctx = 1: the output is that token's V, exactly
    blk = b.block_tables[0, 0]
    for h in range(b.num_heads):
        assert np.array_equal(got[0, h], vf[blk, 0, h // b.group_size])


# --------------------------------------------------------------------------
# copy-on-write block copy
# --------------------------------------------------------------------------

def _cow_fork(b, kc, vc, s_fork, free_block):
    """Sequence s_fork shares its last, partial block with sequence 0; copy
    that block to free_block and point s_fork's table there."""
    B = b.block_size
    last = (int(b.context_lens[s_fork]) - 1) // B
    bt = b.block_tables.copy()
    src = int(bt[s_fork, last])
    kc2, vc2 = c_oracle.copy_blocks(kc, vc, [[src, free_block]])
    bt[s_fork, last] = free_block
    return kc2, vc2, bt, src


def test_copy_blocks_c_and_numpy_agree_and_skip_invalid_pairs():
    b = workloads.llama3_8b(num_seqs=4, max_ctx=120, min_ctx=40, poison=False)
    pairs = [[3, 7], [5, 5], [2, b.num_blocks + 1], [-1, 9], [11, 1]]
    ck, cv = c_oracle.copy_blocks(b.k_cache, b.v_cache, pairs)
    nk, nv = numpy_oracle.copy_blocks(b.k_cache, b.v_cache, pairs)
    assert np.array_equal(ck.view(np.uint16), nk.view(np.uint16))
    assert np.array_equal(cv.view(np.uint16), nv.view(np.uint16))
    changed = np.any(ck.view(np.uint16) != b.k_cache.view(np.uint16), axis=(1, 2, 3))
    assert set(np.nonzero(changed)[0]) <= {7, 1}
    assert np.array_equal(ck[7].view(np.uint16), b.k_cache[3].view(np.uint16))
    with pytest.raises(c_oracle.OracleError):
        c_oracle.copy_blocks(b.k_cache, b.v_cache, [[1, 2], [2, 3]])  # a destination is also a source


def test_copy_on_write_keeps_the_original_and_forks_the_copy():
    # two sequences share every block (a sample forked from a 37-token prompt)
    rng = np.random.default_rng(4)
    B, Hk, H, d, n = 16, 2, 4, 64, 37
    K = rng.standard_normal((n, Hk, d), dtype=np.float32).astype(np.float16)
    V = rng.standard_normal((n, Hk, d), dtype=np.float32).astype(np.float16)
    q = rng.standard_normal((2, H, d), dtype=np.float32).astype(np.float16)
    N = 8
    ids = np.array([5, 2, 6], np.int32)
    kc = np.full((N, B, Hk, d), np.float16(np.nan), np.float16)
    vc = np.full_like(kc, np.float16(np.nan))
    for t in range(n):
        kc[ids[t // B], t % B] = K[t]
        vc[ids[t // B], t % B] = V[t]
    batch = workloads.PagedBatch(name="cow", num_seqs=2, num_heads=H, num_kv_heads=Hk, head_dim=d, block_size=B,
                                 num_blocks=N, max_blocks_per_seq=3, scale=0.125, q=q, k_cache=kc, v_cache=vc,
                                 block_tables=np.stack([ids, ids]), context_lens=np.array([n, n], np.int32),
                                 key=K[:0], value=V[:0], slot_mapping=np.zeros(0, np.int64),
                                 partition_size=16, unique_blocks=3)
    kc2, vc2, bt, src = _cow_fork(batch, kc, vc, 1, free_block=0)
    # sequence 1 now writes its 38th token into the private copy (slot 5 of block 0)
    newk = rng.standard_normal((1, Hk, d), dtype=np.float32).astype(np.float16)
    newv = rng.standard_normal((1, Hk, d), dtype=np.float32).astype(np.float16)
    kc3, vc3 = c_oracle.reshape_and_cache(newk, newv, kc2, vc2, np.array([0 * B + n % B]))
    cl = np.array([n, n + 1], np.int32)
    out = c_oracle.decode(q, kc3, vc3, bt, cl, 0.125)
    before = c_oracle.decode(q, kc, vc, np.stack([ids, ids]), np.array([n, n], np.int32), 0.125)
    assert np.array_equal(out[0], before[0])           # the original sequence is untouched
    assert np.array_equal(kc3[src].view(np.uint16), kc[src].view(np.uint16))  # and so is its block
    ks = np.concatenate([K, newk]).astype(np.float64)
    vs = np.concatenate([V, newv]).astype(np.float64)
    ref = _sdpa_contiguous(q[1], ks, vs, 0.125, H // Hk)
    np.testing.assert_allclose(out[1], ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# FP8 (E4M3) caches
# --------------------------------------------------------------------------

def test_e4m3_decoding_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([c_oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_quantiser_matches_torch_within_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(40.0),
        rng.standard_normal(5000).astype(np.float32) * np.float32(0.004),   # subnormal range
        np.array([1.0625, 1.1875, -3.25, 0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, -464.0, 447.9],
                 np.float32),                                              # ties and edges
    ])
    x = x[np.abs(x) <= 464.0]
    ours = np.array([c_oracle.quantize_e4m3(float(v), 1.0) for v in x], np.uint8)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_e4m3_quantiser_saturates_and_divides_by_the_scale():
    assert c_oracle.quantize_e4m3(1000.0, 1.0) == 0x7E
    assert c_oracle.quantize_e4m3(-1e30, 1.0) == 0xFE
    assert c_oracle.quantize_e4m3(float("inf"), 1.0) == 0x7E
    assert c_oracle.quantize_e4m3(float("nan"), 1.0) == 0x7F
    # x / scale: 1.5 / 0.25 = 6 exactly
    assert c_oracle.e4m3_to_double(c_oracle.quantize_e4m3(1.5, 0.25)) == 6.0
    # relative error of a normal value is at most half a 3-bit ulp, 2^-4
    rng = np.random.default_rng(8)
    for v in rng.uniform(0.02, 400.0, 2000):
        back = c_oracle.e4m3_to_double(c_oracle.quantize_e4m3(float(v), 1.0))
        assert abs(back - np.float32(v)) <= 2.0 ** -4 * abs(np.float32(v))


def test_fp8_cache_write_and_decode_equal_library_attention_on_dequantised_values():
    b = workloads.build_batch(name="fp8", seed=31, context_lens=[1, 20, 45], num_heads=8, num_kv_heads=2,
                              head_dim=128, block_size=16, kv_dtype="fp8")
    kc, vc = c_oracle.reshape_and_cache_fp8(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping,
                                            b.k_scale, b.v_scale)
    # the new token's row holds the quantised key
    s, pos = 1, 19
    blk = b.block_tables[s, pos // 16]
    want = [c_oracle.quantize_e4m3(float(x), b.k_scale) for x in b.key[s].reshape(-1)]
    assert np.array_equal(kc[blk, pos % 16].reshape(-1), np.array(want, np.uint8))
    got = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale, k_scale=b.k_scale,
                          v_scale=b.v_scale)
    assert np.isfinite(got).all()
    deq = np.vectorize(c_oracle.e4m3_to_double)
    for s in range(b.num_seqs):
        c = int(b.context_lens[s])
        ks = np.stack([deq(kc[b.block_tables[s, t // 16], t % 16]) for t in range(c)]) * b.k_scale
        vs = np.stack([deq(vc[b.block_tables[s, t // 16], t % 16]) for t in range(c)]) * b.v_scale
        ref = _sdpa_contiguous(b.q[s], ks, vs, b.scale, b.group_size)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_cache_write_matches_torch_division_and_conversion_on_every_written_row(dtype):
    # every written row: the code of the float32 quotient x / scale (IEEE division, as
    # torch divides a float32 tensor by a float32 scalar), by torch's float8 conversion;
    # the new tokens are drawn as bfloat16 (or float16) and scaled so that every quotient
    # stays inside the E4M3 range, where torch's conversion rounds and does not saturate
    b = workloads.build_batch(name="fp8w", seed=33, context_lens=[1, 17, 40, 64, 300], num_heads=8,
                              num_kv_heads=4, head_dim=128, block_size=16, kv_dtype="fp8")
    rng = np.random.default_rng(34)
    shape = b.key.shape
    if dtype == "bf16":
        key = workloads.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(3.0))
        value = workloads.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(3.0))
        as_f32 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float()  # noqa: E731
    else:
        key = (rng.standard_normal(shape, dtype=np.float32) * np.float32(3.0)).astype(np.float16)
        value = (rng.standard_normal(shape, dtype=np.float32) * np.float32(3.0)).astype(np.float16)
        as_f32 = lambda a: torch.from_numpy(a).float()  # noqa: E731
    ks, vs = float(np.float32(0.0371)), float(np.float32(0.123))
    kc, vc = c_oracle.reshape_and_cache_fp8(key, value, b.k_cache, b.v_cache, b.slot_mapping, ks, vs, dtype=dtype)
    for x, sc, pool, old in ((key, ks, kc, b.k_cache), (value, vs, vc, b.v_cache)):
        q = as_f32(x) / torch.tensor(sc, dtype=torch.float32)
        assert float(q.abs().max()) < 448.0
        want = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        written = np.zeros(pool.shape[:2], dtype=bool)
        for t, slot in enumerate(b.slot_mapping):
            blk, off = divmod(int(slot), b.block_size)
            assert np.array_equal(pool[blk, off], want[t]), (t, slot)
            written[blk, off] = True
        assert np.array_equal(pool[~written], old[~written])  # nothing else changed


def test_copy_blocks_of_one_byte_pools_matches_the_numpy_statement():
    rng = np.random.default_rng(17)
    k = rng.integers(0, 256, (6, 16, 2, 64), dtype=np.uint8)
    v = rng.integers(0, 256, (6, 16, 2, 64), dtype=np.uint8)
    m = np.array([[0, 3], [2, 5], [4, 4]])
    got = c_oracle.copy_blocks(k, v, m)
    want = numpy_oracle.copy_blocks(k, v, m)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    assert np.array_equal(got[0][3], k[0]) and np.array_equal(got[1][5], v[2])


# --------------------------------------------------------------------------
# prefill (whole prompts and chunks of them)
# --------------------------------------------------------------------------

def _prefill_batch(seed, ctx, qlen, H=4, Hk=2, d=64, B=16):
    return workloads.build_prefill_batch(name="pf", seed=seed, context_lens=ctx, query_lens=qlen, num_heads=H,
                                         num_kv_heads=Hk, head_dim=d, block_size=B)


def _causal_sdpa(q, K, V, first_pos, scale, group, flag=False):
    """Library attention of one sequence's query rows q [n, H, d] at positions
    first_pos.. over K/V [ctx, Hk, d], with a boolean causal mask (or, for a
    whole prompt, the library's own causal flag)."""
    n = q.shape[0]
    ctx = K.shape[0]
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(np.asarray(K, dtype=np.float64)).permute(1, 0, 2).repeat_interleave(group, dim=0)[None]
    vt = torch.from_numpy(np.asarray(V, dtype=np.float64)).permute(1, 0, 2).repeat_interleave(group, dim=0)[None]
    if flag:
        assert first_pos == 0 and n == ctx
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=float(scale))
    else:
        mask = torch.from_numpy(np.arange(ctx)[None, :] <= (first_pos + np.arange(n))[:, None])
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=float(scale))
    return o[0].permute(1, 0, 2).numpy()


def _prefill_pins(prefill_fn):
    """Names of the prefill pins that `prefill_fn(q, kc, vc, bt, cl, qsl, scale)` fails."""
    failed = []
    # library attention with a causal mask: whole prompts and chunks, GQA 2
    b = _prefill_batch(41, ctx=[1, 37, 40, 23], qlen=[1, 37, 9, 1])
    kc, vc = _written(b)
    got = prefill_fn(b.q, kc, vc, b.block_tables, b.context_lens, b.query_start_loc, b.scale)
    qsl = b.query_start_loc
    for s in range(b.num_seqs):
        c, n = int(b.context_lens[s]), int(qsl[s + 1] - qsl[s])
        K = np.stack([kc[b.block_tables[s, t // 16], t % 16] for t in range(c)]).astype(np.float64)
        V = np.stack([vc[b.block_tables[s, t // 16], t % 16] for t in range(c)]).astype(np.float64)
        ref = _causal_sdpa(b.q[qsl[s]:qsl[s + 1]], K, V, c - n, b.scale, b.group_size, flag=(c == n))
        if not (np.isfinite(got[qsl[s]:qsl[s + 1]]).all() and
                np.allclose(got[qsl[s]:qsl[s + 1]], ref, rtol=0, atol=1e-12)):
            failed.append(f"library-causal-{s}")
    # the first row of a whole prompt returns V[0] exactly
    s = 1
    v0 = vc[b.block_tables[s, 0], 0].astype(np.float64)
    if not np.array_equal(got[qsl[s]], np.repeat(v0, b.group_size, axis=0)):
        failed.append("first-row")
    return failed


def test_prefill_pins_pass_on_both_oracles():
    assert _prefill_pins(c_oracle.prefill) == []
    assert _prefill_pins(numpy_oracle.prefill_bruteforce) == []


@pytest.mark.parametrize("mutant", ["not_causal", "exclusive", "chunk_offset_ignored"])
def test_prefill_pins_catch_planted_mistakes(mutant):
    def mutated(q, kc, vc, bt, cl, qsl, scale):
        cl = np.asarray(cl)
        if mutant == "not_causal":  # every row reads the whole context
            rows = np.repeat(np.arange(len(cl)), np.diff(qsl))
            return numpy_oracle.decode_bruteforce(q, kc, vc, np.asarray(bt)[rows], cl[rows], scale)
        out = np.zeros(q.shape, dtype=np.float64)
        for s in range(len(cl)):
            for i, r in enumerate(range(qsl[s], qsl[s + 1])):
                pos = (cl[s] - (qsl[s + 1] - qsl[s]) + i) if mutant == "exclusive" else i
                n = pos if mutant == "exclusive" else pos + 1
                out[r] = numpy_oracle.decode_bruteforce(q[r:r + 1], kc, vc, np.asarray(bt)[s:s + 1], [n], scale)[0]
        return out
    assert _prefill_pins(mutated) != []


def test_prefill_rows_ignore_every_later_key():
    b = _prefill_batch(42, ctx=[60], qlen=[60])
    kc, vc = _written(b)
    base = c_oracle.prefill(b.q, kc, vc, b.block_tables, b.context_lens, b.query_start_loc, b.scale)
    p = 29
    kc2, vc2 = kc.copy(), vc.copy()
    for t in range(p + 1, 60):  # change every key and value after position p
        blk = b.block_tables[0, t // 16]
        kc2[blk, t % 16] = np.float16(3.0)
        vc2[blk, t % 16] = np.float16(-7.0)
    moved = c_oracle.prefill(b.q, kc2, vc2, b.block_tables, b.context_lens, b.query_start_loc, b.scale)
    assert np.array_equal(base[:p + 1], moved[:p + 1])
    assert not np.array_equal(base[p + 1:], moved[p + 1:])


def test_one_row_chunks_equal_decode():
    b = _prefill_batch(43, ctx=[5, 70, 33], qlen=[1, 1, 1], H=8, Hk=2)
    kc, vc = _written(b)
    pf = c_oracle.prefill(b.q, kc, vc, b.block_tables, b.context_lens, b.query_start_loc, b.scale)
    dec = c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    assert np.array_equal(pf, dec)


def test_prefill_flops_count_the_causal_triangle():
    b = _prefill_batch(44, ctx=[5, 40, 33], qlen=[5, 8, 1])
    # keys seen: 1+2+3+4+5, then 8 rows seeing 33..40, then one row seeing 33
    keys = 15 + sum(range(33, 41)) + 33
    assert workloads.prefill_flops(b) == 4 * b.head_dim * b.num_heads * keys
