"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

* reshape_and_cache: the whole pools, byte for byte, after the write.
* decode (single pass and split-K + reduce): max abs error <= 2e-3 against the
  float64 oracle (fp16 inputs, fp32 accumulation, fp16 output).
* invariants that must hold bit for bit on the GPU: relabelled physical
  blocks, shared vs duplicated prefix, ctx = 1 returns V, run-to-run
  determinism; poisoned (NaN) slots never reach the output.
* device-value outcomes: ctx = 0 gives zeros, an impossible ctx or block id
  gives NaN for the affected group only.

Small cases span several 16-token chunks, warps and partitions with a ragged
tail; the full-size workloads are checked on every sequence.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import c_oracle
from paged_kv_cache_173_gb300 import api, workloads

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def dev():
    return torch.device("cuda:0")


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


class Dev:
    """A batch moved to the GPU, with the cache write applied."""

    def __init__(self, b: workloads.PagedBatch, write: bool = True):
        self.b = b
        self.k_cache = T(b.k_cache)
        self.v_cache = T(b.v_cache)
        self.q = T(b.q)
        self.bt = T(b.block_tables)
        self.cl = T(b.context_lens)
        if write:
            api.pa_reshape_and_cache(T(b.key), T(b.value), self.k_cache, self.v_cache, T(b.slot_mapping))

    def decode(self, cl=None, bt=None):
        out = torch.empty_like(self.q)
        api.pa_decode(out, self.q, self.k_cache, self.v_cache, self.bt if bt is None else bt,
                      self.cl if cl is None else cl, self.b.scale)
        return out

    def splitk(self, ps, cl=None, bt=None):
        b = self.b
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
        ws.fill_(float("nan"))  # the reduce must read only what the partitions wrote
        out = torch.empty_like(self.q)
        cl = self.cl if cl is None else cl
        api.pa_decode_splitk(out, self.q, self.k_cache, self.v_cache, self.bt if bt is None else bt, cl,
                             b.scale, ps, ws, P)
        api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out


def oracle_out(b, seqs=None):
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    if seqs is None:
        return c_oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    seqs = np.asarray(seqs)
    return c_oracle.decode(b.q[seqs], kc, vc, b.block_tables[seqs], b.context_lens[seqs], b.scale)


def max_err(gpu_out, ref):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), "non-finite output"
    return float(np.max(np.abs(g - ref)))


SMALL = {
    "tiny": lambda: workloads.tiny(),
    "llama3-8b-s8": lambda: workloads.llama3_8b(num_seqs=8),
    "llama2-70b-b16": lambda: workloads.llama2_70b(num_seqs=2, ctx=3000, block_size=16),
    "llama2-70b-b32": lambda: workloads.llama2_70b(num_seqs=2, ctx=3001, block_size=32),
    "long-context-s": lambda: workloads.long_context(ctxs=(1000, 4097, 7000)),
    "shared-prefix-s": lambda: workloads.shared_prefix(num_prompts=2, samples=4, prompt_len=256,
                                                       max_suffix=100),
    "mha-d64-b64": lambda: workloads.build_batch(name="d64", seed=4, context_lens=[5, 64, 65, 700, 1],
                                                 num_heads=6, num_kv_heads=6, head_dim=64,
                                                 block_size=64),
    "gqa16-d128-b256": lambda: workloads.build_batch(name="g16", seed=5, context_lens=[300, 513, 1],
                                                     num_heads=32, num_kv_heads=2, head_dim=128,
                                                     block_size=256),
    "gqa3-d64-b16": lambda: workloads.build_batch(name="g3", seed=6, context_lens=[17, 250, 31],
                                                  num_heads=9, num_kv_heads=3, head_dim=64,
                                                  block_size=16),
    # 80 sequences x 8 KV heads: more CTAs than resident slots (456 at three
    # per SM), at most twice as many, so pa_decode ranks the sequences
    # longest first (the lengths repeat, so ties occur)
    "ranked-s80": lambda: _ranked(),
}


def _ranked(seed=11):
    ctx = np.random.default_rng(seed).choice([1, 2, 16, 17, 33, 100, 257, 300], size=80)
    return workloads.build_batch(name="ranked", seed=seed, context_lens=ctx.tolist(), num_heads=32,
                                 num_kv_heads=8, head_dim=128, block_size=16)


@pytest.mark.parametrize("name", list(SMALL))
def test_reshape_and_cache_is_bit_exact(name):
    b = SMALL[name]()
    d = Dev(b)
    ref_k, ref_v = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    torch.cuda.synchronize()
    assert np.array_equal(d.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(d.v_cache.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


def test_reshape_and_cache_skips_padding_and_out_of_range_slots():
    b = workloads.llama3_8b(num_seqs=6, max_ctx=200)
    sm = b.slot_mapping.copy()
    sm[1] = -1
    sm[3] = b.num_blocks * b.block_size + 5  # outside the pool: not written
    d = Dev(b, write=False)
    api.pa_reshape_and_cache(T(b.key), T(b.value), d.k_cache, d.v_cache, T(sm))
    ok = sm.copy()
    ok[3] = -1
    ref_k, ref_v = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, ok)
    torch.cuda.synchronize()
    assert np.array_equal(d.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(d.v_cache.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_matches_oracle(name):
    b = SMALL[name]()
    ref = oracle_out(b)
    d = Dev(b)
    assert max_err(d.decode(), ref) <= TOL


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("ps_blocks", [1, 3, 8, 32])
def test_splitk_matches_oracle(name, ps_blocks):
    b = SMALL[name]()
    ref = oracle_out(b)
    d = Dev(b)
    assert max_err(d.splitk(ps_blocks * b.block_size), ref) <= TOL


def test_ctx_one_returns_v_exactly():
    b = workloads.tiny()
    d = Dev(b)
    out = d.decode().cpu().numpy()
    sk = d.splitk(16).cpu().numpy()
    vc = d.v_cache.cpu().numpy()
    blk = b.block_tables[0, 0]
    for h in range(b.num_heads):
        want = vc[blk, 0, h // b.group_size].view(np.uint16)
        assert np.array_equal(out[0, h].view(np.uint16), want)
        assert np.array_equal(sk[0, h].view(np.uint16), want)


def test_relabelled_blocks_and_determinism_are_bitwise():
    b = workloads.llama3_8b(num_seqs=6, max_ctx=900)
    d = Dev(b)
    base = d.decode().cpu().numpy()
    base_sk = d.splitk(128).cpu().numpy()
    assert np.array_equal(d.decode().cpu().numpy().view(np.uint16), base.view(np.uint16))
    pi = np.random.default_rng(2).permutation(b.num_blocks)
    pit = torch.from_numpy(pi).to(dev())
    k2 = torch.empty_like(d.k_cache)
    v2 = torch.empty_like(d.v_cache)
    k2[pit] = d.k_cache
    v2[pit] = d.v_cache
    bt2 = torch.where(d.bt >= 0, pit[d.bt.clamp(min=0).long()].int(), d.bt)
    d.k_cache, d.v_cache = k2, v2
    out = d.decode(bt=bt2).cpu().numpy()
    sk = d.splitk(128, bt=bt2).cpu().numpy()
    assert np.array_equal(out.view(np.uint16), base.view(np.uint16))
    assert np.array_equal(sk.view(np.uint16), base_sk.view(np.uint16))


def test_shared_prefix_equals_duplicated_blocks_bitwise():
    b = workloads.shared_prefix(num_prompts=2, samples=4, prompt_len=128, max_suffix=60)
    d = Dev(b)
    shared = d.decode().cpu().numpy()
    npre = 128 // b.block_size
    bt = b.block_tables.copy()
    kc = d.k_cache.cpu().numpy()
    vc = d.v_cache.cpu().numpy()
    ek, ev = [], []
    nxt = b.num_blocks
    for s in range(b.num_seqs):
        for i in range(npre):
            ek.append(kc[bt[s, i]])
            ev.append(vc[bt[s, i]])
            bt[s, i] = nxt
            nxt += 1
    d.k_cache = T(np.concatenate([kc, np.stack(ek)]))
    d.v_cache = T(np.concatenate([vc, np.stack(ev)]))
    dup = d.decode(bt=T(bt)).cpu().numpy()
    assert np.array_equal(shared.view(np.uint16), dup.view(np.uint16))


def test_device_value_outcomes():
    b = workloads.llama3_8b(num_seqs=5, max_ctx=400)
    d = Dev(b)
    ref = oracle_out(b)
    cl = b.context_lens.copy()
    cl[1] = 0                                   # empty sequence -> zeros
    cl[2] = b.max_blocks_per_seq * b.block_size + 1  # impossible -> NaN
    bt = b.block_tables.copy()
    bt[3, 0] = b.num_blocks + 7                 # block id outside the pool -> NaN for seq 3
    for out in (d.decode(cl=T(cl), bt=T(bt)), d.splitk(64, cl=T(cl), bt=T(bt))):
        o = out.float().cpu().numpy()
        assert np.all(o[1] == 0)
        assert np.isnan(o[2]).all()
        assert np.isnan(o[3]).all()
        for s in (0, 4):
            assert np.max(np.abs(o[s] - ref[s])) <= TOL


def test_ranked_decode_device_value_outcomes():
    # the longest-first launch puts each result in its own sequence's row,
    # whatever rank its context length has (an impossible length ranks first)
    b = _ranked(seed=12)
    d = Dev(b)
    ref = oracle_out(b)
    cl = b.context_lens.copy()
    cl[10] = 0
    cl[20] = b.max_blocks_per_seq * b.block_size + 1
    cl[30] = -4
    bt = b.block_tables.copy()
    bt[40, 0] = b.num_blocks + 7
    o = d.decode(cl=T(cl), bt=T(bt)).float().cpu().numpy()
    assert np.all(o[10] == 0)
    assert np.isnan(o[20]).all() and np.isnan(o[30]).all() and np.isnan(o[40]).all()
    keep = np.setdiff1d(np.arange(b.num_seqs), [10, 20, 30, 40])
    assert np.max(np.abs(o[keep] - ref[keep])) <= TOL


def _few_pairs(ctx, seed=7):
    # few (sequence, KV head) pairs and a large table capacity: pa_decode runs
    # clusters of 8 CTAs per pair, so short sequences leave CTAs without chunks
    return workloads.build_batch(name="few", seed=seed, context_lens=ctx, num_heads=4, num_kv_heads=1,
                                 head_dim=128, block_size=16, max_blocks_per_seq=256)


def test_cluster_decode_with_empty_ctas():
    b = _few_pairs([1, 5, 17, 100, 1000, 4096])
    ref = oracle_out(b)
    d = Dev(b)
    assert max_err(d.decode(), ref) <= TOL
    assert max_err(d.splitk(64), ref) <= TOL


def test_cluster_device_value_outcomes():
    b = _few_pairs([300, 40, 2000, 77])
    d = Dev(b)
    ref = oracle_out(b)
    cl = b.context_lens.copy()
    cl[0] = 0
    cl[1] = b.max_blocks_per_seq * b.block_size + 3
    bt = b.block_tables.copy()
    bt[2, 100] = -5
    o = d.decode(cl=T(cl), bt=T(bt)).float().cpu().numpy()
    assert np.all(o[0] == 0)
    assert np.isnan(o[1]).all()
    assert np.isnan(o[2]).all()
    assert np.max(np.abs(o[3] - ref[3])) <= TOL


def test_empty_batch():
    b = workloads.tiny()
    d = Dev(b)
    out = torch.empty((0, b.num_heads, b.head_dim), dtype=torch.float16, device=dev())
    api.pa_decode(out, d.q[:0], d.k_cache, d.v_cache, d.bt[:0], d.cl[:0], b.scale)


# ------------------------------------------------------------------ full size
FULL = {
    "llama3-8b": (lambda: workloads.llama3_8b(), 512),
    "llama2-70b-b16": (lambda: workloads.llama2_70b(block_size=16), 512),
    "llama2-70b-b32": (lambda: workloads.llama2_70b(block_size=32), 512),
    "long-context": (lambda: workloads.long_context(), 512),
    "shared-prefix": (lambda: workloads.shared_prefix(), 512),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workloads_every_sequence(name):
    # every sequence of the full workload against the oracle, for the single
    # launch and for split-K (the launch shapes bench.py times)
    make, ps = FULL[name]
    b = make()
    d = Dev(b)
    sk = d.splitk(ps)
    single = d.decode()
    ref = oracle_out(b)
    assert max_err(sk, ref) <= TOL
    assert max_err(single, ref) <= TOL
    # the cache write at full size, byte for byte
    ref_k, ref_v = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    assert np.array_equal(d.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(d.v_cache.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


# ------------------------------------------------------------ copy-on-write
@pytest.mark.parametrize("shape", [(16, 8, 128), (256, 8, 128), (32, 4, 64)])
def test_copy_blocks_is_bit_exact(shape):
    B, Hk, d = shape
    b = workloads.build_batch(name="cp", seed=12, context_lens=[B * 3 + 1, B * 2], num_heads=Hk,
                              num_kv_heads=Hk, head_dim=d, block_size=B, num_blocks=20, poison=True)
    srcs = [int(b.block_tables[0, 0]), int(b.block_tables[0, 3]), int(b.block_tables[1, 1])]
    free = [i for i in range(b.num_blocks) if i not in set(b.block_tables[b.block_tables >= 0].tolist())]
    pairs = np.array([[srcs[0], free[0]], [srcs[1], free[1]], [4, 4],
                      [2, b.num_blocks + 3], [srcs[2], free[2]]], np.int64)
    kc, vc = T(b.k_cache), T(b.v_cache)
    api.pa_copy_blocks(kc, vc, T(pairs))
    ref_k, ref_v = c_oracle.copy_blocks(b.k_cache, b.v_cache, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


def test_copy_on_write_fork_then_decode():
    # 8 samples share a 2-block prompt whose last block is partial (20 tokens);
    # sample 3 forks: its shared last block is copied, repointed, then written
    B, S = 16, 8
    b = workloads.build_batch(name="fork", seed=13, context_lens=[20], num_heads=8, num_kv_heads=2,
                              head_dim=128, block_size=B, new_token=False, poison=True, num_blocks=12)
    q = np.random.default_rng(3).standard_normal((S, 8, 128), dtype=np.float32).astype(np.float16)
    bt = np.repeat(b.block_tables, S, axis=0)
    kc_h, vc_h = b.k_cache.copy(), b.v_cache.copy()
    # the shared prompt: every sample reads blocks bt[0]
    free = [i for i in range(b.num_blocks) if i not in set(bt[0].tolist())][0]
    shared_last = int(bt[0, 1])
    newk = np.random.default_rng(1).standard_normal((1, 2, 128), dtype=np.float32).astype(np.float16)
    newv = np.random.default_rng(2).standard_normal((1, 2, 128), dtype=np.float32).astype(np.float16)
    slot = np.array([free * B + 20 % B], np.int64)
    bt2 = bt.copy()
    bt2[3, 1] = free
    cl = np.full(S, 20, np.int32)
    cl[3] = 21
    # oracle: copy, write, decode
    ok, ov = c_oracle.copy_blocks(kc_h, vc_h, [[shared_last, free]])
    ok, ov = c_oracle.reshape_and_cache(newk, newv, ok, ov, slot)
    ref = c_oracle.decode(q, ok, ov, bt2, cl, b.scale)
    # GPU: the same three calls
    kc, vc = T(kc_h), T(vc_h)
    api.pa_copy_blocks(kc, vc, T(np.array([[shared_last, free]], np.int64)))
    api.pa_reshape_and_cache(T(newk), T(newv), kc, vc, T(slot))
    out = torch.empty_like(T(q))
    api.pa_decode(out, T(q), kc, vc, T(bt2), T(cl), b.scale)
    assert max_err(out, ref) <= TOL
    # the other samples still read the shared block, unchanged
    assert np.array_equal(kc.cpu().numpy()[shared_last].view(np.uint16), kc_h[shared_last].view(np.uint16))


# ------------------------------------------------------------ maximum sizes
def test_the_largest_batch_every_sequence():
    # num_seqs at its limit (65535, the grid's z extent): every entry point, every sequence
    rng = np.random.default_rng(61)
    b = workloads.build_batch(name="max-batch", seed=61, rng=rng, context_lens=rng.integers(1, 33, size=65535),
                              num_heads=8, num_kv_heads=1, head_dim=64, block_size=16)
    assert b.num_seqs == 65535
    ref = oracle_out(b)
    d = Dev(b)
    assert max_err(d.decode(), ref) <= TOL
    assert max_err(d.splitk(16), ref) <= TOL
    ref_k, ref_v = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    assert np.array_equal(d.k_cache.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    # the fused step on fresh pools: the same write and the same attention
    kc, vc = T(b.k_cache), T(b.v_cache)
    out = torch.empty_like(d.q)
    api.pa_append_and_decode(out, d.q, T(b.key), T(b.value), kc, vc, d.bt, d.cl, b.scale)
    assert max_err(out, ref) <= TOL
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), ref_v.view(np.uint16))
