"""GPU parity of the fused decode step (pa_append_and_decode and
pa_append_and_decode_splitk), through the C ABI.

A decode step writes each sequence's new token into its slot, then attends
over the whole context ("Efficient Memory Management for LLM Serving with
PagedAttention -- in-depth reading", section 3.4, steps 1 and 3).  The fused
entry points do both in the decode launch.  Against the oracle:

* the pools after the call equal the oracle's cache write, byte for byte
  (E4M3 pools: the oracle's quantisation), with the slot of position ctx - 1
  taken from the block table;
* the output is within the decode tolerance of the oracle over the written
  pools (2e-3 for fp16 and E4M3, 1e-3 + 2^-8 |ref| for bf16);
* and it is bit-identical to the separate cache write followed by the
  matching decode, since the new row enters the same arithmetic.

Device-value outcomes: an empty sequence writes nothing and gives zeros; an
impossible context length or an out-of-pool block id at the new position
writes nothing and gives NaN; the other sequences are unaffected.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import c_oracle
from paged_kv_cache_173_gb300 import api, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def dev():
    return torch.device("cuda:0")


def T(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(a).to(dev())


def bits(t):
    a = t.cpu()
    if a.dtype in (torch.float16, torch.bfloat16):
        return a.view(torch.int16).numpy()
    return a.numpy()


def check(gpu, ref, dtype):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    if dtype == "bf16":
        assert np.all(err <= 1e-3 + 2.0 ** -8 * np.abs(ref)), float(err.max())
    else:
        assert float(err.max()) <= 2e-3, float(err.max())


def table_slots(b, cl=None):
    """The slot of position ctx - 1 of each sequence, from its table row (-1 where none)."""
    cl = b.context_lens if cl is None else cl
    sm = np.full(b.num_seqs, -1, np.int64)
    for s, c in enumerate(cl):
        c = int(c)
        if 1 <= c <= b.max_blocks_per_seq * b.block_size:
            blk = int(b.block_tables[s, (c - 1) // b.block_size])
            if 0 <= blk < b.num_blocks:
                sm[s] = blk * b.block_size + (c - 1) % b.block_size
    return sm


def oracle_step(b, cl=None, bt=None):
    """The oracle's cache write (slots from the table) and decode over the written pools."""
    cl = b.context_lens if cl is None else cl
    bt = b.block_tables if bt is None else bt
    bb = b if bt is b.block_tables else _with_table(b, bt)
    sm = table_slots(bb, cl)
    if b.kv_dtype == "fp8":
        kc, vc = c_oracle.reshape_and_cache_fp8(b.key, b.value, b.k_cache, b.v_cache, sm, b.k_scale, b.v_scale)
    else:
        kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, sm)
    ref = c_oracle.decode(b.q, kc, vc, bt, cl, b.scale, dtype=b.dtype, k_scale=b.k_scale, v_scale=b.v_scale)
    return kc, vc, ref, sm


def _with_table(b, bt):
    import dataclasses
    return dataclasses.replace(b, block_tables=bt)


class Step:
    """A batch on the GPU, before the new tokens are written."""

    def __init__(self, b):
        self.b = b
        self.k_cache, self.v_cache = T(b.k_cache), T(b.v_cache)
        self.q, self.key, self.value = T(b.q), T(b.key), T(b.value)
        self.bt, self.cl = T(b.block_tables), T(b.context_lens)

    def fused(self, ps=None, cl=None, bt=None):
        b = self.b
        out = torch.full_like(self.q, 7.0)
        cl = self.cl if cl is None else cl
        bt = self.bt if bt is None else bt
        if ps is None:
            api.pa_append_and_decode(out, self.q, self.key, self.value, self.k_cache, self.v_cache, bt, cl, b.scale,
                                     k_scale=b.k_scale, v_scale=b.v_scale)
        else:
            P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
            ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
            ws.fill_(float("nan"))
            api.pa_append_and_decode_splitk(out, self.q, self.key, self.value, self.k_cache, self.v_cache, bt, cl,
                                            b.scale, ps, ws, P, k_scale=b.k_scale, v_scale=b.v_scale)
            api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out

    def separate(self, ps=None):
        """pa_reshape_and_cache(_fp8) with the table's slots, then pa_decode(_splitk)(_fp8)."""
        b = self.b
        sm = T(table_slots(b))
        out = torch.full_like(self.q, 7.0)
        fp8 = b.kv_dtype == "fp8"
        if fp8:
            api.pa_reshape_and_cache_fp8(self.key, self.value, self.k_cache, self.v_cache, sm, b.k_scale, b.v_scale)
        else:
            api.pa_reshape_and_cache(self.key, self.value, self.k_cache, self.v_cache, sm)
        if ps is None:
            if fp8:
                api.pa_decode_fp8(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale, b.k_scale,
                                  b.v_scale)
            else:
                api.pa_decode(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale)
        else:
            P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
            ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
            if fp8:
                api.pa_decode_splitk_fp8(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale,
                                         b.k_scale, b.v_scale, ps, ws, P)
            else:
                api.pa_decode_splitk(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale, ps, ws, P)
            api.pa_splitk_reduce(out, ws, self.cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out


def small(name, dtype="fp16", kv_dtype=""):
    kw = dict(dtype=dtype, kv_dtype=kv_dtype)
    cases = {
        "tiny": lambda: workloads.build_batch(name="tiny", seed=0, context_lens=[1, 15, 16, 37], num_heads=4,
                                              num_kv_heads=4, head_dim=64, block_size=16, num_blocks=16,
                                              max_blocks_per_seq=3, **kw),
        "llama3-8b-s8": lambda: workloads.llama3_8b(num_seqs=8, **kw),
        "llama2-70b-b32": lambda: workloads.llama2_70b(num_seqs=2, ctx=3001, block_size=32, **kw),
        "long-context-s": lambda: workloads.long_context(ctxs=(1000, 4097, 7000), **kw),
        "gqa16-d128-b256": lambda: workloads.build_batch(name="g16", seed=5, context_lens=[300, 513, 1],
                                                         num_heads=32, num_kv_heads=2, head_dim=128,
                                                         block_size=256, **kw),
        "d256-gqa4": lambda: workloads.build_batch(name="d256", seed=9, context_lens=[1, 200, 1500, 16, 17],
                                                   num_heads=16, num_kv_heads=4, head_dim=256, block_size=16, **kw),
        # more (sequence, KV head) pairs than resident CTAs (three per SM at
        # d = 128), but at most twice as many: the single launch ranks the
        # sequences longest first; the lengths repeat
        "ranked": lambda: workloads.build_batch(name="ranked", seed=11, context_lens=RANKED_CTX, num_heads=32,
                                                num_kv_heads=8, head_dim=128, block_size=16, **kw),
        # few (sequence, KV head) pairs, large capacity: the single launch runs clusters
        "cluster": lambda: workloads.build_batch(name="few", seed=7, context_lens=[1, 5, 17, 100, 1000, 4096],
                                                 num_heads=4, num_kv_heads=1, head_dim=128, block_size=16,
                                                 max_blocks_per_seq=256, **kw),
    }
    return cases[name]()


RANKED_CTX = np.random.default_rng(11).choice([1, 2, 16, 17, 33, 100, 257, 300], size=80).tolist()
NAMES = ["tiny", "llama3-8b-s8", "llama2-70b-b32", "long-context-s", "gqa16-d128-b256", "d256-gqa4", "ranked",
         "cluster"]
TYPES = [("fp16", ""), ("bf16", ""), ("fp16", "fp8")]


@pytest.mark.parametrize("dtype,kv_dtype", TYPES, ids=["fp16", "bf16", "e4m3"])
@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("ps_blocks", [None, 1, 4])
def test_append_matches_oracle_and_the_separate_step(name, dtype, kv_dtype, ps_blocks):
    b = small(name, dtype, kv_dtype)
    ps = None if ps_blocks is None else ps_blocks * b.block_size
    kc, vc, ref, _ = oracle_step(b)
    st = Step(b)
    out = st.fused(ps)
    torch.cuda.synchronize()
    assert np.array_equal(bits(st.k_cache), kc.view(bits(st.k_cache).dtype))
    assert np.array_equal(bits(st.v_cache), vc.view(bits(st.v_cache).dtype))
    check(out, ref, dtype)
    sep = Step(b).separate(ps)
    assert np.array_equal(bits(out), bits(sep))


@pytest.mark.parametrize("kv_dtype", ["", "fp8"])
def test_append_ctx_one_returns_the_new_value(kv_dtype):
    # a sequence of one token attends to the token it writes: out = its V row
    b = workloads.build_batch(name="one", seed=3, context_lens=[1, 1, 40], num_heads=8, num_kv_heads=2,
                              head_dim=128, block_size=16, kv_dtype=kv_dtype)
    kc, vc, ref, sm = oracle_step(b)
    out = Step(b).fused().cpu().numpy()
    for s in (0, 1):
        for h in range(8):
            if kv_dtype == "fp8":  # the dequantised code, rounded to fp16
                want = ref[s, h].astype(np.float16)
                assert np.array_equal(out[s, h].view(np.uint16), want.view(np.uint16))
            else:
                assert np.array_equal(out[s, h].view(np.uint16), b.value[s, h // 4].view(np.uint16))


@pytest.mark.parametrize("ps", [None, 64])
def test_append_device_value_outcomes(ps):
    b = workloads.llama3_8b(num_seqs=6, max_ctx=400)
    cl = b.context_lens.copy()
    cl[1] = 0                                          # empty: nothing written, zeros
    cl[2] = b.max_blocks_per_seq * b.block_size + 1    # impossible: nothing written, NaN
    bt = b.block_tables.copy()
    bt[3, (int(cl[3]) - 1) // b.block_size] = b.num_blocks + 7  # the new position's block outside the pool
    sm = table_slots(_with_table(b, bt), cl)
    assert sm[1] == -1 and sm[2] == -1 and sm[3] == -1  # nothing to write for these three
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, sm)
    good = [0, 4, 5]
    ref = c_oracle.decode(b.q[good], kc, vc, b.block_tables[good], b.context_lens[good], b.scale)
    st = Step(b)
    o = st.fused(ps, cl=T(cl), bt=T(bt)).float().cpu().numpy()
    assert np.array_equal(bits(st.k_cache), kc.view(np.int16))
    assert np.array_equal(bits(st.v_cache), vc.view(np.int16))
    assert np.all(o[1] == 0)
    assert np.isnan(o[2]).all()
    assert np.isnan(o[3]).all()
    for i, s in enumerate(good):
        assert np.max(np.abs(o[s] - ref[i])) <= 2e-3


FULL = {
    "llama3-8b": lambda: workloads.llama3_8b(),
    "llama2-70b-b16": lambda: workloads.llama2_70b(block_size=16),
    "long-context": lambda: workloads.long_context(),
    "llama3-8b-e4m3": lambda: workloads.llama3_8b(kv_dtype="fp8"),
}


@pytest.mark.parametrize("name", list(FULL))
def test_append_full_size_every_sequence(name):
    b = FULL[name]()
    kc, vc, ref, _ = oracle_step(b)
    for ps in (None, 512):
        st = Step(b)
        out = st.fused(ps)
        torch.cuda.synchronize()
        assert np.array_equal(bits(st.k_cache), kc.view(bits(st.k_cache).dtype))
        assert np.array_equal(bits(st.v_cache), vc.view(bits(st.v_cache).dtype))
        check(out, ref, b.dtype)
