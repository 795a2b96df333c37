"""GPU parity for shared-prefix split-K decode (pa_decode_prefix_splitk followed
by pa_splitk_reduce), through the C ABI.

The entry point computes ordinary attention and only reads shared blocks
fewer times, so the oracle is the decode oracle on the same batch (whose
tables share the prompt blocks).  The bounds are those of the other tests:
2e-3 absolute for fp16 and E4M3 caches, 1e-3 + 2^-8 |ref| for bf16.
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


def prefix_batch(seed, prompts, samples, prompt_len, max_suffix, H, Hk, d, B=16, num_seqs=None, ctx=None,
                 dtype="fp16", kv_dtype=""):
    """`prompts` groups of `samples` consecutive sequences sharing `prompt_len`
    tokens; contexts prompt_len + U{0..max_suffix} + 1 unless given."""
    rng = np.random.default_rng(seed)
    S = num_seqs or prompts * samples
    if ctx is None:
        ctx = prompt_len + rng.integers(0, max_suffix + 1, size=S) + 1
    groups = [list(range(p * samples, min(S, (p + 1) * samples))) for p in range(prompts)]
    groups = [g for g in groups if g]
    M = -(-int(max(ctx)) // B) + 1
    return workloads.build_batch(name="prefix", seed=seed, rng=rng, context_lens=ctx, num_heads=H,
                                 num_kv_heads=Hk, head_dim=d, block_size=B, max_blocks_per_seq=M,
                                 share_groups=groups, shared_prefix_len=prompt_len, dtype=dtype,
                                 kv_dtype=kv_dtype)


class Dev:
    def __init__(self, b):
        self.b = b
        self.kc, self.vc = T(b.k_cache), T(b.v_cache)
        self.q, self.bt, self.cl = T(b.q), T(b.block_tables), T(b.context_lens)
        if b.kv_dtype == "fp8":
            api.pa_reshape_and_cache_fp8(T(b.key), T(b.value), self.kc, self.vc, T(b.slot_mapping), b.k_scale,
                                         b.v_scale)
        else:
            api.pa_reshape_and_cache(T(b.key), T(b.value), self.kc, self.vc, T(b.slot_mapping))

    def prefix(self, ps, prefix_lens=None, bt=None, cl=None):
        b = self.b
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
        ws.fill_(float("nan"))
        out = torch.full_like(self.q, 7.0)
        pl = T(np.asarray(b.prefix_lens if prefix_lens is None else prefix_lens, dtype=np.int32))
        bt = self.bt if bt is None else bt
        cl = self.cl if cl is None else cl
        api.pa_decode_prefix_splitk(out, self.q, self.kc, self.vc, bt, cl, b.scale, b.seqs_per_group, pl, ps, ws,
                                    P, k_scale=b.k_scale, v_scale=b.v_scale)
        api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out


def oracle_out(b, seqs=None):
    if b.kv_dtype == "fp8":
        kc, vc = c_oracle.reshape_and_cache_fp8(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping, b.k_scale,
                                                b.v_scale)
    else:
        kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    idx = np.arange(b.num_seqs) if seqs is None else np.asarray(seqs)
    return c_oracle.decode(b.q[idx], kc, vc, b.block_tables[idx], b.context_lens[idx], b.scale, dtype=b.dtype,
                           k_scale=b.k_scale, v_scale=b.v_scale)


def check(gpu, ref, dtype="fp16", rows=None):
    g = gpu.double().cpu().numpy()
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    if dtype == "bf16":
        assert np.all(err <= 1e-3 + 2.0 ** -8 * np.abs(ref)), float(err.max())
    else:
        assert float(err.max()) <= 2e-3, float(err.max())


CASES = {
    # name: (prompts, samples, prompt_len, max_suffix, H, Hk, d, B, partition_size)
    "mha8-two-partitions": (3, 8, 512, 300, 4, 4, 128, 16, 256),
    "gqa4-subgroups": (2, 6, 1024, 600, 16, 4, 128, 16, 512),
    "gqa8-d64-b32": (3, 4, 256, 200, 16, 2, 64, 32, 256),
    "gqa16-one-member-per-cta": (2, 3, 512, 100, 32, 2, 128, 16, 512),
    "gqa4-d256": (2, 4, 512, 300, 8, 2, 256, 16, 256),
    "mha16-one-tile-of-16": (1, 16, 256, 50, 2, 2, 128, 16, 256),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefix_decode_matches_oracle(name):
    prompts, samples, L, suf, H, Hk, d, B, ps = CASES[name]
    b = prefix_batch(21, prompts, samples, L, suf, H, Hk, d, B)
    assert b.seqs_per_group == samples and (b.prefix_lens == L).all()
    check(Dev(b).prefix(ps), oracle_out(b))


def test_prefix_decode_short_last_group():
    b = prefix_batch(22, 3, 5, 512, 200, 8, 8, 128, num_seqs=13)
    assert b.seqs_per_group == 5 and len(b.prefix_lens) == 3
    check(Dev(b).prefix(256), oracle_out(b))


def test_prefix_covering_a_whole_one_partition_sequence():
    # member 1 of group 0 decodes with ctx == prefix == partition_size (its new token,
    # written at position 256, is left out): the shared pass writes its output itself
    ctx = np.array([400, 257, 300, 290, 500, 257, 260, 330])
    b = prefix_batch(23, 2, 4, 256, 0, 4, 4, 128, ctx=ctx)
    d = Dev(b)
    cl = d.cl.clone()
    cl[1] = 256
    out = d.prefix(256, cl=cl)
    b.context_lens[1] = 256
    check(out, oracle_out(b))


@pytest.mark.parametrize("dtype,kv", [("bf16", ""), ("fp16", "fp8")])
def test_prefix_decode_other_element_types(dtype, kv):
    b = prefix_batch(24, 2, 8, 512, 400, 8, 8, 128, dtype=dtype, kv_dtype=kv)
    check(Dev(b).prefix(256), oracle_out(b), dtype)


@pytest.mark.parametrize("lens", [[384, 384], [0, 512], [4096, 512], [-256, 512]])
def test_prefix_lengths_that_do_not_qualify_fall_back_to_per_sequence(lens):
    # not a multiple of the partition, zero, longer than the contexts, negative
    b = prefix_batch(25, 2, 4, 512, 300, 4, 4, 128)
    check(Dev(b).prefix(256, prefix_lens=lens), oracle_out(b))


def test_a_member_whose_table_differs_gets_nan_and_the_others_do_not():
    b = prefix_batch(26, 2, 4, 512, 300, 4, 4, 128)
    ref = oracle_out(b)
    d = Dev(b)
    bt = d.bt.clone()
    spare = int(np.setdiff1d(np.arange(b.num_blocks), b.block_tables).min())
    bt[2, 5] = spare  # sequence 2, a block inside its group's shared prefix
    out = d.prefix(256, bt=bt).double().cpu().numpy()
    assert np.isnan(out[2]).all()
    others = [s for s in range(b.num_seqs) if s != 2]
    assert np.isfinite(out[others]).all()
    assert float(np.abs(out[others] - ref[others]).max()) <= 2e-3


def test_bad_context_length_gives_nan_for_that_sequence_only():
    b = prefix_batch(27, 2, 4, 512, 300, 4, 4, 128)
    ref = oracle_out(b)
    d = Dev(b)
    cl = d.cl.clone()
    cl[5] = -3
    out = d.prefix(256, cl=cl).double().cpu().numpy()
    assert np.isnan(out[5]).all()
    others = [s for s in range(b.num_seqs) if s != 5]
    assert float(np.abs(out[others] - ref[others]).max()) <= 2e-3


@pytest.mark.parametrize("kv_dtype", ["", "fp8"])
def test_prefix_full_size_shared_prefix_every_sequence(kv_dtype):
    b = workloads.shared_prefix(kv_dtype=kv_dtype)
    assert b.seqs_per_group == 8 and (b.prefix_lens == 1024).all()
    check(Dev(b).prefix(512), oracle_out(b))


def test_seqs_per_group_one_is_per_sequence_decode():
    b = prefix_batch(28, 3, 1, 512, 300, 4, 4, 128)
    assert b.seqs_per_group == 1
    check(Dev(b).prefix(256), oracle_out(b))
