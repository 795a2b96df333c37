"""GPU parity for paged prefill (pa_prefill after pa_reshape_and_cache), through
the C ABI.

Tolerance, from the arithmetic: scores, softmax and accumulation are float32.
fp16: the attention weights enter P.V rounded to fp16 and the running sums add
the same rounded weights; the 2e-3 absolute bound of the decode tests holds.
bf16: the weights enter as a bf16 value plus its bf16 residual (about 16
bits) and the sums add the unrounded weights, so the error is dominated by
the output's own rounding to bf16 (half an ulp, 2^-8 |out|): the bound is
1e-3 + 2^-8 |ref|, as for bf16 decode.
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


def run(b, cl=None, bt=None):
    kc, vc = T(b.k_cache), T(b.v_cache)
    api.pa_reshape_and_cache(T(b.key), T(b.value), kc, vc, T(b.slot_mapping))
    q = T(b.q)
    out = torch.full_like(q, 5.0)
    qsl = T(b.query_start_loc)
    ql = np.diff(b.query_start_loc)
    api.pa_prefill(out, q, kc, vc, T(b.block_tables) if bt is None else bt,
                   T(b.context_lens) if cl is None else cl, qsl, int(ql.max()) if ql.size else 0, b.scale)
    return out


def oracle(b):
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    return c_oracle.prefill(b.q, kc, vc, b.block_tables, b.context_lens, b.query_start_loc, b.scale,
                            dtype=b.dtype)


def check(gpu, ref, dtype="fp16"):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    if dtype == "bf16":
        assert np.all(err <= 1e-3 + 2.0 ** -8 * np.abs(ref)), float(err.max())
    else:
        assert float(err.max()) <= 2e-3, float(err.max())


def batch(seed, ctx, qlen, H, Hk, d, B=16, dtype="fp16"):
    return workloads.build_prefill_batch(name="pf", seed=seed, context_lens=ctx, query_lens=qlen, num_heads=H,
                                         num_kv_heads=Hk, head_dim=d, block_size=B, dtype=dtype)


CASES = {
    # name: (contexts, query lengths, H, Hk, d, B)
    "whole-prompts-mha": ([1, 15, 16, 17, 64, 65, 300], [1, 15, 16, 17, 64, 65, 300], 4, 4, 128, 16),
    "chunks-gqa4": ([200, 513, 97, 64], [64, 100, 1, 64], 16, 4, 128, 16),
    "mixed-gqa8-d64-b32": ([130, 260, 33], [130, 7, 33], 16, 2, 64, 32),
    "gqa2-b256": ([600, 300], [600, 150], 8, 4, 128, 256),
    "gqa16-d64": ([90, 45], [90, 20], 32, 2, 64, 16),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    ctx, ql, H, Hk, d, B = CASES[name]
    b = batch(31, ctx, ql, H, Hk, d, B)
    check(run(b), oracle(b))


@pytest.mark.parametrize("name", ["whole-prompts-mha", "chunks-gqa4", "mixed-gqa8-d64-b32"])
def test_prefill_bf16_matches_oracle(name):
    ctx, ql, H, Hk, d, B = CASES[name]
    b = batch(32, ctx, ql, H, Hk, d, B, dtype="bf16")
    check(run(b), oracle(b), "bf16")


def test_prompts_spanning_several_tile_pairs_with_a_ragged_last_pair():
    # MHA at d = 64: a tile is 128 tokens, a CTA's pair 256; 700 and 1100 tokens leave a last
    # pair with one partial tile, and 300 leaves a pair whose second tile does not exist
    b = batch(37, [700, 1100, 300], [700, 1100, 300], 4, 4, 64)
    check(run(b), oracle(b))


def test_first_row_of_a_prompt_returns_its_value():
    b = batch(33, [40], [40], 8, 2, 128)
    out = run(b).view(torch.int16).cpu().numpy()
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    v0 = vc[b.block_tables[0, 0], 0].view(np.int16)
    for h in range(8):
        assert np.array_equal(out[0, h], v0[h // 4])


def test_device_value_outcomes():
    b = batch(34, [64, 80, 50], [64, 30, 50], 8, 2, 128)
    ref = oracle(b)
    cl = T(b.context_lens).clone()
    cl[1] = 10  # below its 30 query rows
    bt = T(b.block_tables).clone()
    bt[2, 1] = b.num_blocks + 3  # a block id outside the pool, read by sequence 2
    out = run(b, cl=cl, bt=bt).double().cpu().numpy()
    qsl = b.query_start_loc
    assert np.isnan(out[qsl[1]:qsl[2]]).all()
    assert np.isnan(out[qsl[2]:qsl[3]][16:]).all()  # rows reading block 1 (positions >= 16)
    np.testing.assert_allclose(out[qsl[0]:qsl[1]], ref[qsl[0]:qsl[1]], rtol=0, atol=2e-3)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_full_size_llama3_8b_prompts(dtype):
    # 8 whole prompts of 2048 tokens, Llama-3-8B heads (the bench workload's shape): every row
    # of prompt 3 against the prefill oracle, and the first and last 256 rows of every prompt
    # (each a 256-token prompt of its own, or decode rows over their own prefix)
    b = batch(35, [2048] * 8, [2048] * 8, 32, 8, 128, dtype=dtype)
    out = run(b)
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    qsl = b.query_start_loc

    def close(got, ref):
        check(got, ref, dtype)

    s = 3
    one = c_oracle.prefill(b.q[qsl[s]:qsl[s + 1]], kc, vc, b.block_tables[s:s + 1], b.context_lens[s:s + 1],
                           np.array([0, 2048], np.int32), b.scale, dtype=b.dtype)
    close(out[qsl[s]:qsl[s + 1]], one)
    for s in range(8):
        r0 = qsl[s]
        head = c_oracle.prefill(b.q[r0:r0 + 256], kc, vc, b.block_tables[s:s + 1], np.array([256], np.int32),
                                np.array([0, 256], np.int32), b.scale, dtype=b.dtype)
        close(out[r0:r0 + 256], head)
        tail = c_oracle.decode(b.q[r0 + 1792:r0 + 2048], kc, vc, np.repeat(b.block_tables[s:s + 1], 256, axis=0),
                               np.arange(1793, 2049, dtype=np.int32), b.scale, dtype=b.dtype)
        close(out[r0 + 1792:r0 + 2048], tail)


def test_prefill_is_repeatable_bit_for_bit():
    # the kernel's arithmetic order is fixed, so repeated launches agree to the bit; a
    # race between the pipeline's stages (a buffer reused too early) would show here
    b = batch(36, [700, 1500, 130], [700, 900, 130], 32, 8, 128)
    kc, vc = T(b.k_cache), T(b.v_cache)
    api.pa_reshape_and_cache(T(b.key), T(b.value), kc, vc, T(b.slot_mapping))
    q, bt, cl, qsl = T(b.q), T(b.block_tables), T(b.context_lens), T(b.query_start_loc)
    outs = []
    for _ in range(8):
        out = torch.empty_like(q)
        api.pa_prefill(out, q, kc, vc, bt, cl, qsl, 900, b.scale)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    check(outs[0], oracle(b))
