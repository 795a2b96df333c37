"""GPU parity for E4M3 (FP8) caches, through the C ABI.

The cache write is integer work (a code per element) and must match the
oracle bit for bit: the quotient x / scale is rounded once to float32 on both
sides and then to the nearest code, ties to even, saturating at 448.

Decode tolerance, derived from the arithmetic: codes widen exactly to fp16,
so K and V enter the MMAs without error; q . K is exact products summed in
float32; the weights enter P.V rounded to fp16 (2^-11 relative) and the
output is rounded to fp16 (half an ulp: 2^-11 |out|, |out| <~ 4 here).  The
pools hold N(0,1) values, as in the 16-bit tests, so the 2e-3 absolute bound
of the fp16 tests applies unchanged.
"""
from __future__ import annotations

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
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(a).to(dev())


def fp8_batch(name, seed, **kw):
    return workloads.build_batch(name=name, seed=seed, kv_dtype="fp8", **kw)


class Dev:
    def __init__(self, b: workloads.PagedBatch, key=None, value=None):
        self.b = b
        self.k_cache = T(b.k_cache)
        self.v_cache = T(b.v_cache)
        self.q = T(b.q)
        self.bt = T(b.block_tables)
        self.cl = T(b.context_lens)
        self.key = b.key if key is None else key
        self.value = b.value if value is None else value
        api.pa_reshape_and_cache_fp8(T(self.key), T(self.value), self.k_cache, self.v_cache,
                                     T(b.slot_mapping), b.k_scale, b.v_scale)

    def decode(self):
        out = torch.empty_like(self.q)
        api.pa_decode_fp8(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, self.b.scale,
                          self.b.k_scale, self.b.v_scale)
        return out

    def splitk(self, ps):
        b = self.b
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
        ws.fill_(float("nan"))
        out = torch.empty_like(self.q)
        api.pa_decode_splitk_fp8(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale,
                                 b.k_scale, b.v_scale, ps, ws, P)
        api.pa_splitk_reduce(out, ws, self.cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out


def oracle_caches(b, key=None, value=None, dtype="fp16"):
    return c_oracle.reshape_and_cache_fp8(b.key if key is None else key, b.value if value is None else value,
                                          b.k_cache, b.v_cache, b.slot_mapping, b.k_scale, b.v_scale,
                                          dtype=dtype)


def oracle_out(b, seqs=None):
    kc, vc = oracle_caches(b)
    idx = np.arange(b.num_seqs) if seqs is None else np.asarray(seqs)
    return c_oracle.decode(b.q[idx], kc, vc, b.block_tables[idx], b.context_lens[idx], b.scale,
                           k_scale=b.k_scale, v_scale=b.v_scale)


def check(gpu: torch.Tensor, ref: np.ndarray):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = float(np.abs(g - ref).max())
    assert err <= TOL, err


CASES = {
    # name: (context_lens, H, Hk, d, B)
    "llama3-8b-s6": ([1, 130, 777, 2048, 15, 1031], 32, 8, 128, 16),
    "gqa8-b32": ([3001, 64], 64, 8, 128, 32),
    "mha-d64-b64": ([5, 64, 65, 700], 6, 6, 64, 64),
    "gqa16-d128": ([300, 513, 1], 32, 2, 128, 16),
    "gqa4-d256": ([17, 1000, 2500], 16, 4, 256, 16),
    "gqa8-d256-b128": ([333, 4096], 16, 2, 256, 128),
    "gqa2-d64-b256": ([255, 256, 257, 1], 8, 4, 64, 256),
}


def case(name, seed=11):
    ctx, H, Hk, d, B = CASES[name]
    return fp8_batch(name, seed, context_lens=ctx, num_heads=H, num_kv_heads=Hk, head_dim=d, block_size=B,
                     max_blocks_per_seq=-(-max(ctx) // B) + 1)


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_cache_write_is_bit_exact(name):
    b = case(name)
    d = Dev(b)
    ref_k, ref_v = oracle_caches(b)
    torch.cuda.synchronize()
    assert np.array_equal(d.k_cache.cpu().numpy(), ref_k)
    assert np.array_equal(d.v_cache.cpu().numpy(), ref_v)


def test_fp8_cache_write_ties_saturation_and_bf16_keys():
    b = case("llama3-8b-s6", seed=12)
    rng = np.random.default_rng(5)
    # fp16 keys: midpoints between codes (ties), subnormal codes, values far past 448 * scale
    sc = b.k_scale
    ties = np.array([1.0625, 1.1875, -2.125, 0.5 * 2.0 ** -9, 1.5 * 2.0 ** -9, 460.0, -464.0, 1000.0],
                    np.float64) * sc
    key = (rng.standard_normal(b.key.shape) * 20.0).astype(np.float16)
    key.reshape(-1)[:ties.size] = ties.astype(np.float16)
    value = b.value.copy()
    d = Dev(b, key=key, value=value)
    ref_k, ref_v = oracle_caches(b, key=key, value=value)
    torch.cuda.synchronize()
    got_k = d.k_cache.cpu().numpy()
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(d.v_cache.cpu().numpy(), ref_v)
    assert (ref_k == 0x7E).any() and (ref_k == 0xFE).any()  # saturation was exercised
    # bfloat16 keys and values
    kb = workloads.f32_to_bf16_bits(rng.standard_normal(b.key.shape).astype(np.float32))
    vb = workloads.f32_to_bf16_bits(rng.standard_normal(b.value.shape).astype(np.float32))
    d2 = Dev(b, key=kb, value=vb)
    ref_k2, ref_v2 = oracle_caches(b, key=kb, value=vb, dtype="bf16")
    torch.cuda.synchronize()
    assert np.array_equal(d2.k_cache.cpu().numpy(), ref_k2)
    assert np.array_equal(d2.v_cache.cpu().numpy(), ref_v2)


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_decode_matches_oracle(name):
    b = case(name)
    ref = oracle_out(b)
    d = Dev(b)
    check(d.decode(), ref)
    for ps in (b.block_size, 4 * b.block_size, 512, 2048):
        if ps % b.block_size == 0:
            check(d.splitk(ps), ref)


def test_fp8_single_token_returns_scaled_v():
    b = case("llama3-8b-s6")
    d = Dev(b)
    assert b.context_lens[0] == 1
    out = d.decode().cpu().numpy()
    vc = d.v_cache.cpu().numpy()
    blk = b.block_tables[0, 0]
    for h in range(b.num_heads):
        codes = vc[blk, 0, h // b.group_size]
        want = (np.array([c_oracle.e4m3_to_double(int(c)) for c in codes]) * b.v_scale).astype(np.float16)
        assert np.array_equal(out[0, h].view(np.uint16), want.view(np.uint16))


def test_fp8_device_value_outcomes():
    b = case("gqa16-d128")
    d = Dev(b)
    cl = d.cl.clone()
    cl[0] = 0
    cl[2] = b.max_blocks_per_seq * b.block_size + 1
    bt = d.bt.clone()
    bt[1, 3] = b.num_blocks + 7
    out = torch.full_like(d.q, 5.0)
    api.pa_decode_fp8(out, d.q, d.k_cache, d.v_cache, bt, cl, b.scale, b.k_scale, b.v_scale)
    o = out.cpu().float().numpy()
    assert (o[0] == 0).all()
    assert np.isnan(o[1]).all()
    assert np.isnan(o[2]).all()


def test_fp8_accepts_float8_tensors():
    b = case("mha-d64-b64")
    d = Dev(b)
    ref = oracle_out(b)
    out = torch.empty_like(d.q)
    api.pa_decode_fp8(out, d.q, d.k_cache.view(torch.float8_e4m3fn), d.v_cache.view(torch.float8_e4m3fn), d.bt,
                      d.cl, b.scale, b.k_scale, b.v_scale)
    check(out, ref)


def test_fp8_copy_blocks_is_bit_exact():
    b = case("gqa8-b32")
    d = Dev(b)
    kc0, vc0 = oracle_caches(b)
    used = set(np.unique(b.block_tables).tolist())
    free = [i for i in range(b.num_blocks) if i not in used][:3]
    src = [int(b.block_tables[0, 0]), int(b.block_tables[0, 5]), int(b.block_tables[1, 1])]
    mapping = np.array(list(zip(src, free)), np.int64)
    api.pa_copy_blocks(d.k_cache, d.v_cache, T(mapping))
    ref_k, ref_v = c_oracle.copy_blocks(kc0, vc0, mapping)
    torch.cuda.synchronize()
    assert np.array_equal(d.k_cache.cpu().numpy(), ref_k)
    assert np.array_equal(d.v_cache.cpu().numpy(), ref_v)


@pytest.mark.parametrize("name", ["llama3-8b", "llama2-70b-b16", "long-context"])
def test_fp8_full_size_every_sequence(name):
    make = {"llama3-8b": lambda: workloads.llama3_8b(kv_dtype="fp8"),
            "llama2-70b-b16": lambda: workloads.llama2_70b(block_size=16, kv_dtype="fp8"),
            "long-context": lambda: workloads.long_context(kv_dtype="fp8")}[name]
    b = make()
    d = Dev(b)
    ref = oracle_out(b)
    check(d.decode(), ref)
    check(d.splitk(512), ref)
    check(d.splitk(1024), ref)
