"""GPU parity for bfloat16 caches and for head_dim 256, through the C ABI.

bf16 tolerance, derived from the arithmetic: the output is rounded to bf16
(8 significant bits: at most half an ulp, 2^-8 of |out|); scores, softmax and
accumulation are float32 and the attention weights enter P.V as a bf16 value
plus its bf16 residual (about 16 bits), so the rest of the error stays far
below 1e-3.  The test bound is |gpu - oracle| <= 1e-3 + 2^-8 |oracle|.
fp16 keeps the 2e-3 absolute bound of the other parity tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import c_oracle
from paged_kv_cache_173_gb300 import api, workloads

pytestmark = pytest.mark.gpu
TOL_F16 = 2e-3
ATOL_BF16 = 1e-3
RTOL_BF16 = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def dev():
    return torch.device("cuda:0")


def T(a, dtype="fp16"):
    a = np.ascontiguousarray(a)
    if dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(a).to(dev())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


class Dev:
    def __init__(self, b: workloads.PagedBatch):
        self.b = b
        dt = b.dtype
        self.k_cache = T(b.k_cache, dt)
        self.v_cache = T(b.v_cache, dt)
        self.q = T(b.q, dt)
        self.bt = T(b.block_tables)
        self.cl = T(b.context_lens)
        api.pa_reshape_and_cache(T(b.key, dt), T(b.value, dt), self.k_cache, self.v_cache, T(b.slot_mapping))

    def decode(self):
        out = torch.empty_like(self.q)
        api.pa_decode(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, self.b.scale)
        return out

    def splitk(self, ps):
        b = self.b
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev())
        ws.fill_(float("nan"))
        out = torch.empty_like(self.q)
        api.pa_decode_splitk(out, self.q, self.k_cache, self.v_cache, self.bt, self.cl, b.scale, ps, ws, P)
        api.pa_splitk_reduce(out, ws, self.cl, b.max_blocks_per_seq, b.block_size, ps, P)
        return out


def oracle_out(b, seqs=None):
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    idx = np.arange(b.num_seqs) if seqs is None else np.asarray(seqs)
    return c_oracle.decode(b.q[idx], kc, vc, b.block_tables[idx], b.context_lens[idx], b.scale,
                           dtype=b.dtype)


def check(gpu: torch.Tensor, ref: np.ndarray, dtype: str):
    g = to_f64(gpu)
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    if dtype == "bf16":
        assert np.all(err <= ATOL_BF16 + RTOL_BF16 * np.abs(ref)), float(err.max())
    else:
        assert float(err.max()) <= TOL_F16


def _bf16(name, **kw):
    return workloads.build_batch(name=name, dtype="bf16", **kw)


BF16 = {
    "llama3-8b-s6": lambda: workloads.build_batch(
        name="l3", seed=3, context_lens=[1, 130, 777, 2048, 15, 1031], num_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, max_blocks_per_seq=128, dtype="bf16"),
    "70b-b32": lambda: _bf16("g8", seed=4, context_lens=[3001, 64], num_heads=64, num_kv_heads=8,
                             head_dim=128, block_size=32),
    "mha-d64": lambda: _bf16("d64", seed=5, context_lens=[5, 64, 65, 700], num_heads=6, num_kv_heads=6,
                             head_dim=64, block_size=64),
    "gqa16-d128": lambda: _bf16("g16", seed=6, context_lens=[300, 513, 1], num_heads=32, num_kv_heads=2,
                                head_dim=128, block_size=16),
}

HD256 = {
    "mha": dict(context_lens=[1, 40, 600], num_heads=4, num_kv_heads=4),
    "gqa4": dict(context_lens=[17, 1000, 2500], num_heads=16, num_kv_heads=4),
    "gqa8": dict(context_lens=[333, 4096], num_heads=16, num_kv_heads=2),
}


@pytest.mark.parametrize("name", list(BF16))
def test_bf16_cache_write_is_bit_exact(name):
    b = BF16[name]()
    d = Dev(b)
    ref_k, ref_v = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    torch.cuda.synchronize()
    assert np.array_equal(d.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), ref_k)
    assert np.array_equal(d.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), ref_v)


@pytest.mark.parametrize("name", list(BF16))
def test_bf16_decode_matches_oracle(name):
    b = BF16[name]()
    ref = oracle_out(b)
    d = Dev(b)
    check(d.decode(), ref, "bf16")
    for ps in (b.block_size, 8 * b.block_size, 512):
        if ps % b.block_size == 0:
            check(d.splitk(ps), ref, "bf16")


def test_bf16_single_token_returns_v_exactly():
    b = BF16["llama3-8b-s6"]()
    d = Dev(b)
    assert b.context_lens[0] == 1
    out = d.decode().view(torch.int16).cpu().numpy()
    vc = d.v_cache.view(torch.int16).cpu().numpy()
    blk = b.block_tables[0, 0]
    for h in range(b.num_heads):
        assert np.array_equal(out[0, h], vc[blk, 0, h // b.group_size])


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("shape", list(HD256))
def test_head_dim_256_matches_oracle(dtype, shape):
    b = workloads.build_batch(name="d256", seed=9, head_dim=256, block_size=16, dtype=dtype, **HD256[shape])
    ref = oracle_out(b)
    d = Dev(b)
    check(d.decode(), ref, dtype)
    check(d.splitk(256), ref, dtype)
    check(d.splitk(1024), ref, dtype)


def test_bf16_full_size_llama3_8b_every_sequence():
    b = workloads.llama3_8b(dtype="bf16")
    d = Dev(b)
    ref = oracle_out(b)
    check(d.decode(), ref, "bf16")
    check(d.splitk(512), ref, "bf16")
