"""pa_decode_splitk_static: split-K decode for callers that cannot allocate.

Some callers own no device allocator: a serving runtime that has reserved
nearly all device memory for its KV-cache pool, or a host program that only
holds the tensors it passes through the C ABI.  This entry point keeps the
split-K partials in a fixed array inside the library instead of a caller
workspace.  The GPU test checks it against the workspace-based entry points
(pa_decode_splitk + pa_splitk_reduce) and against the oracle on two calls in
a row: the first leaves NaN partials in the array (a sequence that reads a
block id outside the pool), and the second, of another shape, runs over them.
The CPU tests check that invalid arguments are reported as such, and that a
batch too large for the array is rejected before anything is launched.

This file is named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest

from paged_kv_cache_173_gb300 import _lib, workloads

TOL = 2e-3  # the decode tolerance used by every parity test
SCRATCH_BYTES = 32 * 1024 * 1024


def test_static_scratch_rejects_a_batch_that_does_not_fit():
    from paged_kv_cache_173_gb300.build import build_library
    build_library()
    L = _lib.lib()
    A = 1 << 20  # never dereferenced: the size check comes first
    # 512 sequences x 64 heads x 16 partitions x 130 floats = 272 MB > 32 MiB
    st = L.pa_decode_splitk_static(A, A, A, A, A, 512, A, 512, 64, 8, 128, 16, 100000, 0.1, 0, 512, None)
    assert st == _lib.PA_ERR_UNSUPPORTED
    assert "static scratch" in _lib.last_error()
    need = L.pa_splitk_workspace_bytes(512, 64, 128, 16)
    assert need > SCRATCH_BYTES


def test_static_scratch_checks_arguments_before_the_size():
    from paged_kv_cache_173_gb300.build import build_library
    build_library()
    L = _lib.lib()
    A = 1 << 20
    # the same oversized batch with a partition size that is not a multiple of the block size
    st = L.pa_decode_splitk_static(A, A, A, A, A, 512, A, 512, 64, 8, 128, 16, 100000, 0.1, 0, 500, None)
    assert st == _lib.PA_ERR_INVALID_ARG
    assert "partition_size" in _lib.last_error()
    st = L.pa_decode_splitk_static(A, None, A, A, A, 512, A, 512, 64, 8, 128, 16, 100000, 0.1, 0, 512, None)
    assert st == _lib.PA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_entry_points_on_two_calls():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    from oracle import c_oracle
    from paged_kv_cache_173_gb300 import api

    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    # Call 1: sequence 0 reads a block id outside the pool, so its partition-0 rows in the
    # array become NaN (rows at the start of the array).  Call 2 has another shape whose
    # rows cover those: it must still read only what it wrote itself.
    b1 = workloads.llama3_8b(num_seqs=24, seed=3)
    b2 = workloads.llama2_70b(num_seqs=3, ctx=2500, block_size=32, seed=4)
    assert b1.context_lens[0] > 128  # several partitions of 128 tokens
    bt1 = b1.block_tables.copy()
    bt1[0, 0] = b1.num_blocks + 7
    for b, ps, bt, bad in ((b1, 128, bt1, [0]), (b2, 512, b2.block_tables, [])):
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        assert api.pa_splitk_workspace_bytes(b.num_seqs, b.num_heads, b.head_dim, P) <= SCRATCH_BYTES
        kc, vc = t(b.k_cache), t(b.v_cache)
        api.pa_reshape_and_cache(t(b.key), t(b.value), kc, vc, t(b.slot_mapping))
        q, btd, cl = t(b.q), t(bt), t(b.context_lens)

        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev)
        ref = torch.empty_like(q)
        api.pa_decode_splitk(ref, q, kc, vc, btd, cl, b.scale, ps, ws, P)
        api.pa_splitk_reduce(ref, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)

        out = torch.full_like(q, float("nan"))
        api.pa_decode_splitk_static(out, q, kc, vc, btd, cl, b.scale, ps)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        r = ref.float().cpu().numpy()
        good = [s for s in range(b.num_seqs) if s not in bad]
        assert np.isnan(o[bad]).all()
        assert np.isfinite(o[good]).all()
        assert float(np.max(np.abs(o[good] - r[good]))) <= TOL
        # and against the oracle
        okc, ovc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
        want = c_oracle.decode(b.q[good], okc, ovc, bt[good], b.context_lens[good], b.scale)
        assert float(np.max(np.abs(o[good].astype(np.float64) - want))) <= TOL
