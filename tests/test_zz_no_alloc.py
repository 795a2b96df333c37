"""pa_decode_splitk_static: split-K decode for callers that cannot allocate.

Some callers own no device allocator: a serving runtime that has reserved
nearly all device memory for its KV-cache pool, or a host program that only
holds the tensors it passes through the C ABI.  This entry point keeps the
split-K partials in a fixed array inside the library instead of a caller
workspace.  The GPU test checks it against the workspace-based entry points
(pa_decode_splitk + pa_splitk_reduce) on two calls in a row: the second call
finds the first call's partials still in the array.  The CPU test checks that
a batch too large for the array is rejected before anything is launched.

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


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_entry_points_on_two_calls():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_173_gb300 import api

    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    # a larger batch first, then a smaller one with a different shape, so the
    # second call runs over the first call's stale partials
    batches = [(workloads.llama3_8b(num_seqs=24, seed=3), 256),
               (workloads.llama2_70b(num_seqs=3, ctx=2500, block_size=32, seed=4), 512)]
    for b, ps in batches:
        assert api.pa_splitk_workspace_bytes(
            b.num_seqs, b.num_heads, b.head_dim,
            api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)) <= SCRATCH_BYTES
        kc, vc = t(b.k_cache), t(b.v_cache)
        api.pa_reshape_and_cache(t(b.key), t(b.value), kc, vc, t(b.slot_mapping))
        q, bt, cl = t(b.q), t(b.block_tables), t(b.context_lens)

        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev)
        ref = torch.empty_like(q)
        api.pa_decode_splitk(ref, q, kc, vc, bt, cl, b.scale, ps, ws, P)
        api.pa_splitk_reduce(ref, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)

        out = torch.full_like(q, float("nan"))
        api.pa_decode_splitk_static(out, q, kc, vc, bt, cl, b.scale, ps)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        r = ref.float().cpu().numpy()
        assert np.isfinite(o).all()
        assert float(np.max(np.abs(o - r))) <= TOL
