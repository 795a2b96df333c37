"""Failure detection on the GPU without a fault: every pipeline of the library waits on
mbarriers through one bounded wait, which gives up after its limit instead of spinning
(the kernels then write NaN rows).  pa_selftest_wait runs that wait on a phase that
nothing completes: it must give up after the limit, a completed phase must still be
seen, and the context must stay usable for the next call."""
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


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_a_wait_that_nothing_completes_gives_up_after_its_limit(limit_us):
    r = api.pa_selftest_wait(limit_us=limit_us)
    assert r["gave_up"], r
    assert r["completed"], r
    # the wait re-checks the clock after each suspend of at most 20 us
    assert limit_us <= r["waited_us"] < limit_us + 100_000, r


def test_the_context_stays_usable_after_a_wait_gave_up():
    api.pa_selftest_wait(limit_us=5000)
    dev = torch.device("cuda:0")
    b = workloads.tiny()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    kc, vc = t(b.k_cache), t(b.v_cache)
    api.pa_reshape_and_cache(t(b.key), t(b.value), kc, vc, t(b.slot_mapping))
    out = torch.empty_like(t(b.q))
    api.pa_decode(out, t(b.q), kc, vc, t(b.block_tables), t(b.context_lens), b.scale)
    torch.cuda.synchronize()
    rk, rv = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    ref = c_oracle.decode(b.q, rk, rv, b.block_tables, b.context_lens, b.scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 2e-3
