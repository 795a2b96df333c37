"""Host logic of bench.py that needs no GPU: the staging of a step's inputs for the
end-to-end arm (one pinned buffer, 256-byte-aligned slots, typed views of the copy)."""
from __future__ import annotations

import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_173_gb300 import workloads  # noqa: E402


@pytest.fixture
def no_pinning(monkeypatch):
    # pinned host memory needs a CUDA context; the packing logic does not
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_staged_inputs_pack_every_tensor_bit_for_bit(no_pinning, dtype):
    b = workloads.llama3_8b(num_seqs=5, dtype=dtype)
    host = {k: bench.to_device(getattr(b, k), b.dtype, "cpu")
            for k in ("q", "key", "value", "slot_mapping", "block_tables", "context_lens")}
    st = bench.StagedInputs(host, "cpu")
    st.send()
    base = st.buf.data_ptr()
    for k, t in host.items():
        v = st.dev[k]
        assert v.dtype == t.dtype and v.shape == t.shape, k
        assert (v.data_ptr() - base) % bench.StagedInputs.ALIGN == 0, k
        assert torch.equal(v.contiguous().view(-1).view(torch.uint8), t.contiguous().view(-1).view(torch.uint8)), k
    payload = sum(t.numel() * t.element_size() for t in host.values())
    assert payload <= st.nbytes < payload + len(host) * bench.StagedInputs.ALIGN


def test_staged_inputs_slots_do_not_overlap(no_pinning):
    host = {"a": torch.arange(3, dtype=torch.int32), "b": torch.ones(257, dtype=torch.int64),
            "c": torch.zeros(1, dtype=torch.float16)}
    st = bench.StagedInputs(host, "cpu")
    st.send()
    spans = sorted((v.data_ptr(), v.data_ptr() + v.numel() * v.element_size()) for v in st.dev.values())
    for (s0, e0), (s1, _) in zip(spans, spans[1:]):
        assert e0 <= s1
    assert np.array_equal(st.dev["b"].numpy(), np.ones(257, dtype=np.int64))
