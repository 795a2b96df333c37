"""bench.time_path on a fake torch: what the timed region holds.

The fake records every event record and kernel launch in the order the GPU
would see them, whether enqueued eagerly or replayed from a captured graph.
The timed region (between the first two events created with plain
``enable_timing``, recorded around the replays) must hold exactly K plain
steps of the path's kernels and no other event; the per-kernel split must come
from a pass that runs after it.
"""
from __future__ import annotations

import contextlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeGPU:
    def __init__(self, external_events=True):
        self.stream_log = []  # what the GPU executes, in order
        self.sink = self.stream_log  # where enqueued work goes (a graph while capturing)
        self.events = []
        self.external_events = external_events


class FakeEvent:
    def __init__(self, gpu, external):
        self.gpu = gpu
        self.external = external
        self.id = len(gpu.events)
        self.pos = None
        gpu.events.append(self)

    def record(self):
        if self.gpu.sink is not self.gpu.stream_log and not self.external:
            raise RuntimeError("a plain event cannot be recorded during capture")
        self.gpu.sink.append(("event", self))

    def elapsed_time(self, other):
        assert self.pos is not None and other.pos is not None, "event was never executed"
        return float(other.pos - self.pos)


class FakeGraph:
    def __init__(self, gpu):
        self.gpu = gpu
        self.nodes = []

    def replay(self):
        for n in self.nodes:
            self.gpu.stream_log.append(n)


def make_fake_torch(gpu):
    class Cuda:
        @staticmethod
        def Event(enable_timing=True, external=False):
            if external and not gpu.external_events:
                raise TypeError("external events are not supported")
            return FakeEvent(gpu, external)

        @staticmethod
        def CUDAGraph():
            return FakeGraph(gpu)

        @staticmethod
        @contextlib.contextmanager
        def graph(g, stream=None):
            old = gpu.sink
            gpu.sink = g.nodes
            try:
                yield
            finally:
                gpu.sink = old

        @staticmethod
        @contextlib.contextmanager
        def stream(s):
            yield

        @staticmethod
        def synchronize(dev=None):
            # execution: give every event its position in the log
            for i, (kind, obj) in enumerate(gpu.stream_log):
                if kind == "event":
                    obj.pos = i

    class Torch:
        cuda = Cuda

    return Torch


def run(K, W=3, nrep=3, external=True, nkern=2):
    gpu = FakeGPU(external_events=external)
    torch = make_fake_torch(gpu)
    kernels = [(f"k{j}", (lambda j: lambda r: gpu.sink.append(("kernel", (j, r % nrep))))(j))
               for j in range(nkern)]
    ms, per, walls, mode, G = bench.time_path(torch, None, None, kernels, nrep, K, W)
    return gpu, ms, per, mode, G


def timed_region(gpu):
    # e0 / e1: the two plain events of the timed region, the first plain events created
    plain = [e for e in gpu.events if not e.external]
    e0, e1 = plain[0], plain[1]
    return e0, e1, gpu.stream_log[e0.pos + 1:e1.pos]


@pytest.mark.parametrize("K", [1, 5, 20, 24, 25, 1000])
@pytest.mark.parametrize("external", [True, False])
def test_timed_region_is_exactly_k_plain_steps(K, external):
    nrep, nkern = 3, 3
    gpu, ms, per, mode, G = run(K, nrep=nrep, external=external, nkern=nkern)
    e0, e1, region = timed_region(gpu)
    assert all(kind == "kernel" for kind, _ in region), "an event inside the timed region"
    assert len(region) == K * nkern
    # the steps run the kernels in order, on replicas that rotate step by step
    for i in range(K):
        step = region[i * nkern:(i + 1) * nkern]
        assert [j for _, (j, _) in step] == list(range(nkern))
        assert len({r for _, (_, r) in step}) == 1
    reps = [region[i * nkern][1][1] for i in range(K)]
    if K >= 8 * nrep:
        assert reps == [i % nrep for i in range(K)]
    # ms spans exactly the region (the fake clock counts log entries)
    assert ms == float(e1.pos - e0.pos)
    # the per-kernel pass comes after the timed region
    ev_pass = [i for i, (kind, e) in enumerate(gpu.stream_log) if kind == "event" and e not in (e0, e1)]
    assert ev_pass and min(ev_pass) > e1.pos
    assert len(per) == nkern
    assert "separate pass" in mode
    assert ("graph" in mode) == external


def test_warmup_runs_before_anything_is_timed():
    gpu, *_ = run(K=10, W=7, nrep=2, nkern=1)
    e0, _, _ = timed_region(gpu)
    before = [x for x in gpu.stream_log[:e0.pos] if x[0] == "kernel"]
    assert len(before) >= 7
