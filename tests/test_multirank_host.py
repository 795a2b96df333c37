"""The N > 1 bench path on the CPU: two gloo ranks.

Each rank decodes its own batch (seed + rank, same shape), and the timing is
the maximum over ranks; the data path has no collective.  These tests run the
host logic that does this with world_size 2 on the gloo backend.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # the slower rank sets the job time
        got = bench.max_over_ranks(ms, torch.device("cpu"))
        b, _ = bench.make_workload("llama3-8b", seed=0 + rank, partition_size=512)
        digest = int(np.sum(b.context_lens))
        sizes = torch.tensor([digest, b.num_seqs, b.num_heads], dtype=torch.int64)
        gathered = [torch.zeros_like(sizes) for _ in range(world)]
        dist.all_gather(gathered, sizes)
        out.put((rank, got, [g.tolist() for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_distinct_batches():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gathered in res:
        assert got == 15.0
        (d0, s0, h0), (d1, s1, h1) = gathered
        assert (s0, h0) == (s1, h1) == (64, 32)  # same shape on every rank
        assert d0 != d1                          # but each rank has its own batch


def test_whole_job_throughput_is_weak_scaling():
    one = bench.whole_job_gbs(290_000_000, 100, 1, 5.0)
    two = bench.whole_job_gbs(290_000_000, 100, 2, 5.0)
    assert abs(two - 2 * one) < 1e-9
    assert abs(one - 290_000_000 * 100 / 5e-3 / 1e9) < 1e-9
