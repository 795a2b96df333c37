#!/usr/bin/env python
"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of one layer for a whole batch: reshape_and_cache
(the new token of every sequence into its slot), then paged decode, either as
one pa_decode launch (which merges partial results across the CTAs of a
cluster itself) or as pa_decode_splitk followed by the log-sum-exp reduce.
Both are timed; the faster is the headline and both appear under "paths".  Default workload: the Llama-3-8B-shaped decode layer
(64 sequences, 32 q heads / 8 KV heads, head_dim 128, block_size 16,
contexts uniform in [128, 2048], 1.25x pool with shuffled block ids).

Prints one JSON line.  ``value`` is KV-read GB/s: the algorithmic KV bytes of
a step (sum over sequences of ctx * K+V bytes per token) times the steps,
divided by the device time of the K steps.  The inputs sit in HBM before the
timed region; the KV pools rotate over replicas whose total is far larger
than L2, so no step reads KV bytes that an earlier step left in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the float64 CPU oracle on the host cores on the
same workload (a bounded sample of sequences per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s (% of GB300 HBM peak) and decode tokens/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # the vendor's nominal HBM3e bandwidth of one GB300, for context
# full-size configurations timed after the headline, each as its own entry of "configs"
DEFAULT_CONFIGS = "llama2-70b-b16,llama2-70b-b32,long-context"
CSRC = os.path.join(ROOT, "paged_kv_cache_173_gb300", "csrc")
# ncu DRAM traffic records (JSON): each names the kernel sources whose hash it was taken on
DECODE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_traffic.json")
PREFILL_TRAFFIC = os.path.join(ROOT, "profiles", "prefill_traffic.json")


# ----------------------------------------------------------------- workload
def make_workload(name: str, seed: int, partition_size: int, dtype: str = "fp16", kv_dtype: str = "",
                  draw_pools: bool = True):
    from paged_kv_cache_173_gb300 import workloads
    kw = dict(seed=seed, poison=False, partition_size=partition_size, dtype=dtype, kv_dtype=kv_dtype)
    big = {} if draw_pools else {"draw_pools": False}  # only the presets with large pools take it
    if name == "llama3-8b":
        b = workloads.llama3_8b(**kw)
        desc = ("llama3-8b decode layer: S=64, H=32, Hk=8, d=128, B=16, ctx~U[128,2048], "
                "1.25x pool, shuffled ids, 1 new token/seq")
    elif name in ("llama2-70b-b16", "llama2-70b-b32"):
        bs = int(name[-2:])
        b = workloads.llama2_70b(block_size=bs, **kw, **big)
        desc = f"llama2-70b GQA decode: S=32, H=64, Hk=8, d=128, B={bs}, ctx=8192, 1.25x pool, shuffled"
    elif name == "long-context":
        b = workloads.long_context(**kw, **big)
        desc = "long-context decode: S=4, ctx {32K,64K,96K,128K}, H=32, Hk=8, d=128, B=16"
    elif name == "shared-prefix":
        b = workloads.shared_prefix(**kw)
        desc = "shared-prefix sampling: 16 prompts x 8 samples, prompt 1024, suffix U[0,512], MHA 40, d=128"
    elif name == "head-dim-256":
        rng = np.random.default_rng(seed)
        b = workloads.build_batch(name=name, rng=rng, context_lens=rng.integers(128, 4097, size=32),
                                  num_heads=16, num_kv_heads=4, head_dim=256, block_size=16,
                                  max_blocks_per_seq=256, **kw)
        desc = "head_dim 256 GQA decode: S=32, H=16, Hk=4, d=256, B=16, ctx~U[128,4096], 1.25x pool"
    else:
        raise SystemExit(f"unknown workload {name}")
    if dtype != "fp16":
        desc += f", {dtype}"
    if kv_dtype == "fp8":
        desc += f", E4M3 KV cache (k_scale = v_scale = {b.k_scale:g})"
    return b, desc


def workload_key(args) -> str:
    """Name of the workload and element types, as the traffic records key it."""
    key = args.workload
    if args.dtype != "fp16":
        key += f"-{args.dtype}"
    if args.kv_dtype == "fp8":
        key += "-fp8kv"
    return key


def kv_ops(api, b):
    """The cache write, decode and split-K calls for the batch's cache type."""
    if b.kv_dtype == "fp8":
        ks, vs = b.k_scale, b.v_scale
        return (lambda key, value, kc, vc, sm: api.pa_reshape_and_cache_fp8(key, value, kc, vc, sm, ks, vs),
                lambda out, q, kc, vc, bt, cl: api.pa_decode_fp8(out, q, kc, vc, bt, cl, b.scale, ks, vs),
                lambda out, q, kc, vc, bt, cl, ps, ws, P: api.pa_decode_splitk_fp8(
                    out, q, kc, vc, bt, cl, b.scale, ks, vs, ps, ws, P))
    return (api.pa_reshape_and_cache,
            lambda out, q, kc, vc, bt, cl: api.pa_decode(out, q, kc, vc, bt, cl, b.scale),
            lambda out, q, kc, vc, bt, cl, ps, ws, P: api.pa_decode_splitk(out, q, kc, vc, bt, cl, b.scale,
                                                                           ps, ws, P))


def append_ops(api, b):
    """The fused cache write + decode calls (single pass, split-K) for the batch's cache type."""
    ks, vs = b.k_scale, b.v_scale
    return (lambda out, q, key, value, kc, vc, bt, cl: api.pa_append_and_decode(
                out, q, key, value, kc, vc, bt, cl, b.scale, k_scale=ks, v_scale=vs),
            lambda out, q, key, value, kc, vc, bt, cl, ps, ws, P: api.pa_append_and_decode_splitk(
                out, q, key, value, kc, vc, bt, cl, b.scale, ps, ws, P, k_scale=ks, v_scale=vs))


# kernel launches per step of each path (a call may launch more than one)
LAUNCHES_PER_STEP = {"decode": 2, "splitk": 3, "append": 1, "append_splitk": 2, "prefix": 4}


def decode_index(kernels) -> int:
    """Position of the decode launch in a path's kernel list."""
    return next(i for i, (n, _) in enumerate(kernels) if "decode" in n)


def to_device(a: np.ndarray, dtype: str, dev):
    """A workload array on the device; bfloat16 bit patterns become bf16 tensors."""
    import torch
    a = np.ascontiguousarray(a)
    if dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha(sources) -> str:
    """sha256 of the kernel sources, in order, first 16 hex digits."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str, kernel: str, record: str = DECODE_TRAFFIC):
    """ncu DRAM bytes (read + write) per launch from a JSON record, if they
    were taken on the current kernel sources for this workload and kernel;
    None otherwise."""
    try:
        with open(record) as f:
            rec = json.load(f)
        if rec.get("source_sha") != source_sha(rec["sources"]):
            return None
    except (OSError, ValueError, KeyError, TypeError):
        return None
    return rec.get("per_workload", {}).get(f"{workload}/{kernel}")


# ----------------------------------------------------------- multi-rank
def max_over_ranks(value: float, device) -> float:
    """The largest value over all ranks of the default process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(kv_bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Weak scaling: every rank decodes its own batch of the same shape, so the
    job moves world * steps * kv_bytes in the slowest rank's time."""
    return kv_bytes_per_rank_step * steps * world / (max_ms * 1e-3) / 1e9


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first samples arrive before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.05]
        if not rows and self.lines:
            # the region was shorter than the sampling period: take the nearest sample
            rows = [min(self.lines, key=lambda x: abs(x[0] - (t0 + t1) / 2))[1]]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- GPU arm
def _make_event(torch, external: bool):
    if external:
        return torch.cuda.Event(enable_timing=True, external=True)
    return torch.cuda.Event(enable_timing=True)


def time_path(torch, dev, stream, kernels, nrep: int, K: int, W: int, clocks=None, dist=None):
    """Time exactly K steps of one path; a step calls each of `kernels`
    (name, fn(r)) in order on replica r % nrep.

    The timed region holds the path's own launches and nothing else: CUDA-graph
    replays of plain steps (a graph of G steps replayed K // G times, then a
    graph of the K % G remaining steps), bracketed by two events.  The
    per-kernel split comes from a separate pass after the timed region: G
    more steps with an event between kernels, recorded inside a graph when
    torch supports external events, else enqueued eagerly.  Event nodes keep
    the launches of that pass from overlapping, so its durations are upper
    bounds.  Returns (ms of the K timed steps, per-kernel mean ms of the
    separate pass, wall-clock bounds of the timed region, how the split was
    taken, G)."""
    G = min(K, 8 * nrep)  # a multiple of nrep whenever K >= 8 * nrep
    n_full, tail = divmod(K, G)

    def step(r, ev=None):
        for j, (_, fn) in enumerate(kernels):
            if ev is not None:
                ev[j].record()
            fn(r)
        if ev is not None:
            ev[len(kernels)].record()

    with torch.cuda.stream(stream):
        for i in range(max(W, 3)):  # warm-up; also sets kernel attributes before any capture
            step(i)
    torch.cuda.synchronize(dev)

    def capture(n, evs=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i, evs[i] if evs is not None else None)
        return g

    g_full = capture(G) if n_full else None
    g_tail = capture(tail) if tail else None
    with torch.cuda.stream(stream):  # untimed rehearsal of every graph
        if g_full is not None:
            g_full.replay()
        if g_tail is not None:
            g_tail.replay()
    torch.cuda.synchronize(dev)

    # ---- the timed region: K plain steps
    if clocks:
        clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(n_full):
            g_full.replay()
        if g_tail is not None:
            g_tail.replay()
        e1.record()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    wall1 = time.time()
    if clocks:
        clocks.stop()
    ms = e0.elapsed_time(e1)

    # ---- the per-kernel split: a separate pass of G steps with events
    mode = "separate pass after the timed region, events inside a graph"
    try:
        evs = [[_make_event(torch, True) for _ in range(len(kernels) + 1)] for _ in range(G)]
        g_ev = capture(G, evs)
        with torch.cuda.stream(stream):
            g_ev.replay()  # first replay uploads the graph
            g_ev.replay()
        torch.cuda.synchronize(dev)
        evs[0][0].elapsed_time(evs[0][1])
    except Exception:
        mode = "separate pass after the timed region, eager events"
        evs = [[_make_event(torch, False) for _ in range(len(kernels) + 1)] for _ in range(G)]
        with torch.cuda.stream(stream):
            for i in range(G):
                step(i, evs[i])
        torch.cuda.synchronize(dev)
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(len(kernels))] for i in range(G)])
    return ms, per.mean(axis=0), (wall0, wall1), mode, G


def device_pools(torch, b, dev, seed: int):
    """K and V pools of the batch's shape filled on the device: standard
    normal float32 draws (torch's generator, seeded) rounded to the pool's
    element type; E4M3 pools hold the codes of N(0,1) / k_scale as the host
    recipe does."""
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    pools = []
    for _ in range(2):
        x = torch.randn(b.k_cache.shape, generator=g, device=dev, dtype=torch.float32)
        if b.kv_dtype == "fp8":
            pools.append((x / b.k_scale).to(torch.float8_e4m3fn).view(torch.uint8))
        else:
            pools.append(x.to(torch.bfloat16 if b.dtype == "bf16" else torch.float16))
        del x
    return pools


def other_bytes(b, path: str) -> dict:
    """Bytes a step moves besides the KV reads, by kind: the queries read and
    the outputs written, the block-table entries and context lengths read, the
    new tokens' K/V read and written into the pools (with their slots), and,
    for the split-K and shared-prefix paths, the float32 partial rows written
    by the decode and read by the reduce."""
    S, H, d, B = b.num_seqs, b.num_heads, b.head_dim, b.block_size
    qe = 2
    kve = 1 if b.kv_dtype == "fp8" else 2
    ctx = b.context_lens.astype(np.int64)
    T = b.num_tokens
    r = {
        "q": S * H * d * qe,
        "out": S * H * d * qe,
        "block_tables": int(np.sum((ctx + B - 1) // B)) * 4,
        "context_lens": S * 4,
        # read from the inputs and written into the pools; separate writes also read the slot ids
        "new_tokens": T * b.num_kv_heads * d * (2 * qe + 2 * kve) + (0 if path.startswith("append") else T * 8),
        "splitk_partials": 0,
    }
    if path in ("splitk", "prefix", "append_splitk"):
        nparts = (ctx + b.partition_size - 1) // b.partition_size
        rows = int(np.sum(np.where(nparts > 1, nparts, 0))) * H
        r["splitk_partials"] = 2 * rows * (d + 2) * 4
    return r


def measure_workload(args, name: str, dev, world: int, dist_g, host_pools: bool = True):
    """Time every decode path of one workload (each K steps, as time_path
    does) and return the batch, the device buffers and the per-path results.
    host_pools=False draws the pools on the device (device_pools)."""
    import torch
    from paged_kv_cache_173_gb300 import api, workloads

    rank = int(os.environ.get("RANK", "0"))
    b, desc = make_workload(name, args.seed + rank, args.partition_size, args.dtype, args.kv_dtype,
                            draw_pools=host_pools)
    kv_bytes = workloads.algorithmic_kv_bytes(b)
    write_kv, decode_kv, splitk_kv = kv_ops(api, b)
    ps = b.partition_size
    P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)

    t = lambda a: to_device(a, b.dtype, dev)  # noqa: E731
    pool_bytes = 2 * b.k_cache.nbytes
    l2_bytes = 129 * 2 ** 20
    R = max(2, min(8, math.ceil(4 * l2_bytes / max(1, kv_bytes)) + 1))
    if host_pools:
        k0, v0 = t(b.k_cache), t(b.v_cache)
    else:
        k0, v0 = device_pools(torch, b, dev, args.seed + 7919 * (rank + 1))
    q0 = t(b.q)
    reps = [(k0.clone(), v0.clone(), q0.clone()) if r else (k0, v0, q0) for r in range(R)]
    key, value, sm = t(b.key), t(b.value), t(b.slot_mapping)
    bt, cl = t(b.block_tables), t(b.context_lens)
    out = torch.empty_like(q0)
    ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev)
    M, B = b.max_blocks_per_seq, b.block_size

    def reshape(r):
        kc, vc, _ = reps[r % R]
        write_kv(key, value, kc, vc, sm)

    def decode(r):
        kc, vc, q = reps[r % R]
        decode_kv(out, q, kc, vc, bt, cl)

    def decode_splitk(r):
        kc, vc, q = reps[r % R]
        splitk_kv(out, q, kc, vc, bt, cl, ps, ws, P)

    def reduce(r):
        api.pa_splitk_reduce(out, ws, cl, M, B, ps, P)

    append_kv, append_splitk_kv = append_ops(api, b)

    def append(r):
        kc, vc, q = reps[r % R]
        append_kv(out, q, key, value, kc, vc, bt, cl)

    def append_splitk(r):
        kc, vc, q = reps[r % R]
        append_splitk_kv(out, q, key, value, kc, vc, bt, cl, ps, ws, P)

    paths = {
        "decode": [("reshape_and_cache", reshape), ("paged_decode", decode)],
        "splitk": [("reshape_and_cache", reshape), ("paged_decode_splitk", decode_splitk),
                   ("splitk_reduce", reduce)],
        # the cache write fused into the decode launch
        "append": [("append_and_decode", append)],
        "append_splitk": [("append_and_decode_splitk", append_splitk), ("splitk_reduce", reduce)],
    }
    if b.prefix_lens is not None:  # sequences share prompt blocks in consecutive groups
        plens = t(b.prefix_lens)

        def decode_prefix(r):
            kc, vc, q = reps[r % R]
            api.pa_decode_prefix_splitk(out, q, kc, vc, bt, cl, b.scale, b.seqs_per_group, plens, ps, ws, P,
                                        k_scale=b.k_scale, v_scale=b.v_scale)

        paths["prefix"] = [("reshape_and_cache", reshape), ("paged_decode_prefix", decode_prefix),
                           ("splitk_reduce", reduce)]
    if args.path not in ("auto", *paths):
        raise SystemExit(f"--path {args.path} needs a workload with shared-prefix groups")
    want = list(paths) if args.path == "auto" else [args.path]
    stream = torch.cuda.Stream(dev)
    results = {}
    for pname in want:
        clocks = ClockSampler(dev.index)
        ms, per, walls, mode, G = time_path(torch, dev, stream, paths[pname], R, args.steps, args.warmup, clocks,
                                            dist_g)
        if dist_g is not None:
            ms = max_over_ranks(ms, dev)
        results[pname] = dict(ms=ms, per=per, clocks=clocks.summary(*walls), mode=mode, G=G)
    best = min(results, key=lambda n: results[n]["ms"])  # chosen on the plain timed steps
    return dict(b=b, desc=desc, kv_bytes=kv_bytes, paths=paths, results=results, best=best, R=R,
                pool_bytes=pool_bytes, reps=reps, ws=ws, P=P, stream=stream)


def summarize(m, world: int, K: int, peak: float) -> dict:
    """The per-path figures of one measured workload: step time, whole-job
    GB/s, fractions of the copy bandwidth for the step and for the decode
    launch (its algorithmic bytes over its separate-pass event time)."""
    from paged_kv_cache_173_gb300 import workloads
    b, kv_bytes = m["b"], m["kv_bytes"]
    out = {}
    for pname, v in m["results"].items():
        roof = workloads.unique_kv_bytes(b) if pname == "prefix" else kv_bytes
        t_dec = float(v["per"][decode_index(m["paths"][pname])])
        if len(m["paths"][pname]) == 1:  # one launch per step: the timed region's average
            t_dec = v["ms"] / K
        val = whole_job_gbs(kv_bytes, K, world, v["ms"])
        out[pname] = {
            "ms_per_step": round(v["ms"] / K, 5),
            "value": round(val, 1),
            "step_frac": round(val / world / peak, 4),
            "kernel_ms": {kn: round(float(x), 5) for (kn, _), x in zip(m["paths"][pname], v["per"])},
            "kernel_frac": round(roof / (t_dec * 1e-3) / 1e9 / peak, 4),
        }
    return out


def run_gpu(args, rank: int, world: int):
    import torch
    from paged_kv_cache_173_gb300 import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    import torch.distributed as dist
    dist_g = dist if (world > 1 and dist.is_initialized()) else None
    K, W = args.steps, args.warmup
    peak, peak_kind = load_peak()

    m = measure_workload(args, args.workload, dev, world, dist_g, host_pools=True)
    b, kv_bytes, best = m["b"], m["kv_bytes"], m["best"]
    r0 = m["results"][best]
    kern = m["paths"][best]
    di = decode_index(kern)
    decode_name = kern[di][0]
    t_decode = float(r0["per"][di])

    e2e = run_e2e(args, b, dev, m["reps"], m["ws"], m["P"], kv_bytes, m["stream"], best)

    ms = r0["ms"]
    value = whole_job_gbs(kv_bytes, K, world, ms)
    step_ms = ms / K
    # the shared-prefix path reads each shared block once: its algorithmic
    # bytes are the unique bytes
    roof_bytes = workloads.unique_kv_bytes(b) if best == "prefix" else kv_bytes
    # The decode launch's average duration: on a one-kernel step the timed
    # region holds K launches of it and nothing else, so it is the region's
    # time over K; otherwise its time in the separate event pass.
    one_kernel = len(kern) == 1
    t_roof = step_ms if one_kernel else t_decode
    achieved = roof_bytes / (t_roof * 1e-3) / 1e9
    traffic = load_traffic(workload_key(args), decode_name)
    ob = other_bytes(b, best)
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if b.dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": {
            "workload": m["desc"],
            "kv_cache": "e4m3, one float scale per pool" if b.kv_dtype == "fp8" else b.dtype,
            "kv_bytes_per_step": kv_bytes,
            "path": best,
            "path_chosen_on": "the plain timed steps of each path",
            "step": " -> ".join(n for n, _ in kern),
            "partition_size": b.partition_size if best in ("splitk", "prefix", "append_splitk") else None,
            "roofline_bytes": ("unique KV bytes (each shared block once)" if best == "prefix"
                               else "algorithmic KV bytes"),
            "l2": (f"{m['R']} rotating pool replicas ({m['R'] * m['pool_bytes'] / 1e9:.2f} GB) > 129 MB L2; "
                   "steps back to back"),
            "timed_region": f"{K} plain steps as CUDA-graph replays, no events inside",
            "steps_per_graph": r0["G"],
            "kernel_timing": r0["mode"],
        },
        "hbm_frac_of_step": round(value / world / peak, 4),
        "hbm_peak_gbs": peak,
        "hbm_peak_kind": peak_kind,
        "hbm_frac_of_nominal": round(value / world / NOMINAL_HBM_GBS, 4),
        "nominal_hbm_gbs": NOMINAL_HBM_GBS,
        "tokens_per_s": round(b.num_seqs * world / (step_ms * 1e-3), 1),
        "other_bytes_per_step": ob,
        "other_bytes_frac_of_kv": round(sum(ob.values()) / kv_bytes, 5),
        "kernel_ms": {n: round(float(v), 5) for (n, _), v in zip(kern, r0["per"])},
        "roofline": {
            "kernel": decode_name,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_kind": f"{peak_kind} (copy GB/s)",
            "duration_ms": round(t_roof, 5),
            "duration_from": ("the timed region: K launches, one per step, nothing else" if one_kernel
                              else "the separate event pass (launches kept from overlapping)"),
            "isolated_frac": round(roof_bytes / (t_decode * 1e-3) / 1e9 / peak, 4),
        },
        "gpu_launches": LAUNCHES_PER_STEP[best] * K,
        "e2e": e2e,
        "clocks": r0["clocks"],
        "paths": summarize(m, world, K, peak),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(b, kv_bytes, budget_s=args.cpu_seconds)
    del m
    torch.cuda.empty_cache()

    # the other full-size configurations, each timed the same way
    names = [] if args.configs == "none" else [c for c in args.configs.split(",") if c and c != args.workload]
    if names:
        res["configs"] = {}
        launches = 0
        for name in names:
            mc = measure_workload(args, name, dev, world, dist_g, host_pools=False)
            per_path = summarize(mc, world, K, peak)
            bp = mc["best"]
            entry = {"workload": mc["desc"], "kv_bytes_per_step": mc["kv_bytes"], "path": bp,
                     "partition_size": mc["b"].partition_size if bp in ("splitk", "prefix", "append_splitk") else None,
                     "values": "pools drawn on the device (torch generator, N(0,1))",
                     "clocks": mc["results"][bp]["clocks"], **per_path[bp],
                     "tokens_per_s": round(mc["b"].num_seqs * world / (mc["results"][bp]["ms"] / K * 1e-3), 1),
                     "paths": per_path}
            launches += LAUNCHES_PER_STEP[bp] * K
            res["configs"][name] = entry
            del mc
            torch.cuda.empty_cache()
        res["configs_gpu_launches"] = launches
    return res


class StagedInputs:
    """A step's host inputs packed in one pinned buffer (each tensor at a 256-byte-aligned
    offset) and sent with one host-to-device copy; `dev` holds typed views of the device copy,
    which the library calls take like any other device tensors."""

    ALIGN = 256

    def __init__(self, host: dict, dev):
        import torch
        offs, n = {}, 0
        for k, t in host.items():
            offs[k] = n
            n += -(-t.numel() * t.element_size() // self.ALIGN) * self.ALIGN
        self.host = torch.zeros(max(n, self.ALIGN), dtype=torch.uint8).pin_memory()
        self.buf = torch.empty_like(self.host, device=dev)
        self.dev = {}
        for k, t in host.items():
            nb = t.numel() * t.element_size()
            self.host[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.dev[k] = self.buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        self.nbytes = self.host.numel()

    def send(self):
        self.buf.copy_(self.host, non_blocking=True)


def run_e2e(args, b, dev, reps, ws, P, kv_bytes, stream, path):
    """The same step through the public API with pinned host inputs and output,
    pipelined the way a serving loop runs it: step i + 1's inputs go to the
    device on one copy stream while step i computes, and step i's output comes
    back on another.  Inputs and outputs are double-buffered; a step's
    kernels wait for its inputs, and a buffer is refilled only after the step
    that used it is done (and, for the output, read back).  Every step copies
    all of its inputs in (one pinned buffer, one copy) and its output out.
    The timed region runs from before the first input copy to after the last
    output copy."""
    import torch
    from paged_kv_cache_173_gb300 import api

    names = ["q", "key", "value", "block_tables", "context_lens"]
    if not path.startswith("append"):
        names.append("slot_mapping")
    host = {k: to_device(getattr(b, k), b.dtype, "cpu") for k in names}
    if path == "prefix":
        host["prefix_lens"] = torch.from_numpy(b.prefix_lens)
    staged = [StagedInputs(host, dev) for _ in range(2)]
    outs = [torch.empty_like(staged[0].dev["q"]) for _ in range(2)]
    outs_h = [torch.empty_like(host["q"]).pin_memory() for _ in range(2)]
    h2d = staged[0].nbytes
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    M, B, ps, R = b.max_blocks_per_seq, b.block_size, b.partition_size, len(reps)
    write_kv, decode_kv, splitk_kv = kv_ops(api, b)
    append_kv, append_splitk_kv = append_ops(api, b)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inputs_ready = [ev(), ev()]
    computed = [ev(), ev()]
    read_back = [ev(), ev()]

    def kernels(i, devb, out):
        kc, vc, _ = reps[i % R]
        q, bt, cl = devb["q"], devb["block_tables"], devb["context_lens"]
        if path == "append":
            append_kv(out, q, devb["key"], devb["value"], kc, vc, bt, cl)
            return
        if path == "append_splitk":
            append_splitk_kv(out, q, devb["key"], devb["value"], kc, vc, bt, cl, ps, ws, P)
            api.pa_splitk_reduce(out, ws, cl, M, B, ps, P)
            return
        write_kv(devb["key"], devb["value"], kc, vc, devb["slot_mapping"])
        if path == "decode":
            decode_kv(out, q, kc, vc, bt, cl)
        elif path == "prefix":
            api.pa_decode_prefix_splitk(out, q, kc, vc, bt, cl, b.scale, b.seqs_per_group, devb["prefix_lens"], ps,
                                        ws, P, k_scale=b.k_scale, v_scale=b.v_scale)
            api.pa_splitk_reduce(out, ws, cl, M, B, ps, P)
        else:
            splitk_kv(out, q, kc, vc, bt, cl, ps, ws, P)
            api.pa_splitk_reduce(out, ws, cl, M, B, ps, P)

    def send(i, first=None):
        j = i % 2
        with torch.cuda.stream(up):
            if first is not None:
                up.wait_event(first)
            if i >= 2:
                up.wait_event(computed[j])  # step i - 2 is done with these inputs
            staged[j].send()
            inputs_ready[j].record(up)

    def run(n, e_start=None):
        send(0, e_start)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                send(i + 1)
            stream.wait_event(inputs_ready[j])
            if i >= 2:
                stream.wait_event(read_back[j])  # step i - 2's output has been read back
            with torch.cuda.stream(stream):
                kernels(i, staged[j].dev, outs[j])
                computed[j].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[j])
                outs_h[j].copy_(outs[j], non_blocking=True)
                read_back[j].record(down)
        stream.wait_event(read_back[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(read_back[(n - 2) % 2])

    n = max(3, min(args.steps, args.e2e_steps))
    run(3)  # warm-up
    torch.cuda.synchronize(dev)

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            e0.record()
        t0 = time.perf_counter()
        steps = fn(e0)
        host_s = time.perf_counter() - t0
        with torch.cuda.stream(stream):
            e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1), steps, host_s

    # eager: the host enqueues every call and copy of every step
    ms_e, n_e, host_s = timed(lambda e0: (run(n, e0), n)[1])
    eager = {"value": round(kv_bytes * n_e / (ms_e * 1e-3) / 1e9, 1), "ms_per_step": round(ms_e / n_e, 5),
             "steps": n_e, "host_enqueue_us_per_step": round(host_s / n_e * 1e6, 2)}
    # the host cost of the step's library calls alone (Python binding, ctypes, argument
    # checks, launch), enqueued back to back with no copy and no event between them
    calls = min(n, 500)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for i in range(calls):
            kernels(i, staged[0].dev, outs[0])
        eager["host_us_per_step_calls_only"] = round((time.perf_counter() - t0) / calls * 1e6, 2)
    torch.cuda.synchronize(dev)
    res = {"unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "pipelining": "inputs of step i+1 copied in while step i computes; outputs copied out behind it",
           "eager": eager}
    # graph: the same calls and copies of G pipelined steps captured once and replayed, as a
    # serving loop replays its decode step (G a multiple of the replica and buffer rotations)
    G = min(n, 8 * R)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            start = torch.cuda.Event()
            start.record(stream)
            run(G, start)
        with torch.cuda.stream(stream):
            g.replay()  # the first replay uploads the graph
        torch.cuda.synchronize(dev)

        def replays(e0):
            stream.wait_event(e0)
            with torch.cuda.stream(stream):
                for _ in range(max(1, n // G)):
                    g.replay()
            return max(1, n // G) * G

        ms_g, n_g, _ = timed(replays)
        res.update({"value": round(kv_bytes * n_g / (ms_g * 1e-3) / 1e9, 1), "ms_per_step": round(ms_g / n_g, 5),
                    "steps": n_g, "mode": f"CUDA graph of {G} pipelined steps (copies included), replayed"})
    except Exception as exc:  # no capture: the eager figures are the e2e
        res.update({"value": eager["value"], "ms_per_step": eager["ms_per_step"], "steps": n_e,
                    "mode": f"eager (graph capture failed: {type(exc).__name__})"})
    return res


# ------------------------------------------------------------ copy_blocks
def run_copy_blocks(args):
    """Time pa_copy_blocks: K steps, each copying `--copy-pairs` whole blocks.
    The pools have the workload's block shape and element type, with enough
    blocks that the source half holds at least 4x the L2 of K and V; each
    cycle of steps walks a permutation of the source half (and of the
    destination half), so no block is read twice within a cycle.  Bytes =
    read + write of K and V."""
    import torch
    from paged_kv_cache_173_gb300 import api

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    b, desc = make_workload(args.workload, args.seed, args.partition_size, args.dtype, args.kv_dtype)
    shape = b.k_cache.shape[1:]
    block_bytes = int(np.prod(shape)) * b.k_cache.itemsize
    l2_bytes = 129 * 2 ** 20
    N = max(b.num_blocks, 2 * math.ceil(4 * l2_bytes / (2 * block_bytes)))
    dt = {1: torch.uint8, 2: torch.int16}[b.k_cache.itemsize]
    kc = torch.randint(-100, 100, (N, *shape), dtype=torch.int16, device=dev).to(dt)
    vc = torch.randint(-100, 100, (N, *shape), dtype=torch.int16, device=dev).to(dt)
    if dt == torch.int16:  # bit patterns of the workload's 16-bit type
        kc = kc.view(torch.bfloat16 if b.dtype == "bf16" else torch.float16)
        vc = vc.view(torch.bfloat16 if b.dtype == "bf16" else torch.float16)
    half = N // 2
    n = min(args.copy_pairs, half)
    rng = np.random.default_rng(args.seed)
    src_perm = rng.permutation(half)
    dst_perm = half + rng.permutation(N - half)
    sets = []
    for i in range(half // n):
        pairs = np.stack([src_perm[i * n:(i + 1) * n], dst_perm[i * n:(i + 1) * n]], axis=1)
        sets.append(torch.from_numpy(pairs.astype(np.int64)).to(dev))
    stream = torch.cuda.Stream(dev)
    kernels = [("copy_blocks", lambda r: api.pa_copy_blocks(kc, vc, sets[r % len(sets)]))]
    clocks = ClockSampler(dev.index)
    ms, per, walls, mode, G = time_path(torch, dev, stream, kernels, len(sets), args.steps, args.warmup, clocks)
    moved = 2 * 2 * n * block_bytes  # K and V, read and written
    peak, kind = load_peak()
    value = moved * args.steps / (ms * 1e-3) / 1e9
    return {"metric": "pa_copy_blocks GB/s (bytes read + written)", "value": round(value, 1), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "higher_is_better": True, "dtype": "u8" if b.kv_dtype == "fp8" else ("bf16" if b.dtype == "bf16" else "f16"),
            "data": "synthetic",
            "config": {"workload": desc, "pairs_per_step": n, "block_bytes": block_bytes, "pool_blocks": N,
                       "l2": f"one cycle of {len(sets)} steps reads {half * 2 * block_bytes / 1e9:.2f} GB of "
                             "distinct source blocks (> 4x the 129 MB L2)",
                       "kernel_timing": mode},
            "roofline": {"kernel": "copy_blocks", "bound": "hbm", "achieved": round(value, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                         "peak_kind": f"{kind} (copy GB/s)"},
            "gpu_launches": args.steps, "clocks": clocks.summary(*walls)}


# ---------------------------------------------------------------- prefill
PREFILL_WORKLOADS = {
    # name: (contexts, query lengths, H, Hk, d, B, description)
    "prefill-llama3-8b": ([2048] * 8, [2048] * 8, 32, 8, 128, 16,
                          "Llama-3-8B prompts: 8 x 2048 new tokens, H=32, Hk=8, d=128, B=16"),
    "chunked-prefill-llama3-8b": ([2048] * 16, [512] * 16, 32, 8, 128, 16,
                                  "Llama-3-8B chunked prefill: 16 sequences x (1536 cached + 512 new), B=16"),
    "prefill-long": ([16384] * 2, [16384] * 2, 32, 8, 128, 16,
                     "long prompts: 2 x 16384 new tokens, H=32, Hk=8, d=128, B=16"),
}


def run_prefill(args):
    """Time one prefill step: reshape_and_cache of every new token, then
    pa_prefill; FLOPs = 4 d H x (keys each query row attends to)."""
    import torch
    from paged_kv_cache_173_gb300 import api, workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    name = args.workload if args.workload in PREFILL_WORKLOADS else "prefill-llama3-8b"
    ctx, ql, H, Hk, d, B, desc = PREFILL_WORKLOADS[name]
    b = workloads.build_prefill_batch(name=name, seed=args.seed, context_lens=ctx, query_lens=ql, num_heads=H,
                                      num_kv_heads=Hk, head_dim=d, block_size=B, poison=False, dtype=args.dtype)
    flops = workloads.prefill_flops(b)
    t = lambda a: to_device(a, b.dtype, dev)  # noqa: E731
    l2_bytes = 129 * 2 ** 20
    pool_bytes = 2 * b.k_cache.nbytes
    R = max(2, min(4, math.ceil(2 * l2_bytes / pool_bytes) + 1))
    reps = [(t(b.k_cache), t(b.v_cache)) for _ in range(R)]
    q, key, value, sm = t(b.q), t(b.key), t(b.value), t(b.slot_mapping)
    bt, cl, qsl = t(b.block_tables), t(b.context_lens), t(b.query_start_loc)
    maxq = int(np.diff(b.query_start_loc).max())
    out = torch.empty_like(q)

    def reshape(r):
        kc, vc = reps[r % R]
        api.pa_reshape_and_cache(key, value, kc, vc, sm)

    def prefill(r):
        kc, vc = reps[r % R]
        api.pa_prefill(out, q, kc, vc, bt, cl, qsl, maxq, b.scale)

    kernels = [("reshape_and_cache", reshape), ("paged_prefill", prefill)]
    stream = torch.cuda.Stream(dev)
    clocks = ClockSampler(dev.index)
    K, W = args.steps, args.warmup
    ms, per, walls, mode, G = time_path(torch, dev, stream, kernels, R, K, W, clocks)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured cuBLAS bf16 burst"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    step_ms = ms / K
    value = flops * K / (ms * 1e-3) / 1e12
    achieved = flops / (float(per[1]) * 1e-3) / 1e12

    # e2e: the public calls with pinned host inputs and the output read back
    host = {k: to_device(getattr(b, k), b.dtype, "cpu")
            for k in ("q", "key", "value", "slot_mapping", "block_tables", "context_lens", "query_start_loc")}
    staged = StagedInputs(host, dev)
    devb = staged.dev
    out_h = torch.empty_like(host["q"]).pin_memory()

    def e2e_step(i):
        kc, vc = reps[i % R]
        staged.send()  # every input of the step, one copy
        api.pa_reshape_and_cache(devb["key"], devb["value"], kc, vc, devb["slot_mapping"])
        api.pa_prefill(out, devb["q"], kc, vc, devb["block_tables"], devb["context_lens"], devb["query_start_loc"],
                       maxq, b.scale)
        out_h.copy_(out, non_blocking=True)

    n = max(3, min(K, 50))
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            e2e_step(i)
        e1.record()
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / n
    res = {
        "metric": "paged prefill TFLOP/s (causal attention FLOPs)", "value": round(value, 1), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if b.dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": {"workload": desc, "flops_per_step": flops, "step": "reshape_and_cache -> paged_prefill",
                   "l2": f"{R} rotating pool replicas ({R * pool_bytes / 1e9:.2f} GB); steps back to back",
                   "steps_per_graph": G, "kernel_timing": mode},
        "kernel_ms": {n_: round(float(v), 4) for (n_, _), v in zip(kernels, per)},
        "roofline": {"kernel": "paged_prefill", "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": load_traffic(args.workload + ("-bf16" if b.dtype == "bf16" else ""), "paged_prefill",
                                             PREFILL_TRAFFIC),
                     "peak_kind": f"{peak_kind} (fp16 MMAs take the bf16 figure: the same nominal rate)"},
        "gpu_launches": 2 * K,
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(staged.nbytes),
                "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()), "steps": n,
                "ms_per_step": round(e2e_ms, 4)},
        "clocks": clocks.summary(*walls),
    }
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(b, budget_s=args.cpu_seconds)
    return res


def prefill_cpu_baseline(b, budget_s: float):
    """The oracle on the host cores: the first n rows of sequence 0 as a
    prompt of n tokens, n grown until the sample takes about budget_s / 3."""
    from oracle import c_oracle
    from paged_kv_cache_173_gb300 import workloads
    kc, vc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
    ql0 = int(b.query_start_loc[1])
    n, elapsed, done = 16, 0.0, 0
    while True:
        qsl = np.array([0, n], np.int32)
        t0 = time.perf_counter()
        c_oracle.prefill(b.q[:n], kc, vc, b.block_tables[:1], np.array([n], np.int32), qsl, b.scale, dtype=b.dtype)
        dt = time.perf_counter() - t0
        elapsed += dt
        done += 4 * b.head_dim * b.num_heads * (n * (n + 1) // 2)
        if elapsed > budget_s or n >= ql0:
            break
        n = min(ql0, n * 2)
    return {"value": round(done / elapsed / 1e12, 6), "unit": "TFLOP/s", "cores": c_oracle.max_threads(),
            "kind": "oracle", "sample": f"float64 C oracle prefill of the first 16..{n} rows of one prompt, "
                                        f"{elapsed:.1f} s, host {_cpu_model()}"}


# ------------------------------------------------------------ CPU oracle
def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def oracle_step_runner(b):
    """Returns (run(n_seqs, offset) -> kv_bytes, cores): one oracle decode step
    (reshape_and_cache + decode) over a cyclic sample of n_seqs sequences."""
    from oracle import c_oracle
    from paged_kv_cache_173_gb300 import workloads
    cores = c_oracle.max_threads()
    S = b.num_seqs
    per_tok = workloads.kv_bytes_per_token(b.num_kv_heads, b.head_dim, workloads.kv_elem_bytes(b))
    kc, vc = b.k_cache.copy(), b.v_cache.copy()  # working pools, written in place each step

    def run(n, off):
        idx = (np.arange(n) + off) % S
        if b.kv_dtype == "fp8":
            c_oracle.reshape_and_cache_fp8(b.key[idx], b.value[idx], kc, vc, b.slot_mapping[idx], b.k_scale,
                                           b.v_scale, dtype=b.dtype, inplace=True)
        else:
            c_oracle.reshape_and_cache(b.key[idx], b.value[idx], kc, vc, b.slot_mapping[idx], inplace=True)
        c_oracle.decode(b.q[idx], kc, vc, b.block_tables[idx], b.context_lens[idx], b.scale, dtype=b.dtype,
                        k_scale=b.k_scale, v_scale=b.v_scale)
        return int(np.sum(b.context_lens[idx].astype(np.int64))) * per_tok

    return run, cores


def cpu_baseline(b, kv_bytes, budget_s: float):
    run, cores = oracle_step_runner(b)
    t0 = time.perf_counter()
    nbytes = run(1, 0)
    one = time.perf_counter() - t0
    n = int(max(1, min(b.num_seqs, budget_s / max(one, 1e-6) / 3)))
    done, elapsed, off = 0, 0.0, 1
    while elapsed < budget_s:
        t0 = time.perf_counter()
        done += run(n, off)
        elapsed += time.perf_counter() - t0
        off += n
    return {"value": round(done / elapsed / 1e9, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"float64 C oracle (reshape_and_cache + decode), {n} of {b.num_seqs} sequences per "
                      f"call, {elapsed:.1f} s, {done / 1e9:.2f} GB of KV, host {_cpu_model()}"}


def run_reference(args, rank: int):
    if rank != 0:
        return None
    b, desc = make_workload(args.workload, args.seed, args.partition_size, args.dtype, args.kv_dtype)
    run, cores = oracle_step_runner(b)
    t0 = time.perf_counter()
    run(1, 0)
    one = time.perf_counter() - t0
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    n = int(max(1, min(b.num_seqs, budget / max(one, 1e-6))))
    off = 0
    for _ in range(args.warmup):
        run(n, off)
        off += n
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += run(n, off)
        off += n
    el = time.perf_counter() - t0
    value = done / el / 1e9
    sample = (f"float64 C oracle, {n} of {b.num_seqs} sequences per step (cycling), {args.steps} steps, "
              f"{el:.1f} s, host {_cpu_model()}")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": desc, "kv_bytes_per_step": done // max(1, args.steps)},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main
def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[1])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama3-8b")
    p.add_argument("--partition-size", type=int, default=512)
    p.add_argument("--dtype", choices=["fp16", "bf16"], default="fp16")
    p.add_argument("--kv-dtype", choices=["same", "fp8"], default="same",
                   help="fp8: E4M3 KV pools with one float scale each (float16 queries)")
    p.add_argument("--op", choices=["step", "copy-blocks", "prefill"], default="step",
                   help="step: the decode step (the headline); copy-blocks: time pa_copy_blocks; prefill: "
                        "reshape + pa_prefill on --workload prefill-llama3-8b, chunked-prefill-llama3-8b "
                        "or prefill-long")
    p.add_argument("--copy-pairs", type=int, default=1024)
    p.add_argument("--path", choices=["auto", "decode", "splitk", "append", "append_splitk", "prefix"],
                   default="auto",
                   help="decode: reshape + pa_decode; splitk: reshape + pa_decode_splitk + reduce; append: "
                        "pa_append_and_decode (the cache write fused in); append_splitk: "
                        "pa_append_and_decode_splitk + reduce; prefix (shared-prefix workload): reshape + "
                        "pa_decode_prefix_splitk + reduce; auto: time every path the workload has, report the "
                        "fastest")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--reference-seconds", type=float, default=90.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--configs", default=None,
                   help="comma-separated workloads timed after the headline, each in the line's "
                        f"\"configs\" object (default with the llama3-8b decode step: {DEFAULT_CONFIGS}; "
                        "'none' for none)")
    return p.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.kv_dtype == "same":
        args.kv_dtype = ""
    if args.kv_dtype == "fp8" and args.dtype != "fp16":
        raise SystemExit("--kv-dtype fp8 takes --dtype fp16")
    if args.warmup < 3:
        args.warmup = 3
    if args.configs is None:
        plain = args.workload == "llama3-8b" and args.dtype == "fp16" and not args.kv_dtype and args.path == "auto"
        args.configs = DEFAULT_CONFIGS if plain else "none"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    if args.op == "copy-blocks":
        print(json.dumps(run_copy_blocks(args)), flush=True)
        return 0
    if args.op == "prefill":
        print(json.dumps(run_prefill(args)), flush=True)
        return 0
    res = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
