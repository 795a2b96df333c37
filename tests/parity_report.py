"""Max abs error of every decode entry point against the oracle, on the five
full-size workloads (a report, not a test: the parity tests assert the
bounds; this prints the errors they allow).

    python tests/parity_report.py [--kv-dtype fp8] > report.md

For each workload and entry point: the largest |GPU - oracle| over every
output element, and whether the pools after the cache write equal the
oracle's byte for byte.  Needs a GPU and the built library.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    p = argparse.ArgumentParser(description="decode max abs error against the oracle")
    p.add_argument("--kv-dtype", choices=["same", "fp8"], default="same")
    args = p.parse_args(argv)
    kv = "fp8" if args.kv_dtype == "fp8" else ""

    import torch

    import __graft_entry__
    from oracle import c_oracle
    from paged_kv_cache_173_gb300 import api, workloads

    __graft_entry__.build()
    dev = torch.device("cuda:0")
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    loads = {
        "tiny": lambda: workloads.build_batch(name="tiny", seed=0, context_lens=[1, 15, 16, 37], num_heads=4,
                                              num_kv_heads=4, head_dim=64, block_size=16, num_blocks=16,
                                              max_blocks_per_seq=3, partition_size=16, kv_dtype=kv),
        "llama3-8b": lambda: workloads.llama3_8b(kv_dtype=kv),
        "llama2-70b-b16": lambda: workloads.llama2_70b(block_size=16, kv_dtype=kv),
        "llama2-70b-b32": lambda: workloads.llama2_70b(block_size=32, kv_dtype=kv),
        "long-context": lambda: workloads.long_context(kv_dtype=kv),
        "shared-prefix": lambda: workloads.shared_prefix(kv_dtype=kv),
    }
    print("| workload | KV bytes | entry point | max abs err | pools bit-exact |")
    print("|---|---|---|---|---|")
    for name, make in loads.items():
        t0 = time.time()
        b = make()
        ps = b.partition_size
        ks, vs = b.k_scale, b.v_scale
        if kv == "fp8":
            okc, ovc = c_oracle.reshape_and_cache_fp8(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping, ks, vs)
        else:
            okc, ovc = c_oracle.reshape_and_cache(b.key, b.value, b.k_cache, b.v_cache, b.slot_mapping)
        ref = c_oracle.decode(b.q, okc, ovc, b.block_tables, b.context_lens, b.scale, k_scale=ks, v_scale=vs)
        q, bt, cl, sm = T(b.q), T(b.block_tables), T(b.context_lens), T(b.slot_mapping)
        P = api.max_num_partitions_for(b.max_blocks_per_seq, b.block_size, ps)
        ws = api.alloc_splitk_workspace(b.num_seqs, b.num_heads, b.head_dim, P, dev)

        def fresh():
            return T(b.k_cache), T(b.v_cache)

        def write(kc, vc):
            if kv == "fp8":
                api.pa_reshape_and_cache_fp8(T(b.key), T(b.value), kc, vc, sm, ks, vs)
            else:
                api.pa_reshape_and_cache(T(b.key), T(b.value), kc, vc, sm)

        def run(entry):
            kc, vc = fresh()
            out = torch.empty_like(q)
            if entry.startswith("pa_append"):
                if entry == "pa_append_and_decode":
                    api.pa_append_and_decode(out, q, T(b.key), T(b.value), kc, vc, bt, cl, b.scale, k_scale=ks,
                                             v_scale=vs)
                else:
                    api.pa_append_and_decode_splitk(out, q, T(b.key), T(b.value), kc, vc, bt, cl, b.scale, ps, ws,
                                                    P, k_scale=ks, v_scale=vs)
                    api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
            else:
                write(kc, vc)
                if entry == "pa_decode":
                    if kv == "fp8":
                        api.pa_decode_fp8(out, q, kc, vc, bt, cl, b.scale, ks, vs)
                    else:
                        api.pa_decode(out, q, kc, vc, bt, cl, b.scale)
                elif entry == "pa_decode_splitk":
                    if kv == "fp8":
                        api.pa_decode_splitk_fp8(out, q, kc, vc, bt, cl, b.scale, ks, vs, ps, ws, P)
                    else:
                        api.pa_decode_splitk(out, q, kc, vc, bt, cl, b.scale, ps, ws, P)
                    api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
                else:  # pa_decode_prefix_splitk
                    api.pa_decode_prefix_splitk(out, q, kc, vc, bt, cl, b.scale, b.seqs_per_group, T(b.prefix_lens),
                                                ps, ws, P, k_scale=ks, v_scale=vs)
                    api.pa_splitk_reduce(out, ws, cl, b.max_blocks_per_seq, b.block_size, ps, P)
            torch.cuda.synchronize()
            exact = (np.array_equal(kc.cpu().numpy().view(np.uint8), okc.view(np.uint8)) and
                     np.array_equal(vc.cpu().numpy().view(np.uint8), ovc.view(np.uint8)))
            err = float(np.max(np.abs(out.double().cpu().numpy() - ref)))
            return err, exact

        entries = ["pa_decode", "pa_decode_splitk", "pa_append_and_decode", "pa_append_and_decode_splitk"]
        if b.prefix_lens is not None:
            entries.append("pa_decode_prefix_splitk")
        kvb = workloads.algorithmic_kv_bytes(b)
        for e in entries:
            err, exact = run(e)
            suffix = f" (ps {ps})" if "splitk" in e else ""
            print(f"| {name} | {kvb:,} | {e}{suffix} | {err:.3e} | {'yes' if exact else 'NO'} |", flush=True)
        sys.stderr.write(f"{name}: {time.time() - t0:.1f} s\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
