"""The pages' two measured claims, re-measured on GB300:

1. Pipeline depth ("Double Buffering" technique page, the paragraph on the
   cost of the second buffer; "Case Study: The Double-Buffered GEMM", the
   three-regimes paragraph): single-buffered vs double-buffered vs deeper
   rings, whose winner changes with the problem size.
2. Barrier coalescing ("Dependence-aware group synchronization on M1 Max",
   "Transformation and safety boundary" and "Controlled implementation
   comparison"): publishing A and B with one synchronisation instead of one
   each, with the dynamic barrier counts beside the time.
3. Fragment loads of the SIMT kernel ("Case Study: The Double-Buffered GEMM",
   kernel listing: fragments of the staged tiles feed the multiply-adds):
   16-byte shared-memory loads that lanes needing the same values share
   (broadcast) against one read per distinct value and warp shuffles, on the
   small shapes and at 2048^3.

For every benchmark shape each variant is planned with forced options and
timed as CUDA-graph replays of back-to-back runs (device time, no host
launch overhead).  Prints a JSON document (and a markdown table with --md):

    python -m software_pipelined_gb300.ablation --json ablation.json --md
    python -m software_pipelined_gb300.ablation --only fragments --md
"""
from __future__ import annotations

import argparse
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import software_pipelined_gb300 as g  # noqa: E402
from software_pipelined_gb300 import inputs  # noqa: E402
from software_pipelined_gb300.tune import time_plan  # noqa: E402

SHAPES = [w for key in ("tiny_32", "small_ragged", "tall_skinny", "square_1024", "large_squares")
          for w in inputs.WORKLOADS[key]]

# (label, plan options, barriers a CTA waits per K-tile of 32/BK, kind)
DEPTH = [
    ("simt 64x64 S=1", dict(variant=1, tile_m=64, tile_n=64, stages=1, split_k=1)),
    ("simt 64x64 S=2", dict(variant=1, tile_m=64, tile_n=64, stages=2, split_k=1)),
    ("simt 64x64 S=3", dict(variant=1, tile_m=64, tile_n=64, stages=3, split_k=1)),
    ("simt 128x128 S=1", dict(variant=1, tile_m=128, tile_n=128, stages=1, split_k=1)),
    ("simt 128x128 S=2", dict(variant=1, tile_m=128, tile_n=128, stages=2, split_k=1)),
    ("simt 128x128 S=3", dict(variant=1, tile_m=128, tile_n=128, stages=3, split_k=1)),
    ("tc 128x128 S=1", dict(variant=2, tile_n=128, stages=1)),
    ("tc 128x128 S=2", dict(variant=2, tile_n=128, stages=2)),
    ("tc 128x128 S=3", dict(variant=2, tile_n=128, stages=3)),
    ("tc 128x256 S=1", dict(variant=2, tile_n=256, stages=1)),
    ("tc 128x256 S=2", dict(variant=2, tile_n=256, stages=2)),
]

COALESCE = [
    ("simt 64x64 S=1", dict(variant=1, tile_m=64, tile_n=64, stages=1, split_k=1)),
    ("simt 64x64 S=2", dict(variant=1, tile_m=64, tile_n=64, stages=2, split_k=1)),
    ("simt 32x32 S=1", dict(variant=1, tile_m=32, tile_n=32, stages=1, split_k=1)),
    ("simt 32x32 S=2", dict(variant=1, tile_m=32, tile_n=32, stages=2, split_k=1)),
    ("tc 128x256 S=2", dict(variant=2, tile_n=256, stages=2)),
    ("tc 128x128 S=3", dict(variant=2, tile_n=128, stages=3)),
]


FRAGMENTS = [
    ("simt 128x128x16 S=2", dict(variant=1, tile_m=128, tile_n=128, stages=2, tile_k=16, split_k=1)),
    ("simt 64x64x16 S=2", dict(variant=1, tile_m=64, tile_n=64, stages=2, tile_k=16, split_k=1)),
    ("simt 64x64x16 S=4 2 K-groups", dict(variant=1, tile_m=64, tile_n=64, stages=4, tile_k=16, k_slices=2,
                                          split_k=1)),
    ("simt 32x32x32 S=3 4 K-groups", dict(variant=1, tile_m=32, tile_n=32, stages=3, tile_k=32, k_slices=4,
                                          split_k=1)),
]
FRAGMENT_SHAPES = [w for key in ("tiny_32", "small_ragged", "tall_skinny", "square_1024")
                   for w in inputs.WORKLOADS[key]] + [("2048x2048x2048", 2048, 2048, 2048, "uniform", 7001, 7002)]


def barrier_count(opts, sep, K, bk):
    """Dynamic barriers one CTA executes over L = ceil(K/bk) K-tiles.
    SIMT: block-wide __syncthreads; tensor cores: mbarrier waits of the MMA
    thread on landed tiles (plus one empty-slot wait of the producer per tile,
    the same in both forms)."""
    L = -(-K // bk)
    if opts["variant"] == 1:
        if opts["stages"] == 1:
            return {"formula": "3L" if sep else "2L", "count": (3 if sep else 2) * L}
        return {"formula": "2L" if sep else "L", "count": (2 if sep else 1) * L}
    return {"formula": "2L full + L empty" if sep else "L full + L empty", "count": (3 if sep else 2) * L}


def measure(M, N, K, opts, dA, dB, dC, stream):
    try:
        with g.Plan(M, N, K, **opts) as p:
            return round(time_plan(p, dA, dB, dC, stream) * 1e3, 3), p.describe()
    except g.GemmError as e:
        return None, str(e)


def main():
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--json", default=None)
    ap.add_argument("--md", action="store_true")
    ap.add_argument("--only", choices=["depth", "fragments"], default=None,
                    help="depth: the depth and coalescing tables only; fragments: the fragment-load table only")
    args = ap.parse_args()
    g.load()
    stream = torch.cuda.current_stream()
    out = {"depth": [], "coalesce": [], "fragments": []}
    for (name, M, N, K, dist, sa, sb) in (FRAGMENT_SHAPES if args.only != "depth" else []):
        A, B = inputs.make_operands(M, N, K, dist, sa, sb)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for label, o in FRAGMENTS:
            tb, db = measure(M, N, K, dict(o, simt_fragments=0), dA, dB, dC, stream)
            ts, ds = measure(M, N, K, dict(o, simt_fragments=1), dA, dB, dC, stream)
            out["fragments"].append({"shape": name, "variant": label, "broadcast_us": tb, "shuffle_us": ts,
                                     "shuffle_over_broadcast": round(ts / tb, 4) if tb and ts else None})
            print(json.dumps(out["fragments"][-1]), flush=True)
        del dA, dB, dC
    for (name, M, N, K, dist, sa, sb) in (SHAPES if args.only != "fragments" else []):
        A, B = inputs.make_operands(M, N, K, dist, sa, sb)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        big = M * N * K > 2 ** 31
        row = {"shape": name}
        for label, o in DEPTH:
            if big and o["variant"] == 1:
                continue
            row[label] = measure(M, N, K, o, dA, dB, dC, stream)[0]
        out["depth"].append(row)
        for label, o in COALESCE:
            if big and o["variant"] == 1:
                continue
            t1, d1 = measure(M, N, K, dict(o, separate_syncs=0), dA, dB, dC, stream)
            t2, d2 = measure(M, N, K, dict(o, separate_syncs=1), dA, dB, dC, stream)
            bk = 32 if o["variant"] == 2 or o.get("tile_m") == 32 else 16
            out["coalesce"].append({
                "shape": name, "variant": label, "coalesced_us": t1, "separate_us": t2,
                "speedup": round(t2 / t1, 4) if t1 and t2 else None,
                "barriers_coalesced": barrier_count(o, False, K, bk),
                "barriers_separate": barrier_count(o, True, K, bk)})
        print(json.dumps(row), flush=True)
        del dA, dB, dC
    if args.json:
        with open(args.json, "w") as f:
            json.dump(out, f, indent=1)
    if args.md and out["fragments"]:
        print("| shape | variant | broadcast loads (us) | warp shuffles (us) | shuffles/broadcast |")
        print("|---|---|---:|---:|---:|")
        for r in out["fragments"]:
            print(f"| {r['shape']} | {r['variant']} | {r['broadcast_us']} | {r['shuffle_us']} | "
                  f"{r['shuffle_over_broadcast']} |")
        print()
    if args.md and out["depth"]:
        labels = [l for l, _ in DEPTH]
        print("| shape | " + " | ".join(labels) + " |")
        print("|---|" + "---:|" * len(labels))
        for r in out["depth"]:
            print(f"| {r['shape']} | " + " | ".join(str(r.get(l, "")) for l in labels) + " |")
        print()
        print("| shape | variant | one sync (us) | separate (us) | separate/one | barriers one | barriers separate |")
        print("|---|---|---:|---:|---:|---|---|")
        for r in out["coalesce"]:
            print(f"| {r['shape']} | {r['variant']} | {r['coalesced_us']} | {r['separate_us']} | {r['speedup']} | "
                  f"{r['barriers_coalesced']['formula']} = {r['barriers_coalesced']['count']} | "
                  f"{r['barriers_separate']['formula']} = {r['barriers_separate']['count']} |")


if __name__ == "__main__":
    main()
