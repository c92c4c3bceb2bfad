"""Measure every kernel configuration on the benchmark shapes and regenerate
csrc/dispatch_table.inc with the fastest one per shape.

The dispatcher reads that table first ("no single kernel is fastest": the
pages' lesson that libraries pick a variant per shape), and falls back to a
rule for shapes it does not list.  Run on the target GPU:

    python -m software_pipelined_gb300.tune --json tune.json \\
        --inc software_pipelined_gb300/csrc/dispatch_table.inc

With --rule-sweep it checks the rule instead: for shapes the table does not
list (squares, rectangles, skinny and ragged shapes, leading dimensions that
are not multiples of 4) it times the dispatcher's own plan against the best
forced candidate and prints both with their ratio:

    python -m software_pipelined_gb300.tune --rule-sweep --json rule.json --md

Each candidate is planned with forced options, warmed up, and timed as the
median of three replays of a CUDA graph holding back-to-back runs (events
around each replay), so launch overhead on the host does not decide.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import software_pipelined_gb300 as g  # noqa: E402
from software_pipelined_gb300 import inputs  # noqa: E402

# (tile_m, tile_n, stages, tile_k)
SIMT_CFGS = [(128, 128, 2, 16), (128, 128, 3, 16), (128, 128, 1, 16), (64, 64, 2, 16), (64, 64, 3, 16),
             (64, 64, 1, 16), (64, 64, 2, 32), (32, 32, 2, 32), (32, 32, 1, 32), (128, 64, 2, 16),
             (32, 32, 3, 32), (32, 32, 1, 64), (32, 32, 2, 64), (32, 64, 2, 32), (64, 32, 2, 32),
             (32, 32, 4, 32), (32, 32, 3, 64), (64, 64, 4, 16), (32, 64, 3, 32), (64, 32, 3, 32),
             (16, 32, 3, 32), (32, 16, 3, 32)]
TC_BN = [64, 128, 256]
SPLITS = [1, 2, 3, 4, 6, 8, 12, 16]


def time_plan(plan, dA, dB, dC, stream, target_ms=5.0, batches=3):
    """Median device time per run (ms): runs captured back to back in a CUDA
    graph, the graph replayed between two events."""
    import torch
    s = torch.cuda.Stream()
    run = lambda: plan.run_ptr(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), s.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(3):
            run()
        e0.record(s)
        run()
        e1.record(s)
    e1.synchronize()
    reps = int(max(1, min(200, target_ms / max(e0.elapsed_time(e1), 1e-3))))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(reps):
            run()
    res = []
    with torch.cuda.stream(s):  # replay() launches on the current stream
        graph.replay()
        s.synchronize()
        for _ in range(batches):
            e0.record(s)
            graph.replay()
            e1.record(s)
            e1.synchronize()
            res.append(e0.elapsed_time(e1) / reps)
    del graph
    if plan.check(s.cuda_stream) != g.OK:
        raise RuntimeError("device status not OK")
    return statistics.median(res)


def candidates(M, N, K):
    out = []
    macs = M * N * K
    if macs <= 2 ** 31:
        for (bm, bn, st, bk) in SIMT_CFGS:
            for ksl in (1, 2, 4):
                for sp in SPLITS:
                    if sp == 1 or K // sp >= 32:
                        out.append(dict(variant=g.VARIANT_SIMT, tile_m=bm, tile_n=bn, stages=st, split_k=sp,
                                        tile_k=bk, k_slices=ksl))
    if K >= 32 and macs >= 2 ** 27:
        # CTA pairs (256-row tiles): operands split in the kernel, B by the
        # pre-pass, or lo of A and B by the pre-pass (no conversion in the kernel)
        for bn in (256, 128):
            for fused in (2, 3, 4):
                for tk in ((32, 16) if fused == 2 or (fused == 4 and bn == 256) else (32,)):
                    for sp in [0] + SPLITS:
                        if sp <= 1 or (K + 31) // 32 >= sp:
                            out.append(dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=bn, stages=0,
                                            split_k=sp, operand_split=fused, tile_k=tk))
    if K >= 16:
        for bn in TC_BN:
            for fused in ((1, 2, 3, 4) if bn in (128, 256) and K >= 32 else (1,)):
                for tk in ((0, 16) if fused == 2 else (0,)):
                    for sp in [0] + SPLITS:
                        if sp <= 1 or (K + 31) // 32 >= sp:
                            out.append(dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=bn, stages=0, split_k=sp,
                                            operand_split=fused, tile_k=tk))
    return out


# Shapes outside the table: (M, N, K, lda, ldb); lda/ldb None = tight.
RULE_SHAPES = [
    (768, 768, 768, None, None), (1280, 1280, 1280, None, None), (1536, 1536, 1536, None, None),
    (2048, 2048, 2048, None, None), (2560, 2560, 2560, None, None), (3072, 3072, 3072, None, None),
    (6144, 6144, 6144, None, None), (1000, 1000, 1000, None, None), (4100, 4100, 4100, None, None),
    (2048, 8192, 1024, None, None), (8192, 2048, 1024, None, None), (4096, 1024, 4096, None, None),
    (1024, 4096, 4096, None, None), (4096, 4096, 1024, None, None), (3000, 5000, 2000, None, None),
    (777, 1234, 555, None, None), (8192, 256, 1024, None, None), (256, 8192, 1024, None, None),
    (16384, 64, 256, None, None), (64, 16384, 512, None, None), (4096, 128, 4096, None, None),
    (128, 4096, 4096, None, None), (64, 64, 64, None, None), (200, 300, 100, None, None),
    (96, 96, 1024, None, None), (33, 65, 129, None, None), (300, 40, 700, None, None),
    (1023, 1025, 1027, None, None), (2049, 2047, 2051, None, None), (1024, 1024, 1024, 1027, 1029),
    (4096, 4096, 4096, 4097, 4099),
    # many output tiles over a short K
    (1024, 1024, 16, None, None), (2048, 2048, 16, None, None), (4096, 4096, 16, None, None),
    (3000, 5000, 20, None, None), (8192, 2048, 24, None, None), (1500, 1500, 31, None, None),
    (800, 800, 16, None, None), (800, 800, 64, None, None), (640, 640, 24, None, None),
    (16384, 4096, 20, None, None), (4096, 4096, 24, None, None), (2048, 8192, 28, None, None),
]


def rule_sweep(args):
    """The dispatcher's plan against the best forced candidate on RULE_SHAPES."""
    import torch
    stream = torch.cuda.current_stream()
    results = []
    only = set(args.rule_shapes.split(",")) if args.rule_shapes else None
    for (M, N, K, lda, ldb) in RULE_SHAPES:
        if only and f"{M}x{N}x{K}" not in only:
            continue
        lda, ldb = lda or K, ldb or N
        A = inputs.uniform_pm1(8001, M, K, ld=lda if lda != K else None)
        B = inputs.uniform_pm1(8002, K, N, ld=ldb if ldb != N else None)
        dA = torch.full((M * lda,), float("nan"), device="cuda")
        dA.view(M, lda)[:, :K] = torch.from_numpy(inputs.uniform_pm1(8001, M, K)).cuda()
        dB = torch.full((K * ldb,), float("nan"), device="cuda")
        dB.view(K, ldb)[:, :N] = torch.from_numpy(inputs.uniform_pm1(8002, K, N)).cuda()
        del A, B
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        with g.Plan(M, N, K, lda, ldb, N) as p:
            auto_desc = p.describe()
            auto_us = round(time_plan(p, dA, dB, dC, stream) * 1e3, 3)
        best = (auto_us, auto_desc)
        cands = candidates(M, N, K)
        if M * N * K > 2 ** 34:  # big products: every tile sliced in K is never the answer
            cands = [c for c in cands if c.get("split_k", 0) <= 2]
        for c in cands:
            try:
                with g.Plan(M, N, K, lda, ldb, N, **c) as p:
                    us = round(time_plan(p, dA, dB, dC, stream) * 1e3, 3)
                    if us < best[0]:
                        best = (us, p.describe())
            except g.GemmError:
                continue
        shape = f"{M}x{N}x{K}" + (f" lda={lda} ldb={ldb}" if (lda, ldb) != (K, N) else "")
        r = dict(shape=shape, rule_us=auto_us, rule_plan=auto_desc, best_us=best[0], best_plan=best[1],
                 rule_over_best=round(auto_us / best[0], 4))
        results.append(r)
        print(json.dumps(r), flush=True)
        del dA, dB, dC
    if args.json:
        with open(args.json, "w") as f:
            json.dump(results, f, indent=1)
    if args.md:
        short = lambda d: " ".join(t for t in d.split() if not t.startswith(("terms=", "ws=", "kp=", "resident=",
                                                                             "whole=", "pairs=", "tiles=", "thread=")))
        print("| shape | rule's plan | us | best forced plan | us | rule / best |")
        print("|---|---|---:|---|---:|---:|")
        for r in results:
            print(f"| {r['shape']} | {short(r['rule_plan'])} | {r['rule_us']} | {short(r['best_plan'])} | "
                  f"{r['best_us']} | {r['rule_over_best']} |")


def main():
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--json", default=None)
    ap.add_argument("--inc", default=None)
    ap.add_argument("--workloads", default="tiny_32,small_ragged,tall_skinny,square_1024,large_squares")
    ap.add_argument("--rule-sweep", action="store_true")
    ap.add_argument("--rule-shapes", default=None, help="with --rule-sweep: only these MxNxK, comma-separated")
    ap.add_argument("--md", action="store_true")
    args = ap.parse_args()
    g.load()
    if args.rule_sweep:
        return rule_sweep(args)
    stream = torch.cuda.current_stream()
    results = []
    for key in args.workloads.split(","):
        for (name, M, N, K, dist, sa, sb) in inputs.WORKLOADS[key]:
            A, B = inputs.make_operands(M, N, K, dist, sa, sb)
            dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
            dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
            rows = []
            for c in candidates(M, N, K):
                try:
                    with g.Plan(M, N, K, **c) as p:
                        ms = time_plan(p, dA, dB, dC, stream)
                        rows.append(dict(opts=c, us=round(ms * 1e3, 3), plan=p.describe()))
                except g.GemmError:
                    continue
            rows.sort(key=lambda r: r["us"])
            if rows[0]["opts"]["variant"] == g.VARIANT_TCGEN05:
                # the tile order of the winner: tile-rows per raster group
                for grp in (4, 8, 12, 16, 24):
                    c = dict(rows[0]["opts"], tile_group=grp)
                    with g.Plan(M, N, K, **c) as p:
                        rows.append(dict(opts=c, us=round(time_plan(p, dA, dB, dC, stream) * 1e3, 3),
                                         plan=p.describe()))
                rows.sort(key=lambda r: r["us"])
            with g.Plan(M, N, K) as p:
                auto_desc = p.describe()
                auto_us = round(time_plan(p, dA, dB, dC, stream) * 1e3, 3)
            results.append(dict(shape=name, M=M, N=N, K=K, best=rows[0], top=rows[:40],
                                auto=dict(plan=auto_desc, us=auto_us), n_candidates=len(rows)))
            print(f"{name:18s} best {rows[0]['us']:10.3f} us  {rows[0]['plan']}   (auto {auto_us} us)",
                  flush=True)
            del dA, dB, dC
    if args.json:
        with open(args.json, "w") as f:
            json.dump(results, f, indent=1)
    if args.inc:
        write_inc(results, args.inc)


def effective_split(desc: str) -> int:
    """The table's split field for the configuration a plan description shows:
    SIMT: its split_k; tensor cores: 1 = no split tile, 0 = only the last wave
    split (automatic), n = every tile in n K-slices."""
    import re
    if desc.startswith("simt"):
        return int(re.search(r"split_k=(\d+)", desc).group(1))
    whole = int(re.search(r"whole=(\d+)", desc).group(1))
    tiles, slices = (int(v) for v in re.search(r"split=(\d+)x(\d+)", desc).groups())
    if tiles == 0:
        return 1
    return 0 if whole > 0 else slices


def split_where(desc: str) -> int:
    """The table's split field: 0 pre-pass, 1 in the kernel, 2 hybrid, 3 raw A,
    4 A in tensor memory."""
    return (1 if "in-kernel-split" in desc else 2 if "hybrid-split" in desc
            else 3 if "raw-a-split" in desc else 4 if "tmem-a-split" in desc else 0)


def write_inc(results, path):
    lines = [
        "// Per-shape dispatch table: the fastest configuration measured on GB300 for",
        "// each benchmark shape (exact match on M, N, K), written by",
        "// software_pipelined_gb300/tune.py from its timing sweep.  Shapes not listed",
        "// fall back to the rule in choose().  Fields: variant (1 SIMT, 2 tcgen05),",
        "// tile_m (tcgen05: 256 = CTA pairs), tile_n, stages (0 = compiled default), split_k (0 = automatic",
        "// last-wave split, 1 = none, >= 2 = every tile in that many K-slices),",
        "// split (tcgen05: 0 pre-pass, 1 inside the kernel, 2 A inside and B by the pre-pass,",
        "// 3 hi of A read from A, 4 A split into tensor memory by the CTA pair),",
        "// tile_group (tcgen05: tile-rows per raster group, 0 = default), tile_k (SIMT:",
        "// K-tile depth; tcgen05: k per stage, 32 or 16; 0 = default), k_slices (SIMT:",
        "// K-slice groups inside the CTA) and split_reduce (0 = the reduction kernel).",
        "struct TableRow {",
        "    int64_t M, N, K;",
        "    DispatchChoice c;",
        "};",
        "",
        "const TableRow kTable[] = {",
    ]
    for r in results:
        o = r["best"]["opts"]
        split = effective_split(r["best"]["plan"])
        lines.append(f"    {{{r['M']}, {r['N']}, {r['K']}, {{{o['variant']}, {o['tile_m']}, {o['tile_n']}, "
                     f"{o['stages']}, {split}, {split_where(r['best']['plan'])}, {o.get('tile_group', 0)}, "
                     f"{o.get('tile_k', 0)}, {o.get('k_slices', 0)}, {o.get('split_reduce', 0)}}}}},"
                     f"  // {r['best']['us']} us")
    lines += [
        "    {0, 0, 0, {0, 0, 0, 0, 0, 0, 0, 0, 0, 0}},  // sentinel",
        "};",
        "",
        "bool table_lookup(int64_t M, int64_t N, int64_t K, DispatchChoice& out)",
        "{",
        "    for (const TableRow& r : kTable) {",
        "        if (r.M == M && r.N == N && r.K == K && r.c.variant != 0) {",
        "            out = r.c;",
        "            return true;",
        "        }",
        "    }",
        "    return false;",
        "}",
        "",
    ]
    with open(path, "w") as f:
        f.write("\n".join(lines))


if __name__ == "__main__":
    main()
