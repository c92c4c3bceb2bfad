#!/usr/bin/env python
"""FP32 GEMM benchmark: TFLOP/s (2MNK / CUDA-event time) per shape and % of roofline.

Headline workload: the large squares 4096x4096x4096 and 8192x8192x8192 (A, B
uniform[-1,1) from seeded SplitMix64).  One step = one GEMM of each shape
through the C-ABI (gemm_f32_run), inputs resident in HBM; both shapes' operands
exceed the 129 MB L2, so no flush is needed between steps.  `value` is
2*sum(MNK) per step over the device-timed step (CUDA events, max over ranks),
times the number of ranks.

Also printed, in the same JSON line:
  roofline      the dominant kernel (tcgen05 main GEMM) timed live with CUDA
                events recorded by the library around each launch (tracing
                API), against the 3xTF32-effective tensor peak;
  per_shape     every shape of every configuration: TFLOP/s, roofline fraction,
                chosen kernel, max normalised error against the CPU oracle;
  e2e           the same metric through gemm_f32_run_host with pinned host
                buffers (host->device copies of A, B and the copy of C back
                inside the timed region);
  cpu_baseline  the CPU oracle timed on a bounded sample of the workload.

`--impl reference` times the CPU oracle itself (the reference arm: there is no
runnable reference implementation for this GPU) on the same workload.
With torchrun (N > 1) every rank runs an independent replica (weak scaling);
there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP32 GEMM TFLOP/s (2MNK/CUDA-event time) per shape; % of roofline"
HEADLINE = "large_squares"
TF32_OVER_BF16 = 1.1 / 2.25          # nominal dense TF32 : BF16 tensor ratio
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "measured"
    try:
        with open(path) as f:
            p = json.load(f)
    except (OSError, ValueError):
        p, src = dict(FALLBACK), "fallback"
    hbm = float(p.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    bf16 = float(p.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    bf16s = float(p.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]))
    return {
        "source": src,
        "hbm_gbs": hbm,
        # 3xTF32-effective FP32 peak = dense TF32 peak / 3, the TF32 peak taken
        # as the measured BF16 peak times the nominal TF32:BF16 ratio.
        "f32_3xtf32_tflops_burst": bf16 * TF32_OVER_BF16 / 3.0,
        "f32_3xtf32_tflops_sustained": bf16s * TF32_OVER_BF16 / 3.0,
        # FP32 SIMT: 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz (nominal).
        "f32_simt_tflops_nominal": 152 * 128 * 2 * 2.07e9 / 1e12,
    }


def shapes_of(workload, shape=None):
    """The (name, M, N, K, dist, seed_A, seed_B) entries of a workload, or a
    single M x N x K shape (uniform inputs) when `shape` is given."""
    from software_pipelined_gb300 import inputs
    if shape:
        M, N, K = (int(v) for v in shape.lower().split("x"))
        return [(f"{M}x{N}x{K}", M, N, K, "uniform", 5001, 5002)]
    return inputs.WORKLOADS[workload]


def algorithmic_bytes(M, N, K):
    return 4 * (M * K + K * N + M * N)


def max_over_ranks(value, dist, device):
    """The largest of the ranks' values (every rank gets it); the value itself
    without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_rank_step, world, seconds_per_step):
    """Whole-job throughput in TFLOP/s: every rank runs one replica of the
    step, and the job's step time is the slowest rank's."""
    return world * flops_per_rank_step / seconds_per_step / 1e12


# ---------------------------------------------------------------------------
# Clocks sampled during the timed region.
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm).
# ---------------------------------------------------------------------------

def oracle_rows_rate(A, B, rows):
    """Time the oracle on the first `rows` rows of A*B; returns (seconds, flops)."""
    import oracle
    Asub = np.ascontiguousarray(A[:rows])
    t0 = time.perf_counter()
    oracle.gemm_f64(Asub, B, with_scale=False)
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows * B.shape[1] * A.shape[1]


def oracle_sample(A, B, target_s):
    """Largest row block (a multiple of the thread count) the oracle finishes in
    about target_s seconds, timed; returns (tflops, rows, seconds, threads)."""
    import oracle
    threads = oracle.get_threads()
    cal = max(threads, 1)
    dt, fl = oracle_rows_rate(A, B, cal)
    rows = int(max(cal, min(A.shape[0], cal * max(1, round(target_s / max(dt, 1e-6))))))
    rows = max(threads, rows // threads * threads) if rows >= threads else rows
    dt, fl = oracle_rows_rate(A, B, rows)
    return fl / dt / 1e12, rows, dt, threads


# ---------------------------------------------------------------------------
# GPU arm.
# ---------------------------------------------------------------------------

def time_batches(plan_run, stream, target_ms=20.0, batches=5, warm_ms=100.0):
    """Median per-run time (ms) over batches of back-to-back runs, CUDA events."""
    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # one timed run to size the batch
    for _ in range(3):
        plan_run()
    ev0.record(stream)
    plan_run()
    ev1.record(stream)
    ev1.synchronize()
    one = max(ev0.elapsed_time(ev1), 1e-3)
    reps = int(max(1, min(2000, target_ms / one)))
    t_end = time.perf_counter() + warm_ms / 1e3
    while time.perf_counter() < t_end:
        for _ in range(reps):
            plan_run()
        torch.cuda.synchronize()
    res = []
    for _ in range(batches):
        ev0.record(stream)
        for _ in range(reps):
            plan_run()
        ev1.record(stream)
        ev1.synchronize()
        res.append(ev0.elapsed_time(ev1) / reps)
    return statistics.median(res), min(res), max(res), reps


def time_graph(run_on, target_ms=20.0, batches=5):
    """Median per-run device time (ms) with the runs captured back to back in a
    CUDA graph and replayed, so host launch overhead is not in the number.
    run_on(stream_handle) enqueues one run on the given stream."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            run_on(s.cuda_stream)
    s.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s)
    run_on(s.cuda_stream)
    ev1.record(s)
    ev1.synchronize()
    reps = int(max(1, min(500, target_ms / max(ev0.elapsed_time(ev1), 1e-3))))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(reps):
            run_on(s.cuda_stream)
    res = []
    with torch.cuda.stream(s):  # replay() launches on the current stream
        for _ in range(2):
            graph.replay()
        s.synchronize()
        for _ in range(batches):
            ev0.record(s)
            graph.replay()
            ev1.record(s)
            ev1.synchronize()
            res.append(ev0.elapsed_time(ev1) / reps)
    del graph
    return statistics.median(res), min(res), max(res), reps


class CublasCompare:
    """cuBLAS through ctypes, for the comparison columns only (never on the
    measured path): FP32 emulated with BF16 pieces (compute type
    CUBLAS_COMPUTE_32F_EMULATED_16BFX9, emulation strategy EAGER so that it is
    used at every size) and single TF32 (CUBLAS_COMPUTE_32F_FAST_TF32, not
    FP32-accurate: the tensor pipe's own rate).  Row-major C = A B is computed
    as the column-major C^T = B^T A^T.  Unavailable (None times) when the
    library or a call is missing."""

    COMPUTE = {"bf16x9": 78, "tf32": 77, "sgemm": 68}

    def __init__(self):
        import ctypes
        import glob
        import torch
        self.ok = False
        self.why = None
        torch.mm(torch.zeros(8, 8, device="cuda"), torch.zeros(8, 8, device="cuda"))  # torch's cuBLAS loaded
        cands = ["libcublas.so.13"]
        for p in sys.path:
            cands += sorted(glob.glob(os.path.join(p, "nvidia", "cu13", "lib", "libcublas.so.*")))
            cands += sorted(glob.glob(os.path.join(p, "nvidia", "cublas", "lib", "libcublas.so.*")))
        cands.append("/usr/local/cuda/lib64/libcublas.so")
        self.lib = None
        for c in cands:
            try:
                self.lib = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if self.lib is None:
            self.why = "libcublas not found"
            return
        self.c = ctypes
        self.h = ctypes.c_void_p()
        if self.lib.cublasCreate_v2(ctypes.byref(self.h)) != 0:
            self.why = "cublasCreate failed"
            return
        ver = ctypes.c_int()
        self.lib.cublasGetVersion_v2(self.h, ctypes.byref(ver))
        self.version = ver.value
        self.ws = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        if self.lib.cublasSetWorkspace_v2(self.h, ctypes.c_void_p(self.ws.data_ptr()),
                                          ctypes.c_size_t(self.ws.numel())) != 0:
            self.why = "cublasSetWorkspace failed"
            return
        try:
            emu = self.lib.cublasSetEmulationStrategy(self.h, 2)
        except AttributeError:
            emu = -1
        self.emulation = emu == 0
        vp, i = ctypes.c_void_p, ctypes.c_int
        self.lib.cublasGemmEx.argtypes = [vp, i, i, i, i, i, vp, vp, i, i, vp, i, i, vp, vp, i, i, i, i]
        self.lib.cublasSetStream_v2.argtypes = [vp, vp]
        self.one, self.zero = ctypes.c_float(1.0), ctypes.c_float(0.0)
        self.ok = True

    def gemm(self, kind, st, dA, dB, dC, M, N, K):
        c = self.c
        self.lib.cublasSetStream_v2(self.h, c.c_void_p(st))
        return self.lib.cublasGemmEx(self.h, 0, 0, N, M, K, c.byref(self.one), dB.data_ptr(), 0, N,
                                     dA.data_ptr(), 0, K, c.byref(self.zero), dC.data_ptr(), 0, N,
                                     self.COMPUTE[kind], -1)

    def time(self, kind, dA, dB, dC, M, N, K):
        """Graph-replayed per-call time (ms) of one compute type, or None."""
        import torch
        if not self.ok or (kind == "bf16x9" and not self.emulation):
            return None
        if self.gemm(kind, torch.cuda.current_stream().cuda_stream, dA, dB, dC, M, N, K) != 0:
            return None
        torch.cuda.synchronize()
        try:
            med, _, _, _ = time_graph(lambda st: self.gemm(kind, st, dA, dB, dC, M, N, K))
        except RuntimeError:
            return None
        finally:
            self.lib.cublasSetStream_v2(self.h, self.c.c_void_p(torch.cuda.current_stream().cuda_stream))
        return med

    def close(self):
        if self.ok:
            import torch
            torch.cuda.synchronize()
            self.lib.cublasDestroy_v2(self.h)
            self.ok = False


def make_device_operands(M, N, K, dist, sa, sb):
    import torch
    from software_pipelined_gb300 import inputs
    A, B = inputs.make_operands(M, N, K, dist, sa, sb)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    return A, B, dA, dB, dC


def capture_for_check(A, B, Cd, full_limit=2 ** 31):
    """What the oracle comparison needs of a GPU result (no oracle here): the
    whole output for moderate sizes (always, with full_limit None), 1028
    sampled entries beyond."""
    M, K = A.shape
    N = B.shape[1]
    if full_limit is None or M * N * K <= full_limit:
        return {"A": A, "B": B, "kind": "full", "C": Cd.cpu().numpy()}
    rng = np.random.default_rng(12345)
    rows = np.concatenate([[0, M - 1, 0, M - 1], rng.integers(0, M, 1024)])
    cols = np.concatenate([[0, 0, N - 1, N - 1], rng.integers(0, N, 1024)])
    import torch
    vals = Cd[torch.from_numpy(rows).to(Cd.device), torch.from_numpy(cols).to(Cd.device)].cpu().numpy()
    return {"A": A, "B": B, "kind": "sampled-1028", "rows": rows, "cols": cols, "vals": vals}


def compare_with_oracle(chk, cache=None):
    """Max normalised error of a captured GPU result against the oracle.  With
    a cache (a dict), the oracle's product of the same A and B objects is
    computed once."""
    import oracle
    A, B = chk["A"], chk["B"]
    K = A.shape[1]
    if chk["kind"] == "full":
        key = (id(A), id(B))
        if cache is not None and key in cache:
            Cr, S = cache[key]
        else:
            Cr, S = oracle.gemm_f64(A, B)
            if cache is not None:
                cache[key] = (Cr, S)
        return round(oracle.normalised_error(chk["C"], Cr, S, K), 4), "full"
    c, s = oracle.gemm_f64_entries(A, B, chk["rows"], chk["cols"])
    return round(oracle.normalised_error(chk["vals"], c, s, K), 4), chk["kind"]


def time_oracle(A, B, n):
    """Median host wall time (s) of n full oracle products."""
    import oracle
    ts = []
    for _ in range(n):
        t0 = time.perf_counter()
        oracle.gemm_f64(A, B, with_scale=False)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts)


def run_environment(device):
    """Where the numbers were taken: device, SM count, driver and CUDA versions,
    host cores, and the sources (git revision where .git exists, else a hash
    of the CUDA sources, the header and the dispatch table)."""
    import subprocess
    import torch
    props = torch.cuda.get_device_properties(device)
    env = {"device": props.name, "sm_count": props.multi_processor_count,
           "memory_gib": round(props.total_memory / 2 ** 30, 1),
           "cuda_runtime": torch.version.cuda, "torch": torch.__version__, "host_cores": os.cpu_count()}
    try:
        env["driver"] = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                                        "-i", str(device)], capture_output=True, text=True,
                                       timeout=20).stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        env["driver"] = None
    try:
        env["git_revision"] = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                                             text=True, timeout=20).stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        env["git_revision"] = None
    csrc = os.path.join(ROOT, "software_pipelined_gb300", "csrc")
    env["sources_sha256_16"] = source_hash(sorted(os.path.join(csrc, f) for f in os.listdir(csrc)) +
                                           [os.path.join(ROOT, "include", "gemm_f32.h")])
    return env


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_src_hash, plans):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, for each shape whose plan (its description: tile, operand split,
    stages, K-slices, tile order) and kernel sources are those the capture was
    taken on; plans: {shape name: plan description}."""
    path = os.path.join(ROOT, "profiles", "tcgen05_main_dram_traffic.txt")
    try:
        with open(path) as f:
            lines = [l.split("#")[0].strip() for l in f]
    except OSError:
        return None, "no ncu traffic summary"
    kv = dict(l.split("=", 1) for l in lines if "=" in l)
    if kv.get("kernel_source_sha256_16") != kernel_src_hash:
        return None, "kernel changed since the ncu capture"
    out = {}
    for name, desc in plans.items():
        if kv.get("plan_" + name) == desc and "bytes_per_launch_" + name in kv:
            try:
                out[name] = float(kv["bytes_per_launch_" + name])
            except ValueError:
                return None, "unreadable ncu summary"
    return (out, "ncu") if out else (None, "plan changed since the ncu capture")


def run_gpu_arm(args):
    import torch
    import software_pipelined_gb300 as g
    from software_pipelined_gb300 import build as gbuild

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        gbuild.build()
    if dist:
        dist.barrier()
    g.load()
    pk = peaks()
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    dev_name = torch.cuda.get_device_name(local)

    # ---- headline: the large squares, one GEMM of each per step -------------
    work = []
    for (name, M, N, K, dist_name, sa, sb) in shapes_of(args.workload, args.shape):
        A, B, dA, dB, dC = make_device_operands(M, N, K, dist_name, sa, sb)
        variant = {"auto": g.VARIANT_AUTO, "simt": g.VARIANT_SIMT, "tcgen05": g.VARIANT_TCGEN05}[args.variant]
        plan = g.Plan(M, N, K, variant=variant)
        plan.trace_enable(args.steps)
        work.append(dict(name=name, M=M, N=N, K=K, A=A, B=B, dA=dA, dB=dB, dC=dC, plan=plan,
                         run=(lambda p=plan, a=dA, b=dB, c=dC: p.run_ptr(a.data_ptr(), b.data_ptr(),
                                                                         c.data_ptr(), sptr))))
    flops_step = sum(2.0 * w["M"] * w["N"] * w["K"] for w in work)

    def step():
        for w in work:
            s = w["run"]()
            if s != g.OK:
                raise g.GemmError(s, "gemm_f32_run")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for w in work:  # drop warm-up traces; the timed region records afresh
        w["plan"].trace_read(args.steps)
        w["plan"].trace_enable(args.steps)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.1)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dist, "cuda")
    ms_step = ms_total / args.steps
    value = whole_job_rate(flops_step, world, ms_step * 1e-3)
    for w in work:
        s = w["plan"].check()
        if s != g.OK:
            raise g.GemmError(s, "gemm_f32_check")

    # per-kernel durations in the timed region (library-recorded CUDA events)
    main_fl, main_ms, split_ms, red_ms, per_kernel = 0.0, 0.0, 0.0, 0.0, {}
    for w in work:
        runs = w["plan"].trace_read(args.steps)
        sp = sum(r[0] for r in runs) / len(runs)
        mn = sum(r[1] for r in runs) / len(runs)
        rd = sum(r[2] for r in runs) / len(runs)
        main_fl += 2.0 * w["M"] * w["N"] * w["K"]
        main_ms += mn
        split_ms += sp
        red_ms += rd
        per_kernel[w["name"]] = {"plan": w["plan"].describe(), "split_ms": round(sp, 4),
                                 "main_ms": round(mn, 4), "reduce_ms": round(rd, 4),
                                 "main_tflops": round(2.0 * w["M"] * w["N"] * w["K"] / (mn * 1e-3) / 1e12, 2)}
    # The dominant kernel: the tcgen05 main GEMM of the largest shape (the
    # biggest share of the step).  Its peak is the 3xTF32-effective tensor peak
    # from the burst BF16 measurement: the kernel runs at full SM clock with no
    # power-cap reason (see clocks), which is the burst regime.
    big = max(work, key=lambda w: w["M"] * w["N"] * w["K"])
    bk = per_kernel[big["name"]]
    achieved = bk["main_tflops"]
    simt_main = big["plan"].describe().startswith("simt")
    peak = pk["f32_simt_tflops_nominal"] if simt_main else pk["f32_3xtf32_tflops_burst"]
    kern_hash = source_hash([os.path.join(ROOT, "software_pipelined_gb300", "csrc", f)
                             for f in ("tc_kernels.cuh", "tc_pair.cu", "tc_common.cuh", "ptx.cuh")])
    big_desc = big["plan"].describe()
    kname = ("simt_gemm_kernel (FFMA)" if simt_main else
             "tc_pair_kernel (tcgen05 3xTF32 main GEMM on CTA pairs)" if "cta-pair" in big_desc else
             "tc_gemm_kernel (tcgen05 3xTF32 main GEMM)")
    traffic, traffic_src = traffic_for(kern_hash, {w["name"]: w["plan"].describe() for w in work})
    for w in work:
        t = traffic.get(w["name"]) if traffic else None
        per_kernel[w["name"]]["dram_bytes_per_launch"] = t
        per_kernel[w["name"]]["frac"] = round(per_kernel[w["name"]]["main_tflops"] / peak, 4)
    roofline = {"bound": "alu" if simt_main else "tensor", "achieved": achieved, "peak": round(peak, 2),
                "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": per_kernel[big["name"]]["dram_bytes_per_launch"],
                "kernel": f"{kname}, {big['name']} launches",
                "peak_basis": ("nominal FP32 FMA: 152 SMs x 128 lanes x 2 flops x 2.07 GHz" if simt_main else
                               f"of {pk['source']}: burst bf16 x {TF32_OVER_BF16:.4f} (nominal tf32/bf16) / 3"),
                "frac_of_sustained_peak": round(achieved / pk["f32_3xtf32_tflops_sustained"], 4),
                "algorithmic_flops_per_launch": 2.0 * big["M"] * big["N"] * big["K"],
                "algorithmic_bytes_per_launch": algorithmic_bytes(big["M"], big["N"], big["K"]),
                "traffic_source": traffic_src, "kernel_source_sha256_16": kern_hash,
                "main_kernel_share_of_step": round(main_ms / ms_step, 4),
                "split_pass_share_of_step": round(split_ms / ms_step, 4),
                "per_shape": per_kernel}
    # The same fraction per clock: against the tensor pipe's dense TF32 rate at
    # the SM clock sampled in the timed region (2048 TF32 multiply-adds per SM
    # per clock, half of BF16's 4096, as the nominal dense peaks are; three
    # TF32 products per FP32 product).
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    if not simt_main and clk.get("sm_mhz"):
        per_clock = sms * 2 * 2048 / 3.0 * clk["sm_mhz"] * 1e6 / 1e12
        roofline["peak_per_clock"] = round(per_clock, 2)
        roofline["frac_per_clock"] = round(achieved / per_clock, 4)
        roofline["peak_per_clock_basis"] = (f"{sms} SMs x 2048 TF32 FMA/clk x 2 / 3 at the median SM clock "
                                            f"{clk['sm_mhz']:.0f} MHz of the timed region")
    launches = args.steps * sum(w["plan"].kernel_launches for w in work)

    # headline results kept for the comparison with the oracle (below, in the
    # CPU-baseline leg; nothing here runs the oracle)
    headline_parity = {}
    checks = []  # (where to record, captured result)
    if rank == 0 and not args.quick:
        for w in work:
            headline_parity[w["name"]] = {}
            checks.append((headline_parity[w["name"]], capture_for_check(w["A"], w["B"], w["dC"], full_limit=None)))

    # ---- e2e: through the C-ABI host-buffer call ------------------------------
    e2e = None
    if not args.no_e2e:
        hbufs = []
        for w in work:
            hA = torch.from_numpy(w["A"]).pin_memory()
            hB = torch.from_numpy(w["B"]).pin_memory()
            hC = torch.empty((w["M"], w["N"]), dtype=torch.float32).pin_memory()
            hbufs.append((w, hA, hB, hC))

        def e2e_step():
            for (w, hA, hB, hC) in hbufs:
                s = w["plan"].run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), sptr)
                if s != g.OK:
                    raise g.GemmError(s, "gemm_f32_run_host")
        for w in work:
            w["plan"].trace_enable(0)
        for _ in range(max(3, args.warmup)):
            e2e_step()
        n_e2e = max(10, args.steps // 5)
        if dist:
            dist.barrier()
        calls = []
        # the host-side timing runs with Python's cyclic garbage collector
        # paused (as timeit does): a collection inside a call is host noise
        gc_was = gc.isenabled()
        gc.disable()
        try:
            for _ in range(n_e2e):
                t0 = time.perf_counter()
                e2e_step()  # synchronous: the call copies C back and synchronises
                calls.append(time.perf_counter() - t0)
        finally:
            if gc_was:
                gc.enable()
        # The median call: a host-side stall of one call (seen once at 39 ms
        # against 5.5 ms for the others) does not stand for the pipeline; the
        # mean is reported beside it.
        dt = max_over_ranks(statistics.median(calls), dist, "cuda")
        e2e = {"value": round(whole_job_rate(flops_step, world, dt), 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(4 * (w["M"] * w["K"] + w["K"] * w["N"]) for w in work)),
               "d2h_bytes_per_step": int(sum(4 * w["M"] * w["N"] for w in work)),
               "ms_per_step": round(dt * 1e3, 3), "statistic": f"median of {n_e2e} calls", "steps": n_e2e,
               "ms_min": round(min(calls) * 1e3, 3), "ms_median": round(statistics.median(calls) * 1e3, 3),
               "ms_mean": round(sum(calls) / n_e2e * 1e3, 3), "ms_max": round(max(calls) * 1e3, 3),
               "ms_calls": [round(c * 1e3, 2) for c in calls],
               "call": "gemm_f32_run_host (pinned host A, B, C; copies and sync inside the call)"}
        del hbufs

    # ---- per shape: every configuration's shapes ----------------------------
    per_shape = None
    floors = None
    batched = None
    if rank == 0 and not args.no_per_shape:
        per_shape = []
        cublas = None
        try:
            cublas = CublasCompare()
        except (OSError, AttributeError, RuntimeError) as ex:
            cublas_note = f"cuBLAS comparison unavailable: {ex}"
        else:
            cublas_note = (f"cuBLAS {cublas.version}, FP32 emulation (BF16x9, strategy EAGER) "
                           f"{'available' if cublas.emulation else 'not exposed'}" if cublas.ok else
                           f"cuBLAS comparison unavailable: {cublas.why}")
            if not cublas.ok:
                cublas = None
        from software_pipelined_gb300 import inputs
        # every shape's operands and plan, kept for all rounds
        cases = []
        for key in ("tiny_32", "small_ragged", "tall_skinny", "square_1024", "large_squares"):
            for (name, M, N, K, dist_name, sa, sb) in inputs.WORKLOADS[key]:
                if key == args.workload and not args.shape:
                    w = next(x for x in work if x["name"] == name)
                    A, B, dA, dB, dC, plan = w["A"], w["B"], w["dA"], w["dB"], w["dC"], w["plan"]
                    own = False
                else:
                    A, B, dA, dB, dC = make_device_operands(M, N, K, dist_name, sa, sb)
                    plan = g.Plan(M, N, K)
                    own = True
                cases.append(dict(key=key, name=name, M=M, N=N, K=K, A=A, B=B, dA=dA, dB=dB, dC=dC, plan=plan,
                                  own=own, rounds=[], lo=float("inf"), hi=0.0, reps=0))
        # rounds in rotated shape order (timing protocol of the comparison on
        # the pages: a shape's place in the sequence must not favour it);
        # each round: the median of 5 graph-replayed batches per shape
        ROUNDS = 3
        for r in range(ROUNDS):
            for i in range(len(cases)):
                c = cases[(i + r) % len(cases)]
                run_on = (lambda st, p=c["plan"], a=c["dA"], b=c["dB"], cc=c["dC"]:
                          p.run_ptr(a.data_ptr(), b.data_ptr(), cc.data_ptr(), st))
                med, lo, hi, reps = time_graph(run_on)
                c["rounds"].append(med)
                c["lo"], c["hi"], c["reps"] = min(c["lo"], lo), max(c["hi"], hi), reps
        flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")  # 256 MB > L2
        for c in cases:
            key, name, M, N, K = c["key"], c["name"], c["M"], c["N"], c["K"]
            A, B, dA, dB, dC, plan = c["A"], c["B"], c["dA"], c["dB"], c["dC"], c["plan"]
            run = (lambda p=plan, a=dA, b=dB, cc=dC: p.run_ptr(a.data_ptr(), b.data_ptr(), cc.data_ptr(), sptr))
            med = statistics.median(c["rounds"])
            s_med, _, _, _ = time_batches(run, stream)
            # phase breakdown of a few more runs (library-recorded events)
            plan.trace_enable(8)
            for _ in range(8):
                run()
            phases = plan.trace_read(8)
            plan.trace_enable(0)
            ph = [round(sum(r[i] for r in phases) / len(phases) * 1e3, 3) for i in range(3)]
            # cold L2 for the 1024^3 square: a 256 MB write between runs, outside the events
            cold = None
            if name == "1024x1024x1024":
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ts = []
                for _ in range(9):
                    flush.fill_(1.0)
                    ev0.record(stream)
                    run()
                    ev1.record(stream)
                    ev1.synchronize()
                    ts.append(ev0.elapsed_time(ev1))
                cold = round(statistics.median(ts) * 1e3, 3)
            fl = 2.0 * M * N * K
            byts = algorithmic_bytes(M, N, K)
            P = pk["f32_3xtf32_tflops_burst"]
            t_roof = max(fl / (P * 1e12), byts / (pk["hbm_gbs"] * 1e9))
            t_roof_simt = max(fl / (pk["f32_simt_tflops_nominal"] * 1e12), byts / (pk["hbm_gbs"] * 1e9))
            # comparison column, off the measured path: PyTorch's FP32 matmul
            # (cuBLAS SGEMM, TF32 disabled) timed the same way
            torch.backends.cuda.matmul.allow_tf32 = False
            dC2 = torch.empty_like(dC)
            cb, _, _, _ = time_graph(lambda st, a=dA, b=dB, cc=dC2: torch.mm(a, b, out=cc))
            # cuBLAS FP32 emulated with BF16 pieces and single TF32, same protocol
            emu = cublas.time("bf16x9", dA, dB, dC2, M, N, K) if cublas else None
            emu_chk = None
            if emu is not None and not args.quick and M * N * K <= 2 ** 31:
                emu_chk = capture_for_check(A, B, dC2)
            tf1 = cublas.time("tf32", dA, dB, dC2, M, N, K) if cublas else None
            del dC2
            entry = {
                "config": key, "shape": name, "plan": plan.describe(),
                "us": round(med * 1e3, 3), "us_min": round(c["lo"] * 1e3, 3), "us_max": round(c["hi"] * 1e3, 3),
                "us_rounds": [round(x * 1e3, 3) for x in c["rounds"]],
                "us_direct_launch": round(s_med * 1e3, 3),
                "torch_fp32_matmul_us": round(cb * 1e3, 3),
                "cublas_fp32_emulated_bf16x9_us": round(emu * 1e3, 3) if emu is not None else None,
                "cublas_tf32_us": round(tf1 * 1e3, 3) if tf1 is not None else None,
                "phases_us_split_main_reduce": ph,
                "tflops": round(fl / (med * 1e-3) / 1e12, 3),
                "roofline_frac": round(t_roof / (med * 1e-3), 4),
                "roofline_frac_vs_simt_peak": round(t_roof_simt / (med * 1e-3), 4),
                "max_normalised_error": None, "checked": None,  # filled by the CPU-baseline leg
                "l2": "warm (back-to-back)" if byts < 100e6 else "inputs larger than L2",
                "timing": (f"median of {ROUNDS} rounds (rotated shape order) of the median of 5 CUDA-graph "
                           "replays of back-to-back runs, events around each replay"),
                "runs_per_batch": c["reps"]}
            if cold is not None:
                entry["us_cold_l2"] = cold
            per_shape.append(entry)
            if emu_chk is not None:
                checks.append((entry, dict(emu_chk, field="cublas_bf16x9_max_normalised_error")))
            if not args.quick:
                # the headline shapes: the whole output (their oracle product is shared
                # with the headline check); the others up to 2^31 multiply-adds
                checks.append((entry, capture_for_check(A, B, dC, full_limit=None if not c["own"] else 2 ** 31)))
        del flush
        if cublas:
            cublas.close()
        for c in cases:
            if c["own"]:
                c["plan"].close()
        del cases
        # launch/event floors on this stream
        ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(50):
            ev_a.record(stream)
            ev_b.record(stream)
            ev_b.synchronize()
            ts.append(ev_a.elapsed_time(ev_b))
        z = torch.empty((1, 1), dtype=torch.float32, device="cuda")
        zp = g.Plan(1, 1, 0, 1, 1, 1)
        med, _, _, _ = time_batches(lambda: zp.run_ptr(0, 0, z.data_ptr(), sptr), stream)
        gmed, _, _, _ = time_graph(lambda st: zp.run_ptr(0, 0, z.data_ptr(), st))
        zp.close()
        batched = []
        for (bm, bn, bk, nb) in ((32, 32, 32, 1024), (128, 128, 128, 256), (64, 64, 64, 512)):
            from software_pipelined_gb300 import inputs as _in
            Ab = torch.from_numpy(_in.uniform_pm1(6001, nb * bm, bk)).cuda()
            Bb = torch.from_numpy(_in.uniform_pm1(6002, nb * bk, bn)).cuda()
            Cb = torch.empty((nb * bm, bn), dtype=torch.float32, device="cuda")
            with g.Plan(bm, bn, bk, bk, bn, bn, batch=nb, stride_a=bm * bk, stride_b=bk * bn,
                        stride_c=bm * bn) as bp:
                bmed, _, _, _ = time_graph(lambda st, p=bp: p.run_ptr(Ab.data_ptr(), Bb.data_ptr(),
                                                                       Cb.data_ptr(), st))
                bdesc = bp.describe()
            # the last product, kept for the comparison with the oracle
            last = {"A": Ab[(nb - 1) * bm:].cpu().numpy(), "B": Bb[(nb - 1) * bk:].cpu().numpy(),
                    "kind": "full", "C": Cb[(nb - 1) * bm:].cpu().numpy()}
            fl = 2.0 * bm * bn * bk * nb
            batched.append({"products": nb, "shape": f"{bm}x{bn}x{bk}", "plan": bdesc,
                            "us_per_launch": round(bmed * 1e3, 3),
                            "us_per_product": round(bmed * 1e3 / nb, 4),
                            "tflops": round(fl / (bmed * 1e-3) / 1e12, 3)})
            if not args.quick:
                checks.append((batched[-1], dict(last, field="max_normalised_error_last_product")))
            del Ab, Bb, Cb
        floors = {"event_pair_us": round(statistics.median(ts) * 1e3, 3),
                  "smallest_kernel_direct_launch_us": round(med * 1e3, 3),
                  "smallest_kernel_graph_us": round(gmed * 1e3, 3),
                  "note": "smallest kernel = this library's 1x1 zero-fill, back to back",
                  "comparison_columns": cublas_note}

    # ---- CPU-baseline leg: the oracle, on this host's cores ------------------
    # The only part of the GPU arm that runs the oracle: its throughput on a
    # bounded sample of the headline workload, its time beside each small
    # shape, and the comparison of every result kept above against it.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        big = max(work, key=lambda w: w["M"] * w["N"] * w["K"])
        tf, rows, dt, threads = oracle_sample(big["A"], big["B"], args.cpu_seconds)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"first {rows} rows of {big['name']} ({rows}x{big['N']}x{big['K']}), "
                         f"FP64 i-k-j triple loop, {dt:.1f} s"}
        products = {}
        for where, chk in checks:
            err, how = compare_with_oracle(chk, products)
            if "field" in chk:
                where[chk["field"]] = err
            else:
                where["max_normalised_error"], where["checked"] = err, how
            A, B = chk["A"], chk["B"]
            macs = A.shape[0] * B.shape[1] * A.shape[1]
            if "shape" in where and macs <= 1024 ** 3:
                # the oracle timed beside the GPU: median of 3, all cores; one core up to 512^3
                orc = {"ms_all_cores": round(time_oracle(A, B, 3) * 1e3, 3), "cores": threads}
                if macs <= 512 ** 3:
                    oracle.set_threads(1)
                    try:
                        orc["ms_one_core"] = round(time_oracle(A, B, 3) * 1e3, 3)
                    finally:
                        oracle.set_threads(threads)
                where["oracle"] = orc
        del products
    del checks

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64, uniform[-1,1))",
            "config": {"workload": ("large squares: 4096x4096x4096 + 8192x8192x8192 FP32 GEMM, row-major, "
                                    "tight leading dimensions, one GEMM of each per step") if not args.shape
                       else f"single shape {args.shape} FP32 GEMM, row-major, tight leading dimensions",
                       "shapes": [w["name"] for w in work],
                       "l2": "inputs larger than L2 (no flush needed)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "headline_parity": headline_parity, "per_shape": per_shape, "floors": floors,
            "batched": batched,
            "peaks": pk, "device": dev_name,
            "environment": run_environment(local),
            "library_sha256_16": source_hash([g.LIB_PATH]),
        }
        # last key, so that it survives in a tail of the output: per shape
        # [us, TFLOP/s, roofline fraction, max normalised error, plan]
        if per_shape:
            line["per_shape_summary"] = {e["shape"]: [e["us"], e["tflops"], e["roofline_frac"],
                                                      e["max_normalised_error"], plan_tag(e["plan"])]
                                         for e in per_shape}
        print(json.dumps(line), flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                json.dump(line, f, indent=1)
    for w in work:
        w["plan"].close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the same workload.
# ---------------------------------------------------------------------------

def plan_tag(desc):
    """A short form of a plan description: kernel, split form, tile, stages,
    split-K and tile order (drops sizes that follow from the shape)."""
    drop = ("terms=", "ws=", "kp=", "resident=", "whole=", "pairs=", "tiles=", "thread=")
    return " ".join(t for t in desc.split() if not t.startswith(drop) and t != "3xtf32")


def workload_label(workload):
    """What a workload is, with its sizes."""
    shapes = " + ".join(w[0] for w in shapes_of(workload))
    return ("large squares: " if workload == HEADLINE else workload.replace("_", " ") + ": ") + \
        f"{shapes} FP32 GEMM, row-major"


def run_reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from software_pipelined_gb300 import inputs
    oracle.build()
    big = max(shapes_of(args.workload), key=lambda w: w[1] * w[2] * w[3])
    name, M, N, K, dist_name, sa, sb = big
    A, B = inputs.make_operands(M, N, K, dist_name, sa, sb)
    threads = oracle.get_threads()
    # size one step so that warmup + steps take about --ref-seconds in all
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    _, rows, _, _ = oracle_sample(A, B, budget)
    for _ in range(args.warmup):
        oracle_rows_rate(A, B, rows)
    times = []
    fl = 0.0
    for _ in range(args.steps):
        dt, fl = oracle_rows_rate(A, B, rows)
        times.append(dt)
    dt = sum(times) / len(times)
    v = fl / dt / 1e12
    sample = f"first {rows} rows of {name} ({rows}x{N}x{K}) per step, FP64 i-k-j triple loop"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64, uniform[-1,1))",
            "config": {"workload": workload_label(args.workload), "sample": sample},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--shape", default=None, help="time one MxNxK shape instead of the workload")
    ap.add_argument("--variant", choices=["auto", "simt", "tcgen05"], default="auto",
                    help="kernel for the timed shapes (default: the dispatcher's choice)")
    ap.add_argument("--no-per-shape", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the parity checks inside the bench")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for warm-up + timed steps")
    ap.add_argument("--json-out", default=None)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
