"""The bench's multi-rank bookkeeping (replicas, one per GPU) on CPU with a
two-rank gloo process group: the job's step time is the slowest rank's and
the whole-job rate counts every rank's replica."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        worst = bench.max_over_ranks(ms, dist, "cpu")
        rate = bench.whole_job_rate(2.0e12, world, worst * 1e-3)
        dist.barrier()
        out[rank] = (worst, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_rate():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    worst, rate = out[0]
    assert worst == 15.0
    assert rate == pytest.approx(world * 2.0e12 / 0.015 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(1e12, 1, 1.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_quietly():
    # Under torchrun only rank 0 runs and prints the reference arm's line.
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_json_line():
    # The reference arm (the CPU oracle on this host's cores) prints one JSON
    # line with the contract's keys; a few seconds of work here (on the 1024^3
    # workload: the large squares' operands alone take minutes to page in on
    # some hosts).
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--ref-seconds", "3", "--workload", "square_1024"], env=env,
                       capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["unit"] == d["unit"]
    assert d["config"]["workload"].startswith("square 1024: 1024x1024x1024")
