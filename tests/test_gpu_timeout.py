"""Failure detection without a GPU fault: a bounded device wait that runs out.

The tensor-core kernel bounds every mbarrier wait.  The plan option
debug_withhold_stage makes its producer skip one pipeline fill, so the MMA
thread's wait on that stage's "full" barrier can never complete: it must give
up after wait_timeout_cycles, record the timeout in the plan's status word, and
every role must leave its loop, drain its copies and MMAs and free TMEM.  The
host sees GEMM_F32_ERR_TIMEOUT from gemm_f32_check, and the context stays
usable: a normal run afterwards gives the right answer.
"""
import numpy as np
import pytest

import oracle
import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_gb300 import build
    build.build()
    g.load()


@pytest.mark.parametrize("withhold", [1, 3])
def test_withheld_stage_times_out_and_context_survives(withhold):
    import torch
    M, N, K = 256, 256, 256
    A = inputs.uniform_pm1(1501, M, K)
    B = inputs.uniform_pm1(1502, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    # About 2^22 cycles (~2 ms): far above any legitimate wait of this small
    # problem (a whole tile's main loop is ~10^4 cycles), far below a hang.
    with g.Plan(M, N, K, variant=g.VARIANT_TCGEN05, tile_n=128, split_k=1,
                wait_timeout_cycles=1 << 22, debug_withhold_stage=withhold) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.ERR_TIMEOUT
        # the status word was cleared by the check
        assert p.check() == g.OK
    torch.cuda.synchronize()
    # The context is intact: a normal plan computes the right product.
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, variant=g.VARIANT_TCGEN05, tile_n=128) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


def test_short_timeout_does_not_fire_on_a_normal_run():
    import torch
    M, N, K = 512, 384, 1024
    A = inputs.normal(1503, M, K)
    B = inputs.normal(1504, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with g.Plan(M, N, K, variant=g.VARIANT_TCGEN05, wait_timeout_cycles=1 << 22) as p:
        for _ in range(3):
            p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


@pytest.mark.parametrize("mode", [1, 2], ids=["pre_pass", "in_kernel"])
def test_withheld_stage_in_a_cluster(mode):
    # Two K-slices of 3 and 2 k-blocks per tile, summed in a cluster of two.
    # Withholding fill 3 stops only the 3-block slice: its partner finishes,
    # offers its ring, waits for the other CTA's offer, and must give up after
    # the limit without sending anything.  Both CTAs then meet at the cluster's
    # closing barrier; the host sees TIMEOUT and the next run is right.
    import torch
    M, N, K = 256, 256, 160
    A = inputs.uniform_pm1(1505, M, K)
    B = inputs.uniform_pm1(1506, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    opts = dict(variant=g.VARIANT_TCGEN05, tile_n=128, split_k=2, operand_split=mode, split_reduce=2)
    with g.Plan(M, N, K, wait_timeout_cycles=1 << 22, debug_withhold_stage=3, **opts) as p:
        assert "cluster-sum" in p.describe()
        p.run(dA, dB, dC)
        assert p.check() == g.ERR_TIMEOUT
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, **opts) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


def test_withheld_stage_with_last_arriver_sum():
    # Slices of 3 and 2 k-blocks; the 3-block slice never arrives.  Its
    # partner counts its own arrival (not the last) and finishes; nobody sums
    # the tile.  The host sees TIMEOUT; the check clears the arrival counters,
    # and a normal plan afterwards is right.
    import torch
    M, N, K = 256, 256, 160
    A = inputs.uniform_pm1(1507, M, K)
    B = inputs.uniform_pm1(1508, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    opts = dict(variant=g.VARIANT_TCGEN05, tile_n=128, split_k=2, operand_split=1, split_reduce=3)
    with g.Plan(M, N, K, wait_timeout_cycles=1 << 22, debug_withhold_stage=3, **opts) as p:
        assert "last-arriver-sum" in p.describe()
        p.run(dA, dB, dC)
        assert p.check() == g.ERR_TIMEOUT
        assert p.check() == g.OK
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, **opts) as p:
        for _ in range(2):
            p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)
