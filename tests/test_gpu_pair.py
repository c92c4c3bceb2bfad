"""CTA pairs (tile_m = 256): one tcgen05.mma.cta_group::2 per 256 x BN tile.

Each CTA of the pair stages its own 128 rows of A and half of the tile's B
columns, converts them (3xTF32 split inside the kernel), and the even CTA's
MMA thread multiplies the pair's operands out of both CTAs' shared memory
into both CTAs' TMEM.  Checked against the FP64 oracle with the FP32 bound,
on ragged shapes (a pair's second tile row past M, partial B boxes past N, K
not a multiple of the stage depth), whole tiles and K-slices, several units
per pair, both stage depths and tile widths; exact on small integers;
deterministic; a withheld stage must time out on both CTAs and leave the
context usable.
"""
import numpy as np
import pytest

import oracle
import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

from gpu_util import check_against_oracle, run_gemm

pytestmark = pytest.mark.gpu

PAIR = dict(variant=g.VARIANT_TCGEN05, tile_m=256)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_gb300 import build
    build.build()
    g.load()


def _ldb(N):
    return N + (-N % 4)  # raw B rows by TMA: 16-byte aligned


CASES = [
    # M, N, K, tile_n, tile_k, split_k
    (512, 512, 256, 256, 32, 2),
    (512, 512, 256, 128, 32, 1),
    (300, 520, 264, 256, 32, 2),     # second tile row of the last pair past M; N and K ragged
    (300, 520, 264, 128, 16, 3),
    (1024, 1024, 1024, 256, 16, 4),  # the 1024^3 shape, 64 pairs
    (1024, 1024, 1024, 256, 32, 4),
    (1024, 1024, 1024, 128, 32, 2),
    (2048, 2048, 256, 128, 32, 1),   # 128 pair tiles: several units per pair, two accumulators
    (2048, 4096, 256, 256, 32, 1),   # 128 pair tiles of 256: both accumulators of 256 columns in turn
    (2304, 4096, 320, 256, 32, 0),   # 144 pair tiles: a partial last wave split automatically
    (130, 33, 96, 128, 32, 2),       # one pair, most of it past M and N
]
IDS = [f"{m}x{n}x{k}_bn{bn}_k{bk}_s{s}" for m, n, k, bn, bk, s in CASES]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_pair_matches_the_oracle(case):
    M, N, K, bn, bk, split = case
    A = inputs.uniform_pm1(2101, M, K)
    B = inputs.normal(2102, K, N)
    C, desc, canaries, outs = run_gemm(A, B, ldb=_ldb(N), repeat=2, tile_n=bn, tile_k=bk, split_k=split, **PAIR)
    assert "cta-pair" in desc and f"tile=256x{bn}x{bk}" in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


HYBRID_CASES = [
    # M, N, K, tile_n, split_k: B split by the pre-pass, only lo_A in the kernel
    (512, 512, 256, 256, 2),
    (300, 521, 264, 256, 2),      # ldb = 521: B needs no 16-byte rows here
    (1024, 1024, 1024, 256, 4),
    (2048, 2048, 256, 128, 1),    # several units per pair
    (2304, 4096, 320, 256, 0),    # partial last wave split automatically
]


@pytest.mark.parametrize("case", HYBRID_CASES, ids=[f"{m}x{n}x{k}_bn{bn}_s{s}" for m, n, k, bn, s in HYBRID_CASES])
def test_pair_hybrid_matches_the_oracle(case):
    M, N, K, bn, split = case
    A = inputs.uniform_pm1(2115, M, K)
    B = inputs.normal(2116, K, N)
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, tile_n=bn, split_k=split, operand_split=3, **PAIR)
    assert "hybrid-split cta-pair" in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


RAWA_CASES = [
    # M, N, K, tile_n, tile_k, split_k: lo of A and both pieces of B by the
    # pre-pass, hi of A the raw A; no conversion inside the kernel
    (512, 512, 256, 256, 32, 2),
    (300, 521, 264, 256, 32, 2),      # ldb = 521: B needs no 16-byte rows here
    (300, 520, 264, 256, 16, 3),      # half-size stages: 64-byte swizzled boxes of every piece
    (1024, 1024, 1024, 256, 16, 4),
    (1024, 1024, 1024, 256, 32, 4),
    (2048, 2048, 256, 128, 32, 1),    # several units per pair
    (2304, 4096, 320, 256, 32, 0),    # partial last wave split automatically
    (2304, 4096, 320, 256, 16, 0),
    (130, 33, 96, 128, 32, 2),        # one pair, most of it past M and N
]
RAWA_IDS = [f"{m}x{n}x{k}_bn{bn}_k{bk}_s{s}" for m, n, k, bn, bk, s in RAWA_CASES]


@pytest.mark.parametrize("case", RAWA_CASES, ids=RAWA_IDS)
def test_pair_raw_a_matches_the_oracle(case):
    M, N, K, bn, bk, split = case
    A = inputs.uniform_pm1(2121, M, K)
    B = inputs.normal(2122, K, N)
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, tile_n=bn, tile_k=bk, split_k=split, operand_split=4,
                                       **PAIR)
    assert "raw-a-split cta-pair" in desc and f"tile=256x{bn}x{bk}" in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


@pytest.mark.parametrize("bk", [32, 16])
def test_pair_raw_a_small_integers_padding_and_misaligned_fallback(bk):
    M, N, K = 520, 300, 200
    A = inputs.small_int(2123, M, K, -4, 4)
    B = inputs.small_int(2124, K, N, -4, 4)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    opts = dict(PAIR, tile_n=256, tile_k=bk, split_k=2, operand_split=4)
    C, desc, canaries, _ = run_gemm(A, B, **opts)
    assert "raw-a-split cta-pair" in desc and canaries and np.array_equal(C, exact), desc
    # padded rows of A (a multiple of 4), of B (any) and of C
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 8, ldb=N + 3, ldc=N + 5, **opts)
    assert canaries and np.array_equal(C, exact), desc
    # A's base off a 16-byte boundary: the one-CTA pre-pass form (its own maps)
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 4, a_off=1, **opts)
    assert canaries and np.array_equal(C, exact), desc


TMEMA_CASES = [
    # M, N, K, split_k: A split by the kernel's loader warps into tensor memory,
    # hi/lo of B by the pre-pass; 256x256 tiles, one accumulator per pair
    (512, 512, 256, 2),
    (300, 521, 264, 2),       # the second tile row past M; ldb = 521 (B needs no aligned rows)
    (1024, 1024, 1024, 4),
    (4096, 4096, 256, 0),     # 256 pair tiles: several units per pair through the one accumulator
    (2304, 4096, 320, 0),     # partial last wave split automatically
    (130, 33, 96, 2),         # one pair, most of it past M and N
    (640, 768, 1000, 3),      # K not a multiple of 32: the last k-block's tail is zeros
]
TMEMA_IDS = [f"{m}x{n}x{k}_s{s}" for m, n, k, s in TMEMA_CASES]
TMEMA = dict(PAIR, tile_n=256, tile_k=32, operand_split=5)


@pytest.mark.parametrize("case", TMEMA_CASES, ids=TMEMA_IDS)
def test_pair_tmem_a_matches_the_oracle(case):
    M, N, K, split = case
    A = inputs.uniform_pm1(2125, M, K)
    B = inputs.normal(2126, K, N)
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, split_k=split, **TMEMA)
    assert "tmem-a-split cta-pair" in desc and "tile=256x256x32" in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


def test_pair_tmem_a_small_integers_padding_and_misaligned_fallback():
    M, N, K = 520, 300, 200
    A = inputs.small_int(2127, M, K, -4, 4)
    B = inputs.small_int(2128, K, N, -4, 4)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    opts = dict(TMEMA, split_k=2)
    C, desc, canaries, _ = run_gemm(A, B, **opts)
    assert "tmem-a-split cta-pair" in desc and canaries and np.array_equal(C, exact), desc
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 8, ldb=N + 3, ldc=N + 5, **opts)
    assert canaries and np.array_equal(C, exact), desc
    # A's base off a 16-byte boundary: the one-CTA pre-pass form (its own maps)
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 4, a_off=1, **opts)
    assert canaries and np.array_equal(C, exact), desc


def test_pair_tmem_a_refusals_and_withheld_stage():
    import torch
    for kw in (dict(tile_n=128), dict(tile_k=16), dict(tile_m=128)):
        with pytest.raises(g.GemmError):
            g.Plan(512, 512, 512, **dict(TMEMA, **kw))
    with pytest.raises(g.GemmError):
        g.Plan(512, 512, 256, 257, 512, 512, **TMEMA)
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(2129, M, K)
    B = inputs.uniform_pm1(2130, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    for withhold in (1, 5):
        with g.Plan(M, N, K, split_k=2, wait_timeout_cycles=1 << 22, debug_withhold_stage=withhold, **TMEMA) as p:
            p.run(dA, dB, dC)
            assert p.check() == g.ERR_TIMEOUT
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, split_k=2, **TMEMA) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


def test_pair_hybrid_small_integers_and_misaligned_fallback():
    M, N, K = 520, 300, 200
    A = inputs.small_int(2117, M, K, -4, 4)
    B = inputs.small_int(2118, K, N, -4, 4)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    C, desc, canaries, _ = run_gemm(A, B, tile_n=256, split_k=2, operand_split=3, **PAIR)
    assert "hybrid-split cta-pair" in desc and canaries and np.array_equal(C, exact), desc
    # A's base off a 16-byte boundary: the one-CTA pre-pass form (its own B maps)
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 4, a_off=1, tile_n=256, split_k=2, operand_split=3, **PAIR)
    assert canaries and np.array_equal(C, exact), desc


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES[4]], ids=[IDS[0], IDS[3], IDS[4]])
def test_pair_small_integers_bit_exact(case):
    M, N, K, bn, bk, split = case
    A = inputs.small_int(2103, M, K, -4, 4)
    B = inputs.small_int(2104, K, N, -4, 4)
    C, desc, canaries, _ = run_gemm(A, B, ldb=_ldb(N), tile_n=bn, tile_k=bk, split_k=split, **PAIR)
    assert canaries
    assert np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64)), desc


def test_pair_padded_leading_dimensions_and_misaligned_fallback():
    M, N, K = 520, 300, 200
    A = inputs.uniform_pm1(2105, M, K)
    B = inputs.uniform_pm1(2106, K, N)
    # padded rows (multiples of 4): the pair kernel itself
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 8, ldb=N + 4, ldc=N + 3, tile_n=128, split_k=2, **PAIR)
    err, ok = check_against_oracle(C, A, B)
    assert "cta-pair" in desc and canaries and ok, f"{desc}: {err}"
    # A's base 4 bytes off a 16-byte boundary: the one-CTA pre-pass form runs instead
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 8, ldb=N + 4, a_off=1, tile_n=128, split_k=2, **PAIR)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("opts", [
    dict(operand_split=1), dict(stages=2), dict(separate_syncs=1), dict(split_reduce=3),
    dict(tile_n=64), dict(tile_k=64), dict(operand_split=3, tile_k=16), dict(operand_split=4, tile_n=128, tile_k=16),
], ids=["pre_pass", "stages", "separate_syncs", "last_arriver", "bn64", "tile_k64", "hybrid_k16", "raw_a_bn128_k16"])
def test_pair_refusals(opts):
    with pytest.raises(g.GemmError) as e:
        g.Plan(512, 512, 512, **dict(PAIR, **opts))
    assert e.value.status in (g.ERR_UNSUPPORTED, g.ERR_INVALID_ARG)


def test_pair_refuses_unaligned_leading_dimensions():
    # raw A by TMA needs 16-byte rows of A in every pair form; raw B by TMA (the
    # in-kernel split of B) needs them of B, the forms that pre-split B do not
    with pytest.raises(g.GemmError):
        g.Plan(512, 512, 256, 257, 512, 512, **PAIR)
    with pytest.raises(g.GemmError):
        g.Plan(512, 512, 256, 256, 514, 512, operand_split=2, **PAIR)
    with g.Plan(512, 512, 256, 256, 514, 512, **PAIR) as p:
        assert "hybrid-split cta-pair" in p.describe()


def test_pair_withheld_stage_times_out_and_context_survives():
    import torch
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(2107, M, K)
    B = inputs.uniform_pm1(2108, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    for withhold in (1, 3):
        with g.Plan(M, N, K, tile_n=256, split_k=2, wait_timeout_cycles=1 << 22, debug_withhold_stage=withhold,
                    **PAIR) as p:
            p.run(dA, dB, dC)
            assert p.check() == g.ERR_TIMEOUT
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, tile_n=256, split_k=2, **PAIR) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


def test_pair_raw_a_withheld_stage_times_out_and_context_survives():
    # Every piece by TMA, both CTAs' copies completing on the even CTA's
    # barrier: a fill withheld by both producers leaves that barrier short, the
    # MMA thread gives up after the limit, and the next run is right.
    import torch
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(2131, M, K)
    B = inputs.uniform_pm1(2132, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    opts = dict(PAIR, tile_n=256, split_k=2, operand_split=4)
    for withhold in (1, 3, 6):
        with g.Plan(M, N, K, wait_timeout_cycles=1 << 22, debug_withhold_stage=withhold, **opts) as p:
            assert "raw-a-split cta-pair" in p.describe()
            p.run(dA, dB, dC)
            assert p.check() == g.ERR_TIMEOUT
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    with g.Plan(M, N, K, **opts) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


GRIDSUM_CASES = [
    # (M, N, K, operand_split, split_k, tile_n): the grid's own slice sum
    (1024, 1024, 1024, 2, 4, 256),    # every pair tile in 4 slices, one unit per pair
    (4096, 4096, 256, 4, 0, 256),     # raw A: whole tiles, then the last wave's split tiles
    (300, 521, 264, 3, 2, 256),       # hybrid, ragged: the second tile row past M
    (640, 768, 1000, 2, 3, 128),      # K not a multiple of 32, 256x128 pair tiles
    (2560, 4096, 320, 4, 0, 256),     # several units per pair, the last wave split
]
GRIDSUM_IDS = [f"{m}x{n}x{k}_os{o}_s{s}_n{t}" for m, n, k, o, s, t in GRIDSUM_CASES]


@pytest.mark.parametrize("case", GRIDSUM_CASES, ids=GRIDSUM_IDS)
def test_pair_grid_sum_matches_the_reduction_kernel_bit_for_bit(case):
    # The grid sums the slices after a grid-wide barrier, in the reduction
    # kernel's order: the same bits as the reduction launch, within the bound,
    # and the same bits on a second run (the barrier resets itself).
    M, N, K, split, sk, tn = case
    A = inputs.uniform_pm1(2141, M, K)
    B = inputs.normal(2142, K, N)
    opts = dict(PAIR, tile_n=tn, split_k=sk, operand_split=split)
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, split_reduce=4, **opts)
    assert "grid-sum" in desc, desc
    Cr, desc_r, canaries_r, _ = run_gemm(A, B, split_reduce=1, **opts)
    assert "grid-sum" not in desc_r
    assert canaries and canaries_r
    assert np.array_equal(outs[0], outs[1]), desc
    assert np.array_equal(C, Cr), desc
    err, ok = check_against_oracle(C, A, B)
    assert ok, f"{desc}: {err}"


def test_pair_grid_sum_refusals_and_withheld_stage():
    import torch
    # one-CTA tiles and the tensor-memory form have no grid sum
    for kw in (dict(tile_m=128, operand_split=2), dict(tile_m=256, tile_n=256, operand_split=5)):
        with pytest.raises(g.GemmError):
            g.Plan(1024, 1024, 1024, variant=g.VARIANT_TCGEN05, split_k=4, split_reduce=4, **kw)
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(2143, M, K)
    B = inputs.uniform_pm1(2144, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    opts = dict(PAIR, tile_n=256, split_k=2, split_reduce=4)
    for split in (2, 4):
        for withhold in (1, 3):
            with g.Plan(M, N, K, wait_timeout_cycles=1 << 22, debug_withhold_stage=withhold, operand_split=split,
                        **opts) as p:
                assert "grid-sum" in p.describe()
                p.run(dA, dB, dC)
                # the stalled pair gives up and still meets the grid barrier
                assert p.check() == g.ERR_TIMEOUT
        torch.cuda.synchronize()
        dC.fill_(float("nan"))
        with g.Plan(M, N, K, operand_split=split, **opts) as p:
            for _ in range(2):
                p.run(dA, dB, dC)
                assert p.check() == g.OK
        Cref, S = oracle.gemm_f64(A, B)
        assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


def test_pair_launch_count_and_host_run():
    import torch
    M, N, K = 1024, 1024, 1024
    A = inputs.uniform_pm1(2109, M, K)
    B = inputs.uniform_pm1(2110, K, N)
    with g.Plan(M, N, K, tile_n=256, split_k=4, **PAIR) as p:
        assert g.gemm_f32_plan_kernel_launches(p.handle) == 2  # the pair kernel and the reduction
        hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
        hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
        assert p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0) == g.OK
    err, ok = check_against_oracle(hC.numpy().astype(np.float64), A, B)
    assert ok, err


# ---------------------------------------------------------------------------
# K-slices of a pair tile summed inside a cluster of S pairs (split_reduce 2):
# the slices' order of the reduction kernel, so the same bits.
# ---------------------------------------------------------------------------

CLUSTER_CASES = [
    # M, N, K, tile_n, tile_k, split_k
    (1024, 1024, 1024, 256, 32, 4),  # the 1024^3 plan: 16 clusters of 8 CTAs
    (1024, 1024, 1024, 256, 16, 4),
    (512, 512, 512, 128, 32, 2),     # clusters of 4
    (300, 520, 264, 256, 32, 2),     # ragged: quadrants past M, a tile column past N
    (520, 300, 200, 128, 16, 4),
]
CLUSTER_IDS = [f"{m}x{n}x{k}_bn{bn}_k{bk}_s{s}" for m, n, k, bn, bk, s in CLUSTER_CASES]


@pytest.mark.parametrize("case", CLUSTER_CASES, ids=CLUSTER_IDS)
def test_pair_cluster_sum_matches_reduction_kernel(case):
    M, N, K, bn, bk, split = case
    A = inputs.uniform_pm1(2111, M, K)
    B = inputs.normal(2112, K, N)
    opts = dict(PAIR, tile_n=bn, tile_k=bk, split_k=split)
    Cc, dc, okc, runs = run_gemm(A, B, ldb=_ldb(N), repeat=2, split_reduce=2, **opts)
    Ck, dk, okk, _ = run_gemm(A, B, ldb=_ldb(N), split_reduce=1, **opts)
    assert "cluster-sum" in dc and "cluster-sum" not in dk, dc
    assert okc and okk
    assert np.array_equal(runs[0], runs[1]), dc
    assert np.array_equal(Cc, Ck), dc
    err, ok = check_against_oracle(Cc, A, B)
    assert ok, f"{dc}: {err}"


def test_pair_cluster_sum_launch_count_and_refusals():
    with g.Plan(1024, 1024, 1024, tile_n=256, split_k=4, split_reduce=2, **PAIR) as p:
        assert g.gemm_f32_plan_kernel_launches(p.handle) == 1  # no reduction kernel
    for kw in (dict(split_k=3), dict(split_k=1), dict(split_k=0)):
        with pytest.raises(g.GemmError):
            g.Plan(2048, 2048, 1024, tile_n=256, split_reduce=2, **dict(PAIR, **kw))


def test_pair_cluster_sum_withheld_stage_times_out():
    import torch
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(2113, M, K)
    B = inputs.uniform_pm1(2114, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with g.Plan(M, N, K, tile_n=256, split_k=2, split_reduce=2, wait_timeout_cycles=1 << 22,
                debug_withhold_stage=2, **PAIR) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.ERR_TIMEOUT
    torch.cuda.synchronize()
    with g.Plan(M, N, K, tile_n=256, split_k=2, split_reduce=2, **PAIR) as p:
        p.run(dA, dB, dC)
        assert p.check() == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(dC.cpu().numpy(), Cref, S, K)


@pytest.mark.parametrize("mode", [2, 3, 4, 5], ids=["in_kernel", "hybrid", "raw_a", "tmem_a"])
def test_pair_run_host_blocks_ragged_with_splits(mode):
    # Ragged M and N (the last panel's second tile row and the last block's
    # columns past the edge), K-slices in every panel's last wave, padded C:
    # the bound, and the padding untouched.
    import torch
    M, N, K, ldc = 1300, 1100, 300, 1107
    A = inputs.uniform_pm1(2131, M, K)
    B = inputs.uniform_pm1(2132, K, N)
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.full((M, ldc), 321.0, dtype=torch.float32).pin_memory()
    with g.Plan(M, N, K, K, N, ldc, host_panels=3, host_col_blocks=3, tile_n=256, operand_split=mode,
                **PAIR) as p:
        for _ in range(2):
            hC[:, :N] = float("nan")
            assert p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0) == g.OK
            C = hC.numpy()
            err, ok = check_against_oracle(C[:, :N].astype(np.float64), A, B)
            assert ok, f"{p.describe()}: {err}"
            assert (C[:, N:] == 321.0).all()


def test_pair_run_host_first_panel_of_two_shares_bit_identical_to_device_run():
    # A GEMM of 8 waves or more with column blocks: the first row panel takes
    # two shares of the tile rows (8192 x 8192: 12 pair-rows, then 4 panels of
    # 5).  Without a K-split the panel pipeline reproduces the device run bit
    # for bit.
    import torch
    M, N, K = 8192, 8192, 64
    A = inputs.normal(2161, M, K)
    B = inputs.normal(2162, K, N)
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    opts = dict(PAIR, tile_n=256, split_k=1, operand_split=4)
    with g.Plan(M, N, K, host_panels=5, host_col_blocks=3, **opts) as p:
        for _ in range(2):
            assert p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0) == g.OK
    C, desc, canaries, _ = run_gemm(A, B, host_panels=1, **opts)
    assert canaries
    assert np.array_equal(hC.numpy().astype(np.float64), C), desc


@pytest.mark.parametrize("mode", [2, 3, 4, 5], ids=["in_kernel", "hybrid", "raw_a", "tmem_a"])
@pytest.mark.parametrize("panels,cols", [(2, 1), (3, 1), (3, 2), (2, 3)])
def test_pair_run_host_panels_bit_identical_to_device_run(mode, panels, cols):
    # Without a K-split every tile is summed in the same order whichever 256-row
    # panel (or column block of the first panel) it falls in: the panel
    # pipeline must reproduce the device run bit for bit (a wrong panel or
    # block offset cannot hide in the bound).
    import torch
    M, N, K = 1536, 768, 320
    A = inputs.normal(2119, M, K)
    B = inputs.normal(2120, K, N)
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    opts = dict(PAIR, tile_n=256, split_k=1, operand_split=mode)
    with g.Plan(M, N, K, host_panels=panels, host_col_blocks=cols, **opts) as p:
        assert p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0) == g.OK
    C, desc, canaries, _ = run_gemm(A, B, host_panels=1, **opts)
    assert canaries
    assert np.array_equal(hC.numpy().astype(np.float64), C), desc
