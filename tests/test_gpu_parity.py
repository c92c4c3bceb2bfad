"""GPU parity: every kernel path against the CPU oracle, element by element.

Criterion (FP32-level accuracy of the tiled GEMM; the FP64-oracle check of
"Dependence-aware group synchronization on M1 Max", section "Controlled
implementation comparison"):

    |C_gpu - C_oracle| <= 2 * K * 2^-24 * sum_k |A_ik| |B_kj|   for every element,

reported as the maximum normalised error (pass iff <= 2).  Small-integer inputs
make every partial sum exact in FP32, TF32 and FP64, so there the GPU must be
bit-exact.  C starts as NaN inside a sentinel-filled margin: every element must
be written and nothing outside C may be.
"""
import numpy as np
import pytest

import oracle
import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

from gpu_util import check_against_oracle, run_gemm

pytestmark = pytest.mark.gpu

AUTO, SIMT, TC = {}, {"variant": g.VARIANT_SIMT}, {"variant": g.VARIANT_TCGEN05}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_gb300 import build
    build.build()
    g.load()


def _operands(M, N, K, dist, sa, sb, lda=None, ldb=None):
    return inputs.make_operands(M, N, K, dist, sa, sb)


BENCH_SHAPES = [w for key in ("tiny_32", "small_ragged", "tall_skinny", "square_1024")
                for w in inputs.WORKLOADS[key]]


@pytest.mark.parametrize("variant", [AUTO, SIMT, TC], ids=["auto", "simt", "tcgen05"])
@pytest.mark.parametrize("w", BENCH_SHAPES, ids=[w[0] for w in BENCH_SHAPES])
def test_benchmark_shapes_full_output(w, variant):
    name, M, N, K, dist, sa, sb = w
    A, B = _operands(M, N, K, dist, sa, sb)
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries, desc
    assert ok, f"{name} {desc}: max normalised error {err}"


@pytest.mark.parametrize("w", BENCH_SHAPES, ids=[w[0] for w in BENCH_SHAPES])
def test_forced_tiles_on_table_shapes(w):
    # A shape the dispatch table lists, with forced tile/stage options: the
    # table's own K-tile depth and tile order must not leak into the override.
    name, M, N, K, dist, sa, sb = w
    A, B = _operands(M, N, K, dist, sa, sb)
    for kw in (dict(variant=g.VARIANT_SIMT, tile_m=128, tile_n=128, stages=2),
               dict(variant=g.VARIANT_SIMT, tile_m=64, tile_n=64, stages=3)):
        C, desc, canaries, _ = run_gemm(A, B, **kw)
        err, ok = check_against_oracle(C, A, B)
        assert canaries and ok, f"{name} {desc}: {err}"


EDGE = [
    (1, 1, 1), (1, 37, 19), (41, 1, 23), (17, 29, 1), (33, 65, 5), (130, 260, 33),
    (257, 129, 257), (64, 64, 64), (128, 256, 96), (255, 513, 100), (300, 200, 1000),
]


@pytest.mark.parametrize("variant", [SIMT, TC], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("shape", EDGE, ids=[f"{m}x{n}x{k}" for m, n, k in EDGE])
def test_edge_shapes(shape, variant):
    M, N, K = shape
    A = inputs.uniform_pm1(700 + M, M, K)
    B = inputs.normal(800 + N, K, N)
    if variant is TC and K < 16:
        # The 3xTF32 split cannot meet the bound for such short sums: refused.
        with pytest.raises(g.GemmError) as ei:
            g.Plan(M, N, K, variant=g.VARIANT_TCGEN05)
        assert ei.value.status == g.ERR_UNSUPPORTED
        return
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries, desc
    assert ok, f"{shape} {desc}: {err}"


@pytest.mark.parametrize("variant", [SIMT, TC], ids=["simt", "tcgen05"])
def test_padded_leading_dimensions(variant):
    M, N, K = 150, 170, 90
    A = inputs.uniform_pm1(901, M, K)
    B = inputs.uniform_pm1(902, K, N)
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 3, ldb=N + 5, ldc=N + 7, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("variant", [SIMT, TC], ids=["simt", "tcgen05"])
def test_unaligned_base_pointers(variant):
    # Base addresses 4 bytes past a 16-byte boundary: no 16-byte vector path applies.
    M, N, K = 131, 67, 45
    A = inputs.uniform_pm1(911, M, K)
    B = inputs.uniform_pm1(912, K, N)
    C, desc, canaries, _ = run_gemm(A, B, a_off=1, b_off=1, c_off=1, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("variant", [SIMT, TC, {"variant": g.VARIANT_SIMT, "split_k": 4},
                                     {"variant": g.VARIANT_TCGEN05, "split_k": 3}],
                         ids=["simt", "tcgen05", "simt_splitk4", "tcgen05_splitk3"])
def test_small_integers_bit_exact(variant):
    # Entries in [-8, 8], K = 1000: every partial sum is an integer below 2^24,
    # exact in FP32; the hi/lo split of an integer this small is (x, 0).
    M, N, K = 200, 300, 1000
    A = inputs.small_int(921, M, K)
    B = inputs.small_int(922, K, N)
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    Cref, _ = oracle.gemm_f64(A, B)
    assert canaries
    assert np.array_equal(C, Cref), desc


@pytest.mark.parametrize("variant", [AUTO, {"variant": g.VARIANT_SIMT, "split_k": 5},
                                     {"variant": g.VARIANT_TCGEN05, "split_k": 4}],
                         ids=["auto", "simt_splitk5", "tcgen05_splitk4"])
def test_deterministic_repeat(variant):
    M, N, K = 384, 320, 2048
    A = inputs.uniform_pm1(931, M, K)
    B = inputs.uniform_pm1(932, K, N)
    C, desc, _, outs = run_gemm(A, B, repeat=3, **variant)
    assert all(np.array_equal(outs[0], o) for o in outs[1:]), desc
    err, ok = check_against_oracle(C, A, B)
    assert ok, f"{desc}: {err}"


def test_k_zero_writes_zeros():
    A = np.zeros((37, 0), dtype=np.float32)
    B = np.zeros((0, 53), dtype=np.float32)
    C, desc, canaries, _ = run_gemm(A, B, lda=1, ldb=53)
    assert canaries and desc.startswith("zero-fill")
    assert not C.any()


def test_single_tf32_negative_control_fails_the_bound():
    # One TF32 product per k (no compensation terms) must miss the bound; the
    # 3xTF32 run of the same inputs must meet it: the criterion has teeth.
    # With random signs the rounding errors of a single TF32 product grow like
    # sqrt(K) while the bound grows like K*sum|a||b| ~ K^2, so the control is
    # taken at small K (32), where one TF32 product is far outside the bound.
    M, N, K = 256, 256, 32
    A = inputs.uniform_pm1(941, M, K)
    B = inputs.uniform_pm1(942, K, N)
    C1, _, _, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05, tf32_terms=1)
    C3, _, _, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05)
    e1, ok1 = check_against_oracle(C1, A, B)
    e3, ok3 = check_against_oracle(C3, A, B)
    assert not ok1 and e1 > 4, e1
    assert ok3, e3


def test_3xtf32_accuracy_matches_fp32_simt():
    # At K = 4096 the 3xTF32 result is as accurate as plain FP32 FFMA: its
    # maximum normalised error is within a small factor of the SIMT kernel's.
    M, N, K = 256, 256, 4096
    A = inputs.uniform_pm1(943, M, K)
    B = inputs.uniform_pm1(944, K, N)
    Ct, _, _, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05)
    Cs, _, _, _ = run_gemm(A, B, variant=g.VARIANT_SIMT)
    et, okt = check_against_oracle(Ct, A, B)
    es, oks = check_against_oracle(Cs, A, B)
    assert okt and oks
    assert et <= 3 * es + 1e-3, (et, es)


# (tile_m, tile_n, stages, separate barriers, tile_k); 0 = the default K-tile
SIMT_CFGS = [(128, 128, 2, 0, 0), (128, 128, 3, 0, 0), (128, 128, 1, 0, 0), (64, 64, 2, 0, 0),
             (64, 64, 3, 0, 0), (64, 64, 1, 0, 0), (64, 64, 2, 0, 32), (32, 32, 2, 0, 0), (32, 32, 1, 0, 0),
             (128, 64, 2, 0, 0), (32, 32, 3, 0, 0), (32, 32, 1, 0, 64), (32, 32, 2, 0, 64), (32, 64, 2, 0, 0),
             (64, 32, 2, 0, 0),
             (128, 128, 2, 1, 0), (128, 128, 1, 1, 0), (64, 64, 2, 1, 0), (64, 64, 1, 1, 0), (32, 32, 2, 1, 0),
             (32, 32, 1, 1, 0)]


@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "unaligned"])
@pytest.mark.parametrize("cfg", SIMT_CFGS,
                         ids=[f"{a}x{b}s{c}{'sep' if d else ''}k{e}" for a, b, c, d, e in SIMT_CFGS])
def test_every_simt_config(cfg, aligned):
    # separate barriers for A and B: the barrier-coalescing ablation
    bm, bn, st, sep, bk = cfg
    M, N, K = 3 * bm + 5, 2 * bn + 3, 97
    A = inputs.uniform_pm1(951, M, K)
    B = inputs.uniform_pm1(952, K, N)
    kw = {} if aligned else dict(lda=K + 1, ldb=N + 2, a_off=1, b_off=1)
    C, desc, canaries, _ = run_gemm(A, B, variant=g.VARIANT_SIMT, tile_m=bm, tile_n=bn, stages=st,
                                    separate_syncs=sep, tile_k=bk, **kw)
    assert ("separate-syncs" in desc) == bool(sep), desc
    assert f"tile={bm}x{bn}x" in desc and (bk == 0 or f"x{bk} " in desc), desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


# K split inside the CTA: (tile_m, tile_n, stages, tile_k, k_slices)
SIMT_KSL_CFGS = [(64, 64, 3, 16, 2), (64, 64, 2, 16, 2), (64, 64, 2, 32, 2), (64, 64, 2, 32, 4),
                 (32, 32, 1, 64, 4), (32, 32, 2, 64, 4), (32, 32, 2, 32, 2), (32, 32, 2, 32, 4),
                 (32, 64, 2, 32, 2), (64, 32, 2, 32, 2), (32, 32, 3, 32, 4), (32, 32, 4, 32, 4),
                 (32, 32, 3, 64, 4), (64, 64, 4, 16, 2), (32, 64, 3, 32, 2), (64, 32, 3, 32, 2)]


@pytest.mark.parametrize("shape", [(512, 512, 512), (1024, 1024, 1024), (4096, 4096, 4096)])
@pytest.mark.parametrize("stages", [1, 2])
def test_forced_stages_select_the_pre_pass_form(shape, stages):
    # the table picks in-kernel or raw-A splits (fixed depth) for these shapes;
    # a forced depth must give that depth, in the pre-pass form
    bn = 256 if stages == 1 else 128
    with g.Plan(*shape, variant=g.VARIANT_TCGEN05, tile_n=bn, stages=stages) as p:
        d = p.describe()
    assert f"stages={stages}" in d and "in-kernel" not in d and "raw-a" not in d and "hybrid" not in d, d


@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "unaligned"])
@pytest.mark.parametrize("cfg", SIMT_KSL_CFGS, ids=[f"{a}x{b}x{d}s{c}ksl{e}" for a, b, c, d, e in SIMT_KSL_CFGS])
def test_every_sliced_k_simt_config(cfg, aligned):
    bm, bn, st, bk, ksl = cfg
    # ragged in M, N and K (K not a multiple of the tile, so the last tile's
    # slices are partly or wholly zero-filled), with and without split-K
    M, N, K = 2 * bm + 5, 3 * bn + 3, 3 * bk + 7
    A = inputs.uniform_pm1(953, M, K)
    B = inputs.uniform_pm1(954, K, N)
    kw = {} if aligned else dict(lda=K + 1, ldb=N + 2, a_off=1, b_off=1)
    for split in (1, 2):
        C, desc, canaries, runs = run_gemm(A, B, variant=g.VARIANT_SIMT, tile_m=bm, tile_n=bn, stages=st,
                                           tile_k=bk, k_slices=ksl, split_k=split, repeat=2, **kw)
        assert f"k_slices={ksl}" in desc and f"tile={bm}x{bn}x{bk}" in desc, desc
        assert np.array_equal(runs[0], runs[1]), "not deterministic"
        err, ok = check_against_oracle(C, A, B)
        assert canaries and ok, f"{desc}: {err}"


def test_sliced_k_small_integers_bit_exact():
    M, N, K = 70, 90, 200
    A = inputs.small_int(955, M, K)
    B = inputs.small_int(956, K, N)
    C, desc, canaries, _ = run_gemm(A, B, variant=g.VARIANT_SIMT, tile_m=32, tile_n=32, stages=2, tile_k=64,
                                    k_slices=4)
    assert canaries and np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64)), desc


def test_sliced_k_refusals():
    for opts in (dict(k_slices=3), dict(tile_m=128, tile_n=128, stages=2, k_slices=2)):
        with pytest.raises(g.GemmError):
            g.Plan(256, 256, 256, variant=g.VARIANT_SIMT, **opts)


# Fragments handed out by warp shuffles (the fragment-load ablation): the same
# FFMAs in the same order as the broadcast loads, so the same bits.
# (tile_m, tile_n, stages, tile_k, k_slices)
SHFL_CFGS = [(128, 128, 2, 16, 1), (64, 64, 2, 16, 1), (64, 64, 4, 16, 2), (32, 32, 3, 32, 4), (32, 32, 3, 64, 4)]


@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "unaligned"])
@pytest.mark.parametrize("cfg", SHFL_CFGS, ids=[f"{a}x{b}x{d}s{c}ksl{e}" for a, b, c, d, e in SHFL_CFGS])
def test_shuffle_fragments_bit_identical_to_broadcast(cfg, aligned):
    bm, bn, st, bk, ksl = cfg
    M, N, K = 2 * bm + 5, 3 * bn + 3, 3 * bk + 7
    A = inputs.uniform_pm1(957, M, K)
    B = inputs.uniform_pm1(958, K, N)
    kw = {} if aligned else dict(lda=K + 1, ldb=N + 2, a_off=1, b_off=1)
    opts = dict(variant=g.VARIANT_SIMT, tile_m=bm, tile_n=bn, stages=st, tile_k=bk, k_slices=ksl, **kw)
    Cs, ds, oks, _ = run_gemm(A, B, simt_fragments=1, **opts)
    Cb, db, okb, _ = run_gemm(A, B, **opts)
    assert "shuffle-fragments" in ds and "shuffle-fragments" not in db, ds
    assert oks and okb
    assert np.array_equal(Cs, Cb), ds
    err, ok = check_against_oracle(Cs, A, B)
    assert ok, f"{ds}: {err}"


def test_shuffle_fragments_refused_where_not_compiled():
    with pytest.raises(g.GemmError) as e:
        g.Plan(256, 256, 256, variant=g.VARIANT_SIMT, tile_m=64, tile_n=32, stages=2, simt_fragments=1)
    assert e.value.status == g.ERR_UNSUPPORTED
    with pytest.raises(g.GemmError) as e:
        g.Plan(256, 256, 256, variant=g.VARIANT_SIMT, simt_fragments=2)
    assert e.value.status == g.ERR_INVALID_ARG


TC_CFGS = [(128, 3, 0), (256, 2, 0), (64, 4, 0), (256, 1, 0), (128, 1, 0), (128, 2, 0), (64, 2, 0),
           (256, 2, 1), (128, 3, 1)]


@pytest.mark.parametrize("cfg", TC_CFGS, ids=[f"n{a}s{b}{'sep' if c else ''}" for a, b, c in TC_CFGS])
@pytest.mark.parametrize("split", [1, 2])
def test_every_tcgen05_config(cfg, split):
    bn, st, sep = cfg
    # Several M and N tiles plus a ragged edge, and more k-blocks than stages so
    # every ring slot is reused across the loop back-edge.
    M, N, K = 2 * 128 + 17, 3 * bn + 9, 32 * 11 + 7
    A = inputs.uniform_pm1(961, M, K)
    B = inputs.normal(962, K, N)
    C, desc, canaries, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05, tile_n=bn, stages=st, split_k=split,
                                    separate_syncs=sep)
    assert f"stages={st}" in desc and ("separate-syncs" in desc) == bool(sep), desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


def test_persistent_many_tiles_per_cta():
    # More output tiles than SMs: each CTA loops over several tiles and both
    # TMEM accumulator buffers are reused.
    M, N, K = 128 * 20, 128 * 17, 64
    A = inputs.uniform_pm1(971, M, K)
    B = inputs.uniform_pm1(972, K, N)
    C, desc, canaries, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05, tile_n=128, split_k=1)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("opts", [dict(tile_m=128, tile_n=128), dict(tile_m=256, tile_n=256)],
                         ids=["one_cta_128", "pair_256"])
def test_reduction_larger_than_one_grid(opts):
    # Every tile split: more float4 of partial tiles to sum (4096 x 2048 x 2
    # slices, about 2.1 M per slice set) than the reduction's grid has threads
    # (152 SMs x 64 blocks x 192), so its threads take several float4 each.
    M, N, K = 4096, 2048 + 40, 256
    A = inputs.uniform_pm1(983, M, K)
    B = inputs.uniform_pm1(984, K, N)
    C, desc, canaries, outs = run_gemm(A, B, ldb=N + (-N % 4), repeat=2, variant=g.VARIANT_TCGEN05, split_k=2,
                                       **opts)
    assert "whole=0" in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


@pytest.mark.parametrize("shape,bn", [((128 * 20, 128 * 17, 1024), 128), ((128 * 33, 256 * 9 + 40, 640), 256)],
                         ids=["bn128", "bn256_ragged"])
def test_tail_wave_split(shape, bn):
    # More tiles than SMs with a partial last wave: the dispatcher's automatic
    # policy computes those tiles in K-slices (dense partial tiles + fixed-order
    # reduction); the result must meet the bound and be deterministic.
    M, N, K = shape
    A = inputs.uniform_pm1(981, M, K)
    B = inputs.uniform_pm1(982, K, N)
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=bn)
    assert "split=0x" not in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


@pytest.mark.parametrize("w", inputs.WORKLOADS["large_squares"], ids=lambda w: w[0])
def test_large_squares_full_output(w):
    # The launch configuration the bench times (the dispatcher's plan), every
    # element of C against the oracle (at 8192^3 about 15 s of oracle on 16
    # host cores and 1 GB of FP64 C and S).
    name, M, N, K, dist, sa, sb = w
    A, B = _operands(M, N, K, dist, sa, sb)
    C, desc, canaries, _ = run_gemm(A, B)
    assert canaries
    assert np.isfinite(C).all(), desc
    Cref, S = oracle.gemm_f64(A, B)
    del A, B
    err = oracle.normalised_error(C, Cref, S, K)
    assert err <= 2.0, f"{name} {desc}: {err}"


# ---------------------------------------------------------------------------
# Operands split inside the tensor-core kernel (raw A and B by TMA).
# ---------------------------------------------------------------------------

FUSED = {"variant": g.VARIANT_TCGEN05, "operand_split": 2}
FUSED16 = {"variant": g.VARIANT_TCGEN05, "operand_split": 2, "tile_k": 16}
HYBRID = {"variant": g.VARIANT_TCGEN05, "operand_split": 3}
RAWA = {"variant": g.VARIANT_TCGEN05, "operand_split": 4}
MODES = [(FUSED, "in-kernel-split"), (FUSED16, "in-kernel-split"), (HYBRID, "hybrid-split"),
         (RAWA, "raw-a-split")]
MODE_IDS = ["in_kernel", "in_kernel_k16", "hybrid", "raw_a"]


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("split", [1, 2, 0])
def test_in_kernel_split_configs(bn, split, mode):
    # Ragged M and N (last B box partly outside N), K not a multiple of 32, more
    # k-blocks than slots; split 0 = the dispatcher's split policy.
    opts, tag = mode
    M, N, K = 2 * 128 + 17, 3 * bn + 9, 32 * 11 + 4
    A = inputs.uniform_pm1(1601, M, K)
    B = inputs.normal(1602, K, N)
    # B's rows must be 16-byte aligned for the TMA copy of raw B: pad ldb
    ldb = N + (-N % 4) if opts in (FUSED, FUSED16) else N
    C, desc, canaries, outs = run_gemm(A, B, repeat=2, tile_n=bn, split_k=split, ldb=ldb, **opts)
    assert tag in desc, desc
    assert (f"tile=128x{bn}x16" in desc) == (opts is FUSED16), desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"
    assert np.array_equal(outs[0], outs[1]), desc


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_in_kernel_split_many_tiles_and_tail_wave(mode):
    M, N, K = 128 * 21, 256 * 9 + 68, 512
    A = inputs.uniform_pm1(1603, M, K)
    B = inputs.uniform_pm1(1604, K, N)
    C, desc, canaries, _ = run_gemm(A, B, tile_n=256, **mode[0])
    assert mode[1] in desc, desc
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_in_kernel_split_padded_and_misaligned_fallback(mode):
    # lda, ldb multiples of 4 (an in-kernel plan), but base pointers 4 bytes off
    # a 16-byte boundary: the run falls back to the pre-split kernel.
    M, N, K = 300, 260, 96
    A = inputs.uniform_pm1(1605, M, K)
    B = inputs.uniform_pm1(1606, K, N)
    for kw in (dict(lda=K + 4, ldb=N + 4, ldc=N + 3), dict(a_off=1, b_off=1, c_off=1),
               dict(b_off=1), dict(a_off=1)):
        C, desc, canaries, _ = run_gemm(A, B, **mode[0], **kw)
        assert mode[1] in desc
        err, ok = check_against_oracle(C, A, B)
        assert canaries and ok, f"{kw} {desc}: {err}"


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_in_kernel_split_small_integers_bit_exact(mode):
    M, N, K = 200, 300, 1000
    A = inputs.small_int(1607, M, K)
    B = inputs.small_int(1608, K, N)
    C, desc, canaries, _ = run_gemm(A, B, **mode[0])
    Cref, _ = oracle.gemm_f64(A, B)
    assert canaries and np.array_equal(C, Cref), desc


def test_in_kernel_split_refusals():
    with pytest.raises(g.GemmError) as ei:
        g.Plan(64, 64, 16, variant=g.VARIANT_TCGEN05, operand_split=2)      # K < 32
    assert ei.value.status == g.ERR_UNSUPPORTED
    with pytest.raises(g.GemmError) as ei:
        g.Plan(64, 64, 61, variant=g.VARIANT_TCGEN05, operand_split=2)      # lda = 61
    assert ei.value.status == g.ERR_UNSUPPORTED
    with pytest.raises(g.GemmError) as ei:
        g.Plan(64, 64, 64, variant=g.VARIANT_TCGEN05, operand_split=2, tile_n=64)  # no fused 64-wide
    assert ei.value.status == g.ERR_UNSUPPORTED
    for mode in (3, 4):
        with pytest.raises(g.GemmError) as ei:
            g.Plan(64, 64, 61, variant=g.VARIANT_TCGEN05, operand_split=mode)   # lda = 61
        assert ei.value.status == g.ERR_UNSUPPORTED
    with g.Plan(64, 61, 64, variant=g.VARIANT_TCGEN05, operand_split=4) as p:   # any ldb
        assert "raw-a-split" in p.describe()
    # hybrid takes any ldb
    with g.Plan(64, 61, 64, variant=g.VARIANT_TCGEN05, operand_split=3) as p:
        assert "hybrid-split" in p.describe()


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_in_kernel_split_negative_control(mode):
    M, N, K = 256, 256, 32
    A = inputs.uniform_pm1(1609, M, K)
    B = inputs.uniform_pm1(1610, K, N)
    C1, _, _, _ = run_gemm(A, B, tf32_terms=1, **mode[0])
    C3, _, _, _ = run_gemm(A, B, **mode[0])
    e1, ok1 = check_against_oracle(C1, A, B)
    e3, ok3 = check_against_oracle(C3, A, B)
    assert not ok1 and e1 > 4, e1
    assert ok3, e3


# ---------------------------------------------------------------------------
# Host-buffer entry point: copies in, product, copy out, synchronised.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("pad", [False, True], ids=["contiguous", "padded"])
@pytest.mark.parametrize("shape", [(300, 200, 96), (1024, 512, 640)], ids=["small", "tensor_core"])
def test_run_host_buffers(shape, pad):
    M, N, K = shape
    lda, ldb, ldc = (K + 3, N + 5, N + 7) if pad else (K, N, N)
    A = inputs.uniform_pm1(1701, M, K, ld=lda if pad else None)
    B = inputs.uniform_pm1(1702, K, N, ld=ldb if pad else None)
    Abuf = np.lib.stride_tricks.as_strided(A, shape=(M, lda), strides=(4 * lda, 4)) if pad else A
    Bbuf = np.lib.stride_tricks.as_strided(B, shape=(K, ldb), strides=(4 * ldb, 4)) if pad else B
    Cbuf = np.full((M, ldc), 321.0, dtype=np.float32)
    with g.Plan(M, N, K, lda, ldb, ldc) as p:
        for _ in range(2):
            s = p.run_host(Abuf.ctypes.data, Bbuf.ctypes.data, Cbuf.ctypes.data, 0)
            assert s == g.OK, g.gemm_f32_status_string(s)
    Cref, S = oracle.gemm_f64(np.ascontiguousarray(A), np.ascontiguousarray(B))
    assert oracle.within_bound(Cbuf[:, :N], Cref, S, K)
    if pad:
        assert (Cbuf[:, N:] == 321.0).all()


# ---------------------------------------------------------------------------
# The TMA-store epilogue of a CTA's last tile: 32-column boxes staged in two
# alternating buffers; tiles wider than the rest of C store only some boxes
# (one to seven of eight), the last one clipped.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("N", [8, 33, 64, 96, 100, 200])
def test_tma_store_epilogue_partial_boxes(N, bn):
    M, K = 200, 64
    A = inputs.uniform_pm1(1731, M, K)
    B = inputs.uniform_pm1(1732, K, N)
    C, desc, canaries, _ = run_gemm(A, B, variant=g.VARIANT_TCGEN05, tile_n=bn, split_k=1, ldc=N + 4 - N % 4)
    assert canaries, desc
    err, ok = check_against_oracle(C, A, B)
    assert ok, f"{desc}: {err}"


# ---------------------------------------------------------------------------
# K-slices summed inside a thread-block cluster (distributed shared memory)
# instead of by the reduction kernel: the same slice order, so the same bits.
# ---------------------------------------------------------------------------

CLUSTER_CASES = [
    # M, N, K, tile_n, split_k, operand_split
    (1024, 1024, 1024, 128, 2, 2),   # in-kernel split, the 1024^3 plan
    (512, 512, 512, 128, 4, 2),      # 4 slices, clusters of 4
    (1000, 520, 264, 128, 2, 1),     # ragged; slices of 5 and 4 k-blocks; pre-pass
    (500, 520, 256, 128, 4, 4),      # raw A, 4 slices
    (600, 700, 1024, 128, 2, 3),     # hybrid
    (384, 300, 640, 64, 4, 1),       # 128x64 tiles
    (256, 256, 160, 128, 2, 1),      # slices of 3 and 2 k-blocks
]


@pytest.mark.parametrize("case", CLUSTER_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_bn{c[3]}_s{c[4]}_m{c[5]}"
                                                     for c in CLUSTER_CASES])
def test_cluster_sum_matches_reduction_kernel(case):
    M, N, K, bn, split, mode = case
    A = inputs.uniform_pm1(1721, M, K)
    B = inputs.uniform_pm1(1722, K, N)
    opts = dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=bn, split_k=split, operand_split=mode)
    Cc, dc, okc, _ = run_gemm(A, B, split_reduce=2, **opts)
    Ck, dk, okk, _ = run_gemm(A, B, split_reduce=1, **opts)
    assert "cluster-sum" in dc and "cluster-sum" not in dk
    assert okc and okk
    assert np.array_equal(Cc, Ck), dc
    err, ok = check_against_oracle(Cc, A, B)
    assert ok, f"{dc}: {err}"


def test_cluster_sum_misaligned_fallback_and_padding():
    # A misaligned base pointer sends an in-kernel plan to the pre-pass kernel,
    # which sums its slices in a cluster too; padded C stays untouched.
    M, N, K = 512, 512, 512
    A = inputs.uniform_pm1(1723, M, K)
    B = inputs.uniform_pm1(1724, K, N)
    opts = dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=128, split_k=4, operand_split=2, split_reduce=2)
    C, desc, canaries, _ = run_gemm(A, B, lda=K + 4, ldc=N + 5, a_off=1, c_off=3, **opts)
    assert canaries and "cluster-sum" in desc
    err, ok = check_against_oracle(C, A, B)
    assert ok, f"{desc}: {err}"


def test_cluster_sum_launch_count():
    opts = dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=128, split_k=2, operand_split=2)
    with g.Plan(1024, 1024, 1024, split_reduce=2, **opts) as p:
        assert "cluster-sum" in p.describe()
        assert p.kernel_launches == 1
    with g.Plan(1024, 1024, 1024, split_reduce=1, **opts) as p:
        assert "cluster-sum" not in p.describe()
        assert p.kernel_launches == 2


@pytest.mark.parametrize("shape,opts", [
    ((512, 512, 512), dict(tile_n=128, split_k=3)),           # 3 slices: rows do not split in 3
    ((512, 512, 512), dict(tile_n=128, split_k=8)),           # 8 slices: a quadrant is not a block
    ((512, 512, 512), dict(tile_n=256, split_k=2)),           # 128 x 256 tiles: ring too small
    ((512, 512, 512), dict(tile_n=128, stages=1, split_k=2, operand_split=1)),  # 1-stage ring too small
    ((2048, 1024, 1024), dict(tile_n=128, split_k=0)),        # no split at all
    ((2048, 2048, 1024), dict(tile_n=128, split_k=2)),        # more slices than fit at once
], ids=["three_slices", "eight_slices", "wide_tiles", "one_stage", "no_split", "too_many"])
def test_cluster_sum_refusals(shape, opts):
    with pytest.raises(g.GemmError) as e:
        g.Plan(*shape, variant=g.VARIANT_TCGEN05, tile_m=128, split_reduce=2, **opts)
    assert e.value.status == g.ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# K-slices summed by the last slice to arrive (per 32-row quadrant, an atomic
# count) instead of the reduction kernel: the same slice order, the same bits.
# ---------------------------------------------------------------------------

FIXUP_CASES = [
    # M, N, K, tile_n, split_k, operand_split
    (1024, 1024, 1024, 256, 4, 2),   # the 1024^3 plan
    (1024, 1024, 1024, 128, 2, 2),
    (512, 512, 512, 128, 8, 2),      # 8 slices
    (1000, 520, 264, 128, 2, 1),     # ragged; slices of 5 and 4 k-blocks
    (500, 520, 256, 128, 4, 4),      # raw A
    (600, 700, 1024, 256, 2, 3),     # hybrid, 128x256 tiles
    (384, 300, 640, 64, 4, 1),       # 128x64 tiles
    (200, 61, 160, 128, 2, 1),       # N not a multiple of 4: C by direct stores
    (130, 33, 96, 64, 3, 1),         # quadrants past M, three slices
]


@pytest.mark.parametrize("case", FIXUP_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_bn{c[3]}_s{c[4]}_m{c[5]}"
                                                   for c in FIXUP_CASES])
def test_last_arriver_sum_matches_reduction_kernel(case):
    M, N, K, bn, split, mode = case
    A = inputs.uniform_pm1(1741, M, K)
    B = inputs.uniform_pm1(1742, K, N)
    opts = dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=bn, split_k=split, operand_split=mode)
    Cf, df, okf, runs = run_gemm(A, B, split_reduce=3, repeat=3, **opts)
    Ck, dk, okk, _ = run_gemm(A, B, split_reduce=1, **opts)
    assert "last-arriver-sum" in df and "last-arriver-sum" not in dk
    assert okf and okk
    assert all(np.array_equal(r, Cf) for r in runs), "repeat runs differ (counters not reset?)"
    assert np.array_equal(Cf, Ck), df
    err, ok = check_against_oracle(Cf, A, B)
    assert ok, f"{df}: {err}"


def test_last_arriver_sum_tail_wave():
    # 2560^2 with 128x256 tiles: 200 tiles, the last 48 split in 3 (144 units)
    M = N = 2560
    K = 1024
    A = inputs.uniform_pm1(1743, M, K)
    B = inputs.uniform_pm1(1744, K, N)
    opts = dict(variant=g.VARIANT_TCGEN05, tile_n=256, operand_split=4)
    Cf, df, okf, _ = run_gemm(A, B, split_reduce=3, **opts)
    Ck, dk, okk, _ = run_gemm(A, B, split_reduce=1, **opts)
    assert "last-arriver-sum" in df and "whole=152" in df, df
    assert okf and okk and np.array_equal(Cf, Ck)
    rows = np.repeat(np.array([0, 1, 1279, 2047, 2431, 2559]), N)
    cols = np.tile(np.arange(N), 6)
    Cref, S = oracle.gemm_f64_entries(A, B, rows, cols)
    assert oracle.within_bound(Cf[rows, cols], Cref, S, K)


@pytest.mark.parametrize("shape,opts", [
    ((512, 512, 2048), dict(tile_n=128, split_k=16)),                            # 16 slices
    ((512, 512, 512), dict(tile_n=128, stages=1, split_k=2, operand_split=1)),   # ring too small
    ((2048, 2048, 1024), dict(tile_n=128, split_k=2)),                           # two waves of split units
    ((2048, 1024, 1024), dict(tile_n=128, split_k=1)),                           # nothing split
], ids=["sixteen_slices", "one_stage", "two_waves", "no_split"])
def test_last_arriver_sum_refusals(shape, opts):
    with pytest.raises(g.GemmError) as e:
        g.Plan(*shape, variant=g.VARIANT_TCGEN05, split_reduce=3, **opts)
    assert e.value.status == g.ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# The pipelined host-buffer run: row panels of whole 128-row tiles, B copied
# and split once, each panel's A copy / GEMM / C copy overlapped on three
# streams.  Every operand mode, ragged panels, padded leading dimensions,
# pinned host memory, repeated runs (the panel states are kept).
# ---------------------------------------------------------------------------

def _pinned(host, ld):
    import torch
    rows, cols = host.shape
    t = torch.full((rows, ld), 321.0, dtype=torch.float32).pin_memory()
    t[:, :cols] = torch.from_numpy(host)
    return t


@pytest.mark.parametrize("panels,cols", [(2, 1), (3, 1), (7, 1), (3, 3), (2, 2)])
@pytest.mark.parametrize("mode", [1, 2, 3, 4], ids=["pre_pass", "in_kernel", "hybrid", "raw_a"])
def test_run_host_panels(mode, panels, cols):
    # cols > 1: the first panel in column blocks (in-kernel and hybrid splits;
    # the pre-pass forms ignore it); N = 520 leaves a ragged last block, and
    # ldc = N + 3 keeps C from the TMA-store epilogue
    M, N, K = 1000, 520, 264
    lda, ldb, ldc = K + 4, N + 8, N + 3
    A = inputs.uniform_pm1(1711, M, K)
    B = inputs.uniform_pm1(1712, K, N)
    hA, hB = _pinned(A, lda), _pinned(B, ldb)
    hC = _pinned(np.full((M, N), np.nan, dtype=np.float32), ldc)
    with g.Plan(M, N, K, lda, ldb, ldc, variant=g.VARIANT_TCGEN05, operand_split=mode,
                host_panels=panels, host_col_blocks=cols) as p:
        for _ in range(2):
            hC[:, :N] = float("nan")
            s = p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0)
            assert s == g.OK, g.gemm_f32_status_string(s)
            C = hC.numpy()
            Cref, S = oracle.gemm_f64(A, B)
            assert oracle.within_bound(C[:, :N], Cref, S, K), p.describe()
            assert (C[:, N:] == 321.0).all()


@pytest.mark.parametrize("mode,cols", [(1, 0), (4, 0), (2, 3), (3, 2)],
                         ids=["pre_pass", "raw_a", "in_kernel_blocks", "hybrid_blocks"])
def test_run_host_panels_bit_identical_to_device_run(mode, cols):
    # With no K-split every output tile is summed in the same order whichever
    # panel (or column block of the first panel) it falls in, so the panel
    # pipeline must reproduce the one-launch device run bit for bit (a wrong
    # panel or block offset cannot hide in the bound).
    import torch
    M, N, K = 1536, 640, 192
    A = inputs.normal(1713, M, K)
    B = inputs.normal(1714, K, N)
    hA, hB = _pinned(A, K), _pinned(B, N)
    hC = _pinned(np.zeros((M, N), dtype=np.float32), N)
    opts = dict(variant=g.VARIANT_TCGEN05, operand_split=mode, split_k=1, tile_m=128)
    with g.Plan(M, N, K, host_panels=4, host_col_blocks=cols, **opts) as p:
        assert p.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 0) == g.OK
    C, desc, canaries, _ = run_gemm(A, B, host_panels=1, **opts)
    assert canaries
    assert np.array_equal(hC.numpy().astype(np.float64), C), desc


def test_run_host_panel_option_validation():
    for bad in (-1, 65):
        with pytest.raises(g.GemmError):
            g.Plan(256, 256, 256, variant=g.VARIANT_TCGEN05, host_panels=bad)
    # more panels than tile-rows: clamped to one panel per tile-row
    M, N, K = 200, 64, 64
    A = inputs.uniform_pm1(1715, M, K)
    B = inputs.uniform_pm1(1716, K, N)
    C = np.full((M, N), np.nan, dtype=np.float32)
    with g.Plan(M, N, K, variant=g.VARIANT_TCGEN05, host_panels=64) as p:
        assert p.run_host(A.ctypes.data, B.ctypes.data, C.ctypes.data, 0) == g.OK
    Cref, S = oracle.gemm_f64(A, B)
    assert oracle.within_bound(C, Cref, S, K)


# ---------------------------------------------------------------------------
# Non-finite inputs: an Inf in A makes its row of C non-finite, a NaN in B its
# column (the 3xTF32 split turns Inf into NaN, so only non-finiteness is
# asserted); every other element stays finite and within the bound - nothing
# leaks across tiles, K-slices or the operand split.
# ---------------------------------------------------------------------------

NONFINITE_VARIANTS = [SIMT, TC, {"variant": g.VARIANT_TCGEN05, "operand_split": 2},
                      {"variant": g.VARIANT_TCGEN05, "operand_split": 2, "tile_k": 16},
                      {"variant": g.VARIANT_TCGEN05, "operand_split": 3},
                      {"variant": g.VARIANT_TCGEN05, "operand_split": 4},
                      {"variant": g.VARIANT_TCGEN05, "split_k": 4},
                      {"variant": g.VARIANT_TCGEN05, "tile_m": 256, "operand_split": 3},
                      {"variant": g.VARIANT_TCGEN05, "tile_m": 256, "operand_split": 4},
                      {"variant": g.VARIANT_TCGEN05, "tile_m": 256, "tile_n": 256, "operand_split": 5}]


@pytest.mark.parametrize("variant", NONFINITE_VARIANTS,
                         ids=["simt", "tcgen05", "in_kernel", "in_kernel_k16", "hybrid", "raw_a", "split4",
                              "pair_hybrid", "pair_raw_a", "pair_tmem_a"])
def test_non_finite_inputs(variant):
    M, N, K = 300, 260, 100
    A = inputs.uniform_pm1(1751, M, K)
    B = inputs.uniform_pm1(1752, K, N)
    A[5, 17] = np.inf
    B[33, 200] = np.nan
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    assert canaries, desc
    assert not np.isfinite(C[5, :]).any(), desc
    assert not np.isfinite(C[:, 200]).any(), desc
    rest = np.ones((M, N), dtype=bool)
    rest[5, :] = False
    rest[:, 200] = False
    assert np.isfinite(C[rest]).all(), desc
    A0, B0 = A.copy(), B.copy()
    A0[5, 17] = 0.0
    B0[33, 200] = 0.0
    Cref, S = oracle.gemm_f64(A0, B0)
    assert oracle.within_bound(C[rest], Cref[rest], S[rest], K), desc


# ---------------------------------------------------------------------------
# Extreme aspect ratios: a very long K (many k-blocks per tile, long
# accumulation) and a very tall, thin product.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [AUTO, SIMT, TC, FUSED], ids=["auto", "simt", "tcgen05", "in_kernel"])
def test_long_k(variant):
    M, N, K = 128, 96, 262144
    A = inputs.uniform_pm1(1801, M, K)
    B = inputs.uniform_pm1(1802, K, N)
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


@pytest.mark.parametrize("variant", [AUTO, SIMT, TC], ids=["auto", "simt", "tcgen05"])
def test_very_tall(variant):
    M, N, K = 1 << 18, 24, 40
    A = inputs.normal(1803, M, K)
    B = inputs.normal(1804, K, N)
    C, desc, canaries, _ = run_gemm(A, B, **variant)
    err, ok = check_against_oracle(C, A, B)
    assert canaries and ok, f"{desc}: {err}"


def test_plans_on_several_streams_at_once():
    # Different plans on different streams share nothing: two CTA-pair plans
    # (one split in K, one of whole tiles) and a SIMT plan, queued back to back
    # on three streams ten times, give the same bits as each run alone.
    import torch
    shapes = [(1024, 1024, 1024), (2048, 2048, 512), (513, 257, 129)]
    runs = []
    for i, (M, N, K) in enumerate(shapes):
        A = inputs.uniform_pm1(2301 + 2 * i, M, K)
        B = inputs.normal(2302 + 2 * i, K, N)
        ref, desc, ok, _ = run_gemm(A, B)
        assert ok, desc
        runs.append((g.Plan(M, N, K), torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                     torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda"), ref, torch.cuda.Stream()))
    try:
        torch.cuda.synchronize()
        for _ in range(10):
            for p, dA, dB, dC, _, st in runs:
                assert p.run_ptr(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), st.cuda_stream) == g.OK
        for p, _, _, dC, ref, st in runs:
            st.synchronize()
            assert p.check() == g.OK
            assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref), p.describe()
    finally:
        for r in runs:
            r[0].close()


@pytest.mark.parametrize("shape,opts", [
    ((1024, 1024, 1024), {}),                                                   # CTA pairs, 4 K-slices
    ((4096, 4096, 256), {}),                                                    # raw-A pairs: pre-pass, split last wave
    ((768, 768, 768), dict(variant=g.VARIANT_TCGEN05, tile_m=128, split_k=4)),  # one CTA per tile
    ((513, 257, 129), dict(variant=g.VARIANT_SIMT, split_k=2)),                 # SIMT with its reduction
], ids=["pairs", "raw_a_pairs", "one_cta", "simt_split"])
def test_runs_captured_in_a_cuda_graph(shape, opts):
    # Every launch of a run is stream-ordered and allocation-free, so runs can
    # be captured in a CUDA graph: replays give the bits of a plain run.
    import torch
    M, N, K = shape
    A = inputs.uniform_pm1(2311, M, K)
    B = inputs.normal(2312, K, N)
    ref, desc, ok, _ = run_gemm(A, B, **opts)
    assert ok, desc
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with g.Plan(M, N, K, **opts) as p:
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            p.run_ptr(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), st.cuda_stream)  # warm (attributes, maps)
        st.synchronize()
        dC.fill_(float("nan"))
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for _ in range(2):
                p.run_ptr(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), st.cuda_stream)
        with torch.cuda.stream(st):
            for _ in range(3):
                graph.replay()
        st.synchronize()
        assert p.check() == g.OK
        assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref), p.describe()


@pytest.mark.parametrize("shape", [(1024, 1024, 16), (2048, 2048, 8), (700, 900, 5), (640, 640, 24),
                                   (1500, 1500, 31), (2048, 4096, 1)])
def test_short_k_over_many_tiles(shape):
    # Many output tiles over a short K take big SIMT tiles without K-slices
    # (the dispatcher's rule); checked element by element against the oracle.
    M, N, K = shape
    A = inputs.uniform_pm1(2321, M, K)
    B = inputs.normal(2322, K, N)
    C, desc, ok, _ = run_gemm(A, B)
    assert ok, desc
    assert desc.startswith("simt") and (("tile=128x64x16" in desc) or ("tile=64x64x16" in desc)), desc
    err, okb = check_against_oracle(C, A, B)
    assert okb, f"{desc}: {err}"


SHORT_M = [
    # (M, N, K, lda, ldb, ldc): a short A against B, the short-M kernel forced
    (1, 8192, 8192, None, None, None),       # the dispatcher's choice too
    (16, 4096, 4096, None, None, None),
    (5, 1000, 3000, None, None, None),       # N past the last whole block
    (13, 777, 1500, 1503, 781, 790),         # B rows not 16-byte aligned: scalar loads
    (3, 2049, 513, None, None, None),        # K past the last whole piece, N past a quad
    (16, 256, 65536, None, None, None),      # several pieces per block's K-range
    (1, 300, 4096, 4100, None, None),
    (7, 33, 40, None, None, None),           # one block, one piece, one range: C written directly
]


@pytest.mark.parametrize("case", SHORT_M, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in SHORT_M])
def test_short_m_against_the_oracle(case):
    M, N, K, lda, ldb, ldc = case
    A = inputs.uniform_pm1(2331, M, K)
    B = inputs.normal(2332, K, N)
    C, desc, ok, outs = run_gemm(A, B, lda=lda, ldb=ldb, ldc=ldc, repeat=2, variant=g.VARIANT_SHORT_M)
    assert desc.startswith("simt short-m"), desc
    assert ok, desc
    assert np.array_equal(outs[0], outs[1]), desc
    err, okb = check_against_oracle(C, A, B)
    assert okb, f"{desc}: {err}"
    with g.Plan(M, N, K, variant=g.VARIANT_SHORT_M) as p:
        splits = int(p.describe().split("split_k=")[1].split()[0])
        assert p.kernel_launches == (2 if splits > 1 else 1)
    # the dispatcher takes it for up to 8 rows against 2^24 elements of B or more
    chosen = M <= 8 and N * K >= 2 ** 24
    with g.Plan(M, N, K) as p:
        assert p.describe().startswith("simt short-m") == chosen, p.describe()
    # there, options of the SIMT kernel's shape give an ordinary SIMT plan;
    # forced together with the short-M variant, or past 16 rows, it is refused
    if chosen:
        with g.Plan(M, N, K, tile_m=32, tile_n=32) as p:
            assert p.describe().startswith("simt tile=32x32"), p.describe()
    with pytest.raises(g.GemmError):
        g.Plan(M, N, K, variant=g.VARIANT_SHORT_M, tile_m=32, tile_n=32)
    with pytest.raises(g.GemmError):
        g.Plan(17, N, K, variant=g.VARIANT_SHORT_M)


SHORT_N = [
    # (M, N, K, lda, ldb, ldc): a short B against A, the short-N kernel forced
    (8192, 1, 8192, None, None, None),       # the dispatcher's choice too
    (4096, 4, 4100, None, None, None),        # K past a 512-element step
    (300, 16, 4096, None, None, None),
    (5000, 3, 1001, 1003, 5, 7),            # A rows not 16-byte aligned: scalar loads
    (33, 7, 40, None, None, None),
]


@pytest.mark.parametrize("case", SHORT_N, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in SHORT_N])
def test_short_n_against_the_oracle(case):
    M, N, K, lda, ldb, ldc = case
    A = inputs.uniform_pm1(2341, M, K)
    B = inputs.normal(2342, K, N)
    C, desc, ok, outs = run_gemm(A, B, lda=lda, ldb=ldb, ldc=ldc, repeat=2, variant=g.VARIANT_SHORT_N)
    assert desc.startswith("simt short-n"), desc
    assert ok, desc
    assert np.array_equal(outs[0], outs[1]), desc
    err, okb = check_against_oracle(C, A, B)
    assert okb, f"{desc}: {err}"
    with g.Plan(M, N, K) as p:
        assert p.describe().startswith("simt short-n") == (N == 1 and M >= 4096 and M * K >= 2 ** 24), p.describe()
    with pytest.raises(g.GemmError):
        g.Plan(M, 17, K, variant=g.VARIANT_SHORT_N)
