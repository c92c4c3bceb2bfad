"""GPU parity on edge magnitudes, through every form of the operand split.

The tensor-core plans split each FP32 operand into two TF32 pieces.  These
tests hold them to the accuracy the interface states ("Dependence-aware group
synchronization on M1 Max", section "Controlled implementation comparison":
the complete output against an FP64 oracle), on inputs where a split could go
wrong:

  * finite values from the top of FP32's range (rounding them to TF32 would
    carry into the Inf exponent), paired with small values so every product
    and sum stays finite: every output must be finite and within the plain
    bound |C - C_exact| <= 2 K 2^-24 S;
  * magnitudes spread over 2^-100 .. 2^100: the plain bound;
  * subnormal operands and results below FP32's normal range: the bound with
    its underflow terms (``oracle.bound_ratio``): K 2^-149 for gradual
    underflow and, for the tensor-core plans, 2^-136 T for elements below
    2^-113, which TF32 pieces carry only to within 2^-137.
"""
import numpy as np
import pytest

import oracle
import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

TC = g.VARIANT_TCGEN05
FORMS = {
    "simt": dict(variant=g.VARIANT_SIMT),
    "pre_pass": dict(variant=TC, operand_split=1),
    "raw_a": dict(variant=TC, operand_split=4),
    "in_kernel": dict(variant=TC, operand_split=2),
    "in_kernel_k16": dict(variant=TC, operand_split=2, tile_k=16),
    "hybrid": dict(variant=TC, operand_split=3),
    "pair_in_kernel": dict(variant=TC, tile_m=256, operand_split=2),
    "pair_hybrid": dict(variant=TC, tile_m=256, operand_split=3),
    "pair_raw_a": dict(variant=TC, tile_m=256, operand_split=4),
    "pair_raw_a_k16": dict(variant=TC, tile_m=256, tile_n=256, operand_split=4, tile_k=16),
    "pair_tmem_a": dict(variant=TC, tile_m=256, tile_n=256, operand_split=5),
    "split_k4": dict(variant=TC, split_k=4),
}
M, N, K = 300, 520, 264


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_gb300 import build
    build.build()
    g.load()


def _near_max_rows_of_a():
    A = inputs.uniform_pm1(2101, M, K)
    B = inputs.uniform_pm1(2102, K, N) * np.float32(2.0 ** -40)
    cols = np.arange(0, K, 7)
    A[np.ix_([5, 77, 255], cols)] = inputs.top_of_range(2103, 3, len(cols))
    A[9, :] = inputs.top_of_range(2104, 1, K)
    return A, B


def _near_max_columns_of_b():
    A = inputs.uniform_pm1(2111, M, K) * np.float32(2.0 ** -40)
    B = inputs.uniform_pm1(2112, K, N)
    rows = np.arange(0, K, 5)
    B[np.ix_(rows, [3, 130, 511])] = inputs.top_of_range(2113, len(rows), 3)
    B[:, 200] = inputs.top_of_range(2114, K, 1)[:, 0]
    return A, B


def _all_top_a():
    return inputs.top_of_range(2121, M, K), inputs.uniform_pm1(2122, K, N) * np.float32(2.0 ** -22)


def _mixed_magnitudes():
    return inputs.scaled_exponents(2131, M, K, -100, 100), inputs.scaled_exponents(2132, K, N, -20, 20)


def _subnormal_rows_of_a():
    A = inputs.uniform_pm1(2141, M, K)
    A[[3, 100, 299], :] = inputs.subnormal(2142, 3, K)
    return A, inputs.uniform_pm1(2143, K, N)


def _subnormal_a_times_large_b():
    A = inputs.uniform_pm1(2151, M, K)
    A[[0, 131, 298], :] = inputs.subnormal(2152, 3, K)
    return A, inputs.uniform_pm1(2153, K, N) * np.float32(2.0 ** 100)


def _large_a_times_subnormal_b():
    B = inputs.uniform_pm1(2161, K, N)
    B[:, [0, 257, 519]] = inputs.subnormal(2162, K, 3)
    return inputs.uniform_pm1(2163, M, K) * np.float32(2.0 ** 100), B


def _subnormal_results():
    return (inputs.uniform_pm1(2171, M, K) * np.float32(2.0 ** -70),
            inputs.uniform_pm1(2172, K, N) * np.float32(2.0 ** -70))


PLAIN = {"near_max_rows_of_a": _near_max_rows_of_a, "near_max_columns_of_b": _near_max_columns_of_b,
         "all_top_of_range_a": _all_top_a, "magnitudes_2^-100_to_2^100": _mixed_magnitudes}
UNDERFLOW = {"subnormal_rows_of_a": _subnormal_rows_of_a, "subnormal_a_times_2^100_b": _subnormal_a_times_large_b,
             "2^100_a_times_subnormal_b": _large_a_times_subnormal_b, "subnormal_results": _subnormal_results}


@pytest.mark.parametrize("form", list(FORMS), ids=list(FORMS))
@pytest.mark.parametrize("case", list(PLAIN), ids=list(PLAIN))
def test_finite_extremes_within_the_plain_bound(case, form):
    A, B = PLAIN[case]()
    assert np.isfinite(A).all() and np.isfinite(B).all()
    C, desc, canaries, _ = run_gemm(A, B, **FORMS[form])
    Cref, S = oracle.gemm_f64(A, B)
    assert np.isfinite(S).all() and S.max() < 2.0 ** 127
    assert canaries, desc
    assert np.isfinite(C).all(), f"{desc}: {int((~np.isfinite(C)).sum())} non-finite outputs"
    err = oracle.normalised_error(C, Cref, S, K)
    assert err <= 2.0, f"{case} {desc}: max normalised error {err}"


@pytest.mark.parametrize("form", list(FORMS), ids=list(FORMS))
@pytest.mark.parametrize("case", list(UNDERFLOW), ids=list(UNDERFLOW))
def test_underflow_within_the_stated_bound(case, form):
    A, B = UNDERFLOW[case]()
    C, desc, canaries, _ = run_gemm(A, B, **FORMS[form])
    Cref, S = oracle.gemm_f64(A, B)
    T = None if form == "simt" else oracle.tf32_grid_term(A, B)
    assert canaries, desc
    r = oracle.bound_ratio(C, Cref, S, K, T)
    assert r <= 1.0, f"{case} {desc}: error / stated bound = {r}"


def test_subnormal_operands_are_not_flushed():
    # A TF32-exact subnormal (2^-130) times small integers: every tensor-core
    # form must return the exact product (a flushed operand would give 0).
    rng_rows = np.arange(M)
    ks = (rng_rows * 37) % K
    A = np.zeros((M, K), np.float32)
    A[rng_rows, ks] = np.float32(2.0 ** -130)
    B = inputs.small_int(2181, K, N)
    exact = np.float64(2.0 ** -130) * B[ks, :].astype(np.float64)
    for form, opts in FORMS.items():
        C, desc, canaries, _ = run_gemm(A, B, **opts)
        assert canaries and np.array_equal(C, exact), f"{form} {desc}"
