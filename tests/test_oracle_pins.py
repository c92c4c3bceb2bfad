"""Pins for the CPU oracle: each checks it against something other than itself.

The oracle computes C = A*B with FP64 accumulation in ascending k and the scale
S = |A|*|B| (the definition written out; "Dependence-aware group
synchronization on M1 Max", section "Controlled implementation comparison":
complete output checked against an FP64 oracle).  The pins below fix it by
closed forms, exact integer arithmetic, exact rational brute force, a
hand-worked example, an independent library routine and invariants.  Each pin
is also run against deliberately broken variants of the oracle (a transposed
operand, a dropped term, a wrong sign, a shifted index) and must reject every
one of them: the pins have teeth.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from software_pipelined_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_blocks(path):
    blocks, cur, name = {}, None, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0].isalpha():
                name, r, c = parts[0], int(parts[1]), int(parts[2])
                cur = []
                blocks[name] = (r, c, cur)
            else:
                cur.append([float(v) for v in parts])
    return {k: np.array(v, dtype=np.float64).reshape(r, c) for k, (r, c, v) in blocks.items()}


# ---------------------------------------------------------------------------
# Pin checks, written against a callable gemm(A, B) -> (C, S) so that the same
# checks can be run on the oracle and on planted mistakes.
# ---------------------------------------------------------------------------

def pin_hand_example(gemm):
    g = _read_blocks(os.path.join(GOLDEN, "hand_product_2x3x2.txt"))
    C, S = gemm(g["A"].astype(np.float32), g["B"].astype(np.float32))
    return np.array_equal(C, g["C"]) and np.array_equal(S, g["C"])  # all entries positive


def pin_identity(gemm):
    B = inputs.uniform_pm1(11, 24, 17)
    C, _ = gemm(np.eye(24, dtype=np.float32), B)
    A = inputs.uniform_pm1(12, 19, 24)
    C2, _ = gemm(A, np.eye(24, dtype=np.float32))
    return np.array_equal(C, B.astype(np.float64)) and np.array_equal(C2, A.astype(np.float64))


def pin_permutation(gemm):
    rng = np.random.default_rng(5)
    K = 23
    p = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), p] = 1.0  # (P B)[i] = B[p[i]]
    B = inputs.uniform_pm1(13, K, 29)
    C, _ = gemm(P, B)
    A = inputs.uniform_pm1(14, 31, K)
    C2, _ = gemm(A, P)  # (A P)[:, j] = A[:, i] where p[i] == j
    inv = np.argsort(p)
    return (np.array_equal(C, B[p].astype(np.float64))
            and np.array_equal(C2, A[:, inv].astype(np.float64)))


def pin_rank1_weighted(gemm):
    # A_ik = u_i (k+1), B_kj = v_j (k+1)  =>  C_ij = u_i v_j K(K+1)(2K+1)/6, exact.
    M, N, K = 13, 11, 97
    u = np.arange(-6, 7, dtype=np.float64)
    v = np.arange(-5, 6, dtype=np.float64)[::-1].copy()
    kk = np.arange(1, K + 1, dtype=np.float64)
    A = (u[:, None] * kk[None, :]).astype(np.float32)
    B = (kk[:, None] * v[None, :]).astype(np.float32)
    C, S = gemm(A, B)
    s2 = K * (K + 1) * (2 * K + 1) // 6
    return (np.array_equal(C, np.outer(u, v) * s2)
            and np.array_equal(S, np.outer(np.abs(u), np.abs(v)) * s2))


def pin_rank1_ones(gemm):
    # A = u 1^T, B = 1 v^T  =>  C = K u v^T.
    M, N, K = 7, 9, 61
    u = np.linspace(-3, 3, M).astype(np.float32)
    v = np.linspace(-2, 2, N).astype(np.float32)
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    C, _ = gemm(A, B)
    want = K * np.outer(u.astype(np.float64), v.astype(np.float64))
    return np.allclose(C, want, rtol=0, atol=1e-12)


def pin_small_int_exact(gemm):
    # Integers in [-8, 8]: every partial sum is an integer well below 2^53, so the
    # FP64 result is exact and must equal the exact int64 product.
    A = inputs.small_int(21, 37, 53)
    B = inputs.small_int(22, 53, 41)
    C, S = gemm(A, B)
    Ai, Bi = A.astype(np.int64), B.astype(np.int64)
    return (np.array_equal(C, (Ai @ Bi).astype(np.float64))
            and np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64)))


def pin_fraction_bruteforce(gemm):
    # Exact rational sums on tiny shapes; the FP64 sum in ascending k is within
    # (K-1) * 2^-53 * S of it (first-order bound of recursive summation).
    ok = True
    for (M, N, K, sa, sb) in [(1, 1, 1, 31, 32), (3, 5, 7, 33, 34), (4, 4, 9, 35, 36)]:
        A = inputs.uniform_pm1(sa, M, K)
        B = inputs.normal(sb, K, N)
        C, S = gemm(A, B)
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
                mag = sum(abs(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))) for k in range(K))
                err = abs(Fraction(C[i, j]) - exact)
                if err > Fraction(max(K - 1, 0)) * Fraction(1, 2 ** 53) * mag * Fraction(101, 100):
                    ok = False
                if Fraction(S[i, j]) != mag and abs(Fraction(S[i, j]) - mag) > Fraction(K, 2 ** 53) * mag:
                    ok = False
    return ok


def pin_numpy_crosscheck(gemm):
    # An independent FP64 product (numpy's BLAS) agrees within 2*K*2^-53*S at the
    # ragged 127x193x61 shape.
    A = inputs.uniform_pm1(2005, 127, 61)
    B = inputs.uniform_pm1(2006, 61, 193)
    C, S = gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    refS = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    K = 61
    return (bool(np.all(np.abs(C - ref) <= 2 * K * 2.0 ** -53 * refS))
            and bool(np.all(np.abs(S - refS) <= 2 * K * 2.0 ** -53 * refS)))


PINS = [pin_hand_example, pin_identity, pin_permutation, pin_rank1_weighted,
        pin_rank1_ones, pin_small_int_exact, pin_fraction_bruteforce, pin_numpy_crosscheck]


# ---------------------------------------------------------------------------
# The oracle passes every pin.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.gemm_f64)


# ---------------------------------------------------------------------------
# Planted mistakes (on the CPU, in wrappers around the oracle) must each be
# caught by at least one pin.
# ---------------------------------------------------------------------------

def _mut_transposed_b(A, B):  # uses B^T where B is square, else falls back to a wrong shape
    if B.shape[0] == B.shape[1]:
        return oracle.gemm_f64(A, np.ascontiguousarray(B.T))
    C, S = oracle.gemm_f64(A, B)
    return C.T.reshape(C.shape) if C.shape[0] == C.shape[1] else C * 1.0000001, S


def _mut_dropped_last_term(A, B):
    K = A.shape[1]
    if K <= 1:
        C, S = oracle.gemm_f64(A, B)
        return C * 0.5, S
    return oracle.gemm_f64(np.ascontiguousarray(A[:, :K - 1]), np.ascontiguousarray(B[:K - 1]))


def _mut_wrong_sign(A, B):
    A2 = A.copy()
    A2[:, -1] = -A2[:, -1]
    C, _ = oracle.gemm_f64(A2, B)
    _, S = oracle.gemm_f64(A, B)
    return C, S


def _mut_shifted_row(A, B):
    C, S = oracle.gemm_f64(A, B)
    return np.roll(C, 1, axis=0), S


def _mut_scale_without_abs(A, B):
    C, _ = oracle.gemm_f64(A, B)
    return C, C.copy()


def _mut_float32_accumulation(A, B):
    C, S = oracle.gemm_f64(A, B)
    C32 = np.zeros(C.shape, dtype=np.float32)
    for k in range(A.shape[1]):
        C32 += np.outer(A[:, k], B[k]).astype(np.float32)
    return C32.astype(np.float64), S


MUTANTS = [_mut_transposed_b, _mut_dropped_last_term, _mut_wrong_sign, _mut_shifted_row,
           _mut_scale_without_abs, _mut_float32_accumulation]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_reject_planted_mistake(mutant):
    caught = [p.__name__ for p in PINS if not p(mutant)]
    assert caught, f"no pin rejects {mutant.__name__}"


# ---------------------------------------------------------------------------
# Further oracle behaviour: padded leading dimensions, K = 0, sampled entries,
# and the accuracy criterion itself.
# ---------------------------------------------------------------------------

def test_padded_leading_dimensions_ignore_padding():
    # Padding columns hold NaN; a reader that touched them would propagate NaN.
    A = inputs.uniform_pm1(41, 33, 45, ld=52)
    B = inputs.uniform_pm1(42, 45, 27, ld=31)
    C, S = oracle.gemm_f64(A, B)
    C2, S2 = oracle.gemm_f64(np.ascontiguousarray(A), np.ascontiguousarray(B))
    assert np.isfinite(C).all()
    assert np.array_equal(C, C2) and np.array_equal(S, S2)


def test_k_zero_is_empty_sum():
    A = np.zeros((5, 0), dtype=np.float32)
    B = np.zeros((0, 7), dtype=np.float32)
    C, S = oracle.gemm_f64(A, B)
    assert C.shape == (5, 7) and not C.any() and not S.any()


def test_entries_equal_full_product():
    A = inputs.uniform_pm1(51, 40, 70)
    B = inputs.normal(52, 70, 30)
    C, S = oracle.gemm_f64(A, B)
    rows = np.array([0, 39, 17, 5, 39])
    cols = np.array([0, 29, 3, 28, 0])
    c, s = oracle.gemm_f64_entries(A, B, rows, cols)
    assert np.array_equal(c, C[rows, cols]) and np.array_equal(s, S[rows, cols])


def test_normalised_error_detects_planted_error():
    A = inputs.uniform_pm1(61, 20, 64)
    B = inputs.uniform_pm1(62, 64, 20)
    C, S = oracle.gemm_f64(A, B)
    K = 64
    assert oracle.normalised_error(C, C, S, K) == 0.0
    Cbad = C.copy()
    Cbad[3, 4] += 3 * K * 2.0 ** -24 * S[3, 4]
    assert 2.9 < oracle.normalised_error(Cbad, C, S, K) < 3.1
    assert not oracle.within_bound(Cbad, C, S, K)
    Cnan = C.copy()
    Cnan[0, 0] = np.nan
    assert oracle.normalised_error(Cnan, C, S, K) == np.inf
    Z = np.zeros((2, 2))
    assert oracle.normalised_error(np.array([[0.0, 1e-30], [0, 0]]), Z, Z, K) == np.inf


def test_fp32_rounding_of_oracle_meets_bound():
    # Rounding the FP64 result to FP32 costs at most 2^-24 relative, well inside
    # the bound: the criterion is satisfiable.
    A = inputs.uniform_pm1(71, 64, 300)
    B = inputs.uniform_pm1(72, 300, 64)
    C, S = oracle.gemm_f64(A, B)
    assert oracle.normalised_error(C.astype(np.float32), C, S, 300) <= 1.0 / 300 + 1e-12


def test_threads_setting_does_not_change_result():
    A = inputs.uniform_pm1(81, 64, 128)
    B = inputs.uniform_pm1(82, 128, 48)
    n0 = oracle.get_threads()
    oracle.set_threads(1)
    C1, S1 = oracle.gemm_f64(A, B)
    oracle.set_threads(max(n0, 2))
    C2, S2 = oracle.gemm_f64(A, B)
    oracle.set_threads(n0)
    assert np.array_equal(C1, C2) and np.array_equal(S1, S2)


# ---------------------------------------------------------------------------
# The underflow terms of the bound (tensor-core plans on tiny inputs; results
# below FP32's normal range).  Pinned by closed forms, the threshold's two
# sides, a symmetry, and planted mistakes.
# ---------------------------------------------------------------------------

def _grid_term_closed_forms(term):
    K = 37
    ok = True
    # normal-range data has no TF32 term at all
    A = inputs.uniform_pm1(61, 9, K)
    B = inputs.uniform_pm1(62, K, 11)
    ok &= bool(np.array_equal(term(A, B), np.zeros((9, 11))))
    # A all tiny (c < 2^-113), B = 1 * v^T (normal): T_ij = K |v_j|
    c = np.float32(2.0 ** -120)
    v = inputs.uniform_pm1(63, 1, 11)[0] + np.float32(2.0)
    T = term(np.full((9, K), c, np.float32), np.tile(v, (K, 1)))
    ok &= bool(np.array_equal(T, np.tile(K * np.abs(v.astype(np.float64)), (9, 1))))
    # B all tiny, A = u * 1^T (normal): T_ij = K |u_i|
    u = inputs.uniform_pm1(64, 9, 1)[:, 0] - np.float32(2.0)
    T = term(np.tile(u[:, None], (1, K)), np.full((K, 11), -c, np.float32))
    ok &= bool(np.array_equal(T, np.tile(K * np.abs(u.astype(np.float64))[:, None], (1, 11))))
    # both tiny: each k counts both ways, |b| + |a| = 2c per k
    T = term(np.full((2, K), c, np.float32), np.full((K, 3), c, np.float32))
    ok &= bool(np.array_equal(T, np.full((2, 3), 2.0 * K * float(c))))
    return ok


def _grid_term_threshold(term):
    # exactly 2^-113 is carried in full; the next float below is not; zero never counts;
    # a value between 2^-126 and 2^-113 (normal FP32, but below full resolution) does
    vals = np.array([2.0 ** -113, np.nextafter(np.float32(2.0 ** -113), np.float32(0)), 0.0, 2.0 ** -120],
                    dtype=np.float32)
    A = vals[:, None]                      # 4 x 1
    B = np.array([[3.0]], dtype=np.float32)
    T = term(A, B)[:, 0]
    return bool(np.array_equal(T, np.array([0.0, 3.0, 0.0, 3.0])))


def _grid_term_symmetry(term):
    A = inputs.scaled_exponents(65, 7, 13, -130, -100)
    B = inputs.scaled_exponents(66, 13, 5, -130, -100)
    return bool(np.allclose(term(A, B), term(B.T, A.T).T, rtol=1e-15, atol=0))


GRID_PINS = [_grid_term_closed_forms, _grid_term_threshold, _grid_term_symmetry]


@pytest.mark.parametrize("pin", GRID_PINS, ids=lambda p: p.__name__)
def test_tf32_grid_term_pin(pin):
    assert pin(oracle.tf32_grid_term)


def _grid_mutants():
    def only_a(A, B):  # dropped second term
        a, b = np.abs(A.astype(np.float64)), np.abs(B.astype(np.float64))
        return ((a > 0) & (a < 2.0 ** -113)).astype(np.float64) @ b

    def low_threshold(A, B):  # FP32's normal boundary instead of TF32's full-resolution one
        a, b = np.abs(A.astype(np.float64)), np.abs(B.astype(np.float64))
        ma = ((a > 0) & (a < 2.0 ** -126)).astype(np.float64)
        mb = ((b > 0) & (b < 2.0 ** -126)).astype(np.float64)
        return ma @ b + a @ mb

    def counts_zero(A, B):  # zero entries counted as tiny
        a, b = np.abs(A.astype(np.float64)), np.abs(B.astype(np.float64))
        return (a < 2.0 ** -113).astype(np.float64) @ b + a @ (b < 2.0 ** -113).astype(np.float64)

    def transposed_mask(A, B):  # mask of B applied on the A side
        a, b = np.abs(A.astype(np.float64)), np.abs(B.astype(np.float64))
        ma = ((a > 0) & (a < 2.0 ** -113)).astype(np.float64)
        return ma @ b + ma @ b
    return [only_a, low_threshold, counts_zero, transposed_mask]


@pytest.mark.parametrize("mutant", _grid_mutants(), ids=lambda m: m.__name__)
def test_grid_pins_reject_planted_mistake(mutant):
    assert not all(p(mutant) for p in GRID_PINS)


def test_bound_ratio_terms():
    K = 64
    C = inputs.uniform_pm1(67, 5, 6).astype(np.float64)
    S = np.abs(C) + 1.0
    T = np.full((5, 6), 2.0 ** 118)  # a TF32 term as large as the relative one
    tol = 2 * K * 2.0 ** -24 * S + K * 2.0 ** -149 + 2.0 ** -136 * T
    assert oracle.bound_ratio(C + tol, C, S, K, T) == pytest.approx(1.0, rel=1e-12)
    assert oracle.bound_ratio(C + 0.5 * tol, C, S, K, T) == pytest.approx(0.5, rel=1e-12)
    # without T the same error exceeds the bound
    assert oracle.bound_ratio(C + tol, C, S, K) > 1.0
    # the underflow term alone: S = 0, an error of K 2^-149 passes, twice that fails
    Z = np.zeros((5, 6))
    assert oracle.bound_ratio(Z + K * 2.0 ** -149, Z, Z, K) == pytest.approx(1.0)
    assert oracle.bound_ratio(Z + 2 * K * 2.0 ** -149, Z, Z, K) == pytest.approx(2.0)
    # non-finite GPU values never pass; the relative bound is the underflow-free special case
    bad = C.copy()
    bad[1, 2] = np.nan
    assert oracle.bound_ratio(bad, C, S, K) == np.inf
    err = oracle.normalised_error(C + tol, C, S, K)
    assert err > 2.0


def test_subnormal_products_of_the_oracle_are_exact():
    # FP64 holds every product of two FP32 values exactly, subnormals included
    # (2^-149 * 2^-149 = 2^-298 is above FP64's 2^-1074): the oracle's C of
    # subnormal operands is the exact rational sum.
    A = inputs.subnormal(68, 3, 4)
    B = inputs.subnormal(69, 4, 2)
    C, _ = oracle.gemm_f64(A, B)
    for i in range(3):
        for j in range(2):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(4))
            assert abs(Fraction(C[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
