"""CPU oracle for the FP32 GEMM C = A*B.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference arms may import this package.  The product (``software_pipelined_gb300``)
never imports it and it never imports the product; the two share nothing but
the seeded input generators, which live in a module of their own and hold none
of the product's arithmetic.

The arithmetic lives in ``gemm_oracle.c`` (plain C, FP64 accumulation in
ascending k, i-k-j loop; see its header for the definition and the passages it
follows).  This module compiles it with gcc on first use and wraps it with
ctypes, plus the accuracy criterion the GPU result must meet:

    |C_gpu[i][j] - C[i][j]| <= 2 * K * 2^-24 * S[i][j],   S = sum_k |A_ik||B_kj|

reported as the normalised error  |C_gpu - C| / (K * 2^-24 * S)  (pass iff <= 2;
where S == 0 the GPU value must be exactly 0).

That bound is the usual one for a K-term FP32 dot product and assumes that no
result or intermediate falls below FP32's normal range.  For inputs where one
can, ``bound_ratio`` adds the two absolute terms that hold without that
assumption:

    |C_gpu - C| <= 2 K 2^-24 S + K 2^-149 + 2^-136 T

K 2^-149: gradual underflow (an FP32 operation whose result is subnormal is
off by up to 2^-150, half the subnormal step), K of them per element with a
factor of 2 as in the first term.  2^-136 T, T = ``tf32_grid_term(A, B)``: a
product split into TF32 pieces cannot resolve anything finer than 2^-136
(TF32's smallest subnormal), so an element below 2^-113 in magnitude (whose
remainder after the first piece lies below that step) is carried to within
2^-137; T is the sum of the magnitudes such an element multiplies.  Only the
tensor-core plans have that term (T = None for the SIMT plans).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "libgemm_oracle.so")
_lock = threading.Lock()
_lib = None

EPS_F32 = 2.0 ** -24  # unit roundoff of FP32 round-to-nearest


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into a shared library beside it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_gemm_f64.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, vp, i64]
            lib.oracle_gemm_f64.restype = None
            lib.oracle_gemm_f64_entries.argtypes = [i64, vp, vp, i64, vp, i64, vp, i64, vp, vp]
            lib.oracle_gemm_f64_entries.restype = None
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_get_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_rowmajor_f32(X: np.ndarray, name: str):
    """Return (array, ld) for a 2-D float32 array whose rows may be padded."""
    if X.dtype != np.float32 or X.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if X.strides[1] != 4 or X.strides[0] % 4 != 0 or X.strides[0] < 4 * X.shape[1]:
        X = np.ascontiguousarray(X)
    ld = X.strides[0] // 4 if X.shape[0] > 1 else max(X.shape[1], 1)
    return X, ld


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def gemm_f64(A: np.ndarray, B: np.ndarray, with_scale: bool = True):
    """C = A @ B summed in FP64 in ascending k; also S = |A| @ |B| if asked.

    A: (M, K) float32, B: (K, N) float32; either may be a row-padded view.
    Returns (C, S) as contiguous float64 arrays (S is None if not asked).
    """
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_scale else None
    if M and N:
        _load().oracle_gemm_f64(M, N, K, A.ctypes.data, lda, B.ctypes.data, ldb,
                                C.ctypes.data, S.ctypes.data if S is not None else None, N)
    return C, S


def gemm_f64_entries(A: np.ndarray, B: np.ndarray, rows, cols):
    """C[rows[t], cols[t]] and S[rows[t], cols[t]] for sampled outputs."""
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and equally long")
    M, K = A.shape
    _, N = B.shape
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise IndexError("sample index out of range")
    c = np.empty(rows.size, dtype=np.float64)
    s = np.empty(rows.size, dtype=np.float64)
    if rows.size:
        _load().oracle_gemm_f64_entries(rows.size, rows.ctypes.data, cols.ctypes.data, K,
                                        A.ctypes.data, lda, B.ctypes.data, ldb,
                                        c.ctypes.data, s.ctypes.data)
    return c, s


def normalised_error(C_gpu, C_ref, S_ref, K: int):
    """max over elements of |C_gpu - C_ref| / (K * 2^-24 * S_ref).

    Elements with S_ref == 0 must match exactly: an exact match counts 0, any
    difference counts +inf.  A non-finite GPU value counts +inf.  For K == 0
    the reference is 0 and the GPU value must be exactly 0.
    """
    Cg = np.asarray(C_gpu, dtype=np.float64)
    diff = np.abs(Cg - C_ref)
    scale = max(K, 1) * EPS_F32 * S_ref
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0),
                     np.where(diff == 0, 0.0, np.inf))
    r = np.where(np.isfinite(Cg), r, np.inf)
    return float(r.max()) if r.size else 0.0


TF32_FINEST = 2.0 ** -136   # TF32's smallest subnormal (10 stored mantissa bits below 2^-126)
TF32_FULL = 2.0 ** -113     # smallest magnitude whose TF32 pieces carry it to full FP32 accuracy
UNDERFLOW_STEP = 2.0 ** -149  # FP32's smallest subnormal


def tf32_grid_term(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """T[i][j] = sum_k |B_kj| [0 < |A_ik| < 2^-113] + |A_ik| [0 < |B_kj| < 2^-113],
    in FP64 (a matrix product of the masks with the magnitudes)."""
    a = np.abs(np.asarray(A, dtype=np.float64))
    b = np.abs(np.asarray(B, dtype=np.float64))
    ma = ((a > 0) & (a < TF32_FULL)).astype(np.float64)
    mb = ((b > 0) & (b < TF32_FULL)).astype(np.float64)
    return ma @ b + a @ mb


def bound_ratio(C_gpu, C_ref, S_ref, K: int, T=None) -> float:
    """max over elements of |C_gpu - C_ref| / (2 K 2^-24 S + K 2^-149 + 2^-136 T)
    (pass iff <= 1).  T None: no TF32 term.  A non-finite GPU value counts +inf;
    a zero tolerance (K == 0) demands an exact match."""
    Cg = np.asarray(C_gpu, dtype=np.float64)
    diff = np.abs(Cg - C_ref)
    tol = 2.0 * max(K, 1) * EPS_F32 * S_ref + K * UNDERFLOW_STEP
    if T is not None:
        tol = tol + TF32_FINEST * T
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(tol > 0, diff / np.where(tol > 0, tol, 1.0), np.where(diff == 0, 0.0, np.inf))
    r = np.where(np.isfinite(Cg), r, np.inf)
    return float(r.max()) if r.size else 0.0


def within_bound(C_gpu, C_ref, S_ref, K: int, factor: float = 2.0) -> bool:
    """True iff |C_gpu - C_ref| <= factor * K * 2^-24 * S_ref for every element."""
    return normalised_error(C_gpu, C_ref, S_ref, K) <= factor
