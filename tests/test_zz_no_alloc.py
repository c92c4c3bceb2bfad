"""gemm_f32_run_splitk_noalloc: the entry point for callers that cannot
allocate device memory (an allocator being set up or torn down, an arena that
owns all device memory, a path that must not take allocator locks).

It keeps its split-K partial sums in the library's fixed device array instead
of cudaMalloc'd scratch.  Its result must agree with the planned entry point's
split-K SIMT result within the accuracy bound the other tests use, on two calls
in a row (the second call reuses the array the first one left behind).  This
file is collected last so a failure here never hides another test's result.
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


def _planned(A, dA, dB, M, N, K, split):
    import torch
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with g.Plan(M, N, K, variant=g.VARIANT_SIMT, tile_m=64, tile_n=64, stages=2, split_k=split) as p:
        p.run(dA, dB, C)
        assert p.check() == g.OK
    return C.cpu().numpy().astype(np.float64)


def _noalloc(dA, dB, M, N, K, split, lda=None, ldb=None, ldc=None, pad=None):
    import torch
    ldc = ldc or N
    Cbuf = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    if pad is not None and ldc > N:
        Cbuf[:, N:] = pad
    stream = torch.cuda.current_stream()
    s = g.gemm_f32_run_splitk_noalloc(M, N, K, lda or K, ldb or N, ldc, dA.data_ptr(), dB.data_ptr(),
                                      Cbuf.data_ptr(), split, stream.cuda_stream)
    assert s == g.OK, g.gemm_f32_status_string(s)
    stream.synchronize()
    if pad is not None and ldc > N:
        assert (Cbuf[:, N:].cpu().numpy() == pad).all(), "a store landed in C's padding"
    return Cbuf[:, :N].cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape,split", [((300, 200, 1000), 4), ((127, 193, 61), 2), ((513, 257, 129), 3)])
def test_noalloc_matches_planned_entry_twice(shape, split):
    import torch
    M, N, K = shape
    A = inputs.uniform_pm1(1301 + M, M, K)
    B = inputs.uniform_pm1(1302 + N, K, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    Cp = _planned(A, dA, dB, M, N, K, split)
    Cref, S = oracle.gemm_f64(A, B)
    scale = 2.0 * K * 2.0 ** -24 * S
    for _ in range(2):
        Cn = _noalloc(dA, dB, M, N, K, split)
        assert np.isfinite(Cn).all()
        assert np.all(np.abs(Cn - Cp) <= scale), "no-alloc result differs from the planned entry point"
        assert oracle.within_bound(Cn, Cref, S, K)


def test_noalloc_different_shapes_back_to_back():
    # A second call with another shape reuses the array the first one filled.
    import torch
    for (M, N, K, split) in [(256, 512, 2048, 8), (64, 96, 333, 5)]:
        A = inputs.normal(1401 + M, M, K)
        B = inputs.normal(1402 + N, K, N)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        Cp = _planned(A, dA, dB, M, N, K, split)
        Cn = _noalloc(dA, dB, M, N, K, split)
        Cref, S = oracle.gemm_f64(A, B)
        assert np.all(np.abs(Cn - Cp) <= 2.0 * K * 2.0 ** -24 * S)


def test_noalloc_rejects_sizes_beyond_the_array():
    import torch
    # 4 splits x 2048 x 1024 floats = 8.4M floats > 2^21: refused, nothing runs.
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    s = g.gemm_f32_run_splitk_noalloc(2048, 1024, 4096, 4096, 1024, 1024, p, p, p, 4, 0)
    assert s == g.ERR_INVALID_ARG
    assert g.gemm_f32_run_splitk_noalloc(16, 16, 16, 16, 16, 16, p, p, p, 1, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_run_splitk_noalloc(16, 16, 16, 16, 16, 16, p, p, p, 65, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_run_splitk_noalloc(0, 16, 16, 16, 16, 16, 0, 0, 0, 2, 0) == g.OK


def test_noalloc_padded_leading_dimensions():
    # Operands inside wider rows whose padding holds NaN (a read of it would
    # poison the result) and a C whose padding holds a sentinel (a store to it
    # is caught): the same result as the planned entry point on tight copies.
    import torch
    M, N, K, split = 200, 150, 500, 4
    lda, ldb, ldc = K + 7, N + 5, N + 9
    A = inputs.uniform_pm1(1501, M, K, ld=lda)
    B = inputs.uniform_pm1(1502, K, N, ld=ldb)
    dAp = torch.from_numpy(np.lib.stride_tricks.as_strided(A, shape=(M, lda), strides=(4 * lda, 4)).copy()).cuda()
    dBp = torch.from_numpy(np.lib.stride_tricks.as_strided(B, shape=(K, ldb), strides=(4 * ldb, 4)).copy()).cuda()
    assert torch.isnan(dAp[:, K:]).all() and torch.isnan(dBp[:, N:]).all()
    At, Bt = np.ascontiguousarray(A), np.ascontiguousarray(B)
    Cp = _planned(At, torch.from_numpy(At).cuda(), torch.from_numpy(Bt).cuda(), M, N, K, split)
    Cref, S = oracle.gemm_f64(At, Bt)
    for _ in range(2):
        Cn = _noalloc(dAp, dBp, M, N, K, split, lda=lda, ldb=ldb, ldc=ldc, pad=12345.0)
        assert np.isfinite(Cn).all()
        assert np.all(np.abs(Cn - Cp) <= 2.0 * K * 2.0 ** -24 * S)
        assert oracle.within_bound(Cn, Cref, S, K)


def test_noalloc_single_slice_writes_c_directly():
    # K no deeper than one 16-deep K-tile: split_k 2 leaves one slice, which
    # writes C itself (no scratch).  Its size would not fit the array as two
    # slices (2 x 4096 x 1024 floats > 2^21), so only the one-slice path runs it.
    import torch
    M, N, K = 4096, 1024, 16
    A = inputs.uniform_pm1(1503, M, K)
    B = inputs.uniform_pm1(1504, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    Cp = _planned(A, dA, dB, M, N, K, 1)
    Cref, S = oracle.gemm_f64(A, B)
    for _ in range(2):
        Cn = _noalloc(dA, dB, M, N, K, 2)
        assert np.all(np.abs(Cn - Cp) <= 2.0 * K * 2.0 ** -24 * S)
        assert oracle.within_bound(Cn, Cref, S, K)


def test_noalloc_allocates_nothing():
    # After a warm-up call, a call leaves the device's free memory (what the
    # driver reports, so any cudaMalloc in the process would show) and torch's
    # allocator untouched.
    import torch
    M, N, K, split = 256, 384, 1024, 4
    dA = torch.from_numpy(inputs.uniform_pm1(1505, M, K)).cuda()
    dB = torch.from_numpy(inputs.uniform_pm1(1506, K, N)).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    args = (M, N, K, K, N, N, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), split, stream.cuda_stream)
    assert g.gemm_f32_run_splitk_noalloc(*args) == g.OK
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        assert g.gemm_f32_run_splitk_noalloc(*args) == g.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
