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


def _noalloc(dA, dB, M, N, K, split, lda=None, ldb=None, ldc=None):
    import torch
    ldc = ldc or N
    Cbuf = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    s = g.gemm_f32_run_splitk_noalloc(M, N, K, lda or K, ldb or N, ldc, dA.data_ptr(), dB.data_ptr(),
                                      Cbuf.data_ptr(), split, stream.cuda_stream)
    assert s == g.OK, g.gemm_f32_status_string(s)
    stream.synchronize()
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
