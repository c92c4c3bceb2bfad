"""Strided-batched GEMM: many independent products in one launch, each checked
against the CPU oracle element by element."""
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


def _run_batched(M, N, K, batch, lda, ldb, ldc, sa, sb, sc, seed, **kw):
    import torch
    As = [inputs.uniform_pm1(seed + 2 * z, M, K) for z in range(batch if sa else 1)]
    Bs = [inputs.normal(seed + 2 * z + 1, K, N) for z in range(batch if sb else 1)]
    dA = torch.full((max(sa * batch, M * lda) + 8,), float("nan"), dtype=torch.float32)
    dB = torch.full((max(sb * batch, K * ldb) + 8,), float("nan"), dtype=torch.float32)
    for z, a in enumerate(As):
        dA[z * sa:z * sa + M * lda].view(M, lda)[:, :K] = torch.from_numpy(a)
    for z, b in enumerate(Bs):
        dB[z * sb:z * sb + K * ldb].view(K, ldb)[:, :N] = torch.from_numpy(b)
    dA, dB = dA.cuda(), dB.cuda()
    dC = torch.full((sc * batch + 8,), 777.0, dtype=torch.float32, device="cuda")
    with g.Plan(M, N, K, lda, ldb, ldc, batch=batch, stride_a=sa, stride_b=sb, stride_c=sc, **kw) as p:
        desc = p.describe()
        s = p.run_ptr(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert s == g.OK
        assert p.check() == g.OK
    C = dC.cpu().numpy()
    worst = 0.0
    for z in range(batch):
        a = As[z if sa else 0]
        b = Bs[z if sb else 0]
        Cref, S = oracle.gemm_f64(a, b)
        got = C[z * sc:z * sc + M * ldc].reshape(M, ldc)[:, :N]
        worst = max(worst, oracle.normalised_error(got, Cref, S, K))
        if ldc > N:  # padding columns untouched
            assert (C[z * sc:z * sc + M * ldc].reshape(M, ldc)[:, N:] == 777.0).all()
    assert (C[sc * batch:] == 777.0).all()
    return worst, desc


@pytest.mark.parametrize("shape,batch", [((32, 32, 32), 256), ((33, 47, 29), 7), ((64, 64, 64), 40),
                                         ((128, 96, 200), 9), ((128, 128, 128), 6), ((127, 193, 61), 3)])
def test_batched_matches_oracle(shape, batch):
    M, N, K = shape
    lda, ldb, ldc = K, N, N
    err, desc = _run_batched(M, N, K, batch, lda, ldb, ldc, M * lda, K * ldb, M * ldc, 1700)
    assert err <= 2.0, (desc, err)
    assert "batch=" in desc


def test_batched_padded_and_shared_b():
    # padded leading dimensions and gaps between products; B shared (stride 0)
    M, N, K, batch = 20, 36, 44, 11
    lda, ldb, ldc = K + 3, N + 5, N + 2
    err, desc = _run_batched(M, N, K, batch, lda, ldb, ldc, M * lda + 17, 0, M * ldc + 9, 1800)
    assert err <= 2.0, (desc, err)


@pytest.mark.parametrize("tile", [32, 64, 128])
def test_batched_forced_tiles(tile):
    M, N, K, batch = 70, 90, 50, 5
    err, desc = _run_batched(M, N, K, batch, K, N, N, M * K, K * N, M * N, 1900,
                             tile_m=tile, tile_n=tile, stages=2)
    assert err <= 2.0 and f"tile={tile}x{tile}" in desc, (desc, err)


def test_batched_k_zero_writes_zeros():
    import torch
    M, N, batch = 9, 13, 6
    dC = torch.full((M * N * batch,), 5.0, dtype=torch.float32, device="cuda")
    with g.Plan(M, N, 0, 1, N, N, batch=batch, stride_a=0, stride_b=0, stride_c=M * N) as p:
        assert p.run_ptr(0, 0, dC.data_ptr(), torch.cuda.current_stream().cuda_stream) == g.OK
        assert p.check() == g.OK
    assert not dC.cpu().numpy().any()
