"""Maximum sizes: operands and results with more than 2^31 elements, so every
element offset past the 2^31 boundary must be computed in 64 bits (the
kernels' C stores, the SIMT tile copies, the operand pre-pass's transposed B,
the tensor maps).  Rows on both sides of the boundary are checked against the
oracle, and guard values past the end of C must stay untouched.  The checks
run on the device where the buffers are too large to copy back."""
import numpy as np
import pytest

import oracle
import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 12345.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from software_pipelined_gb300 import build
    build.build()
    g.load()
    yield
    torch.cuda.empty_cache()


def _rows_around(boundary_elems, ld, M):
    r = boundary_elems // ld
    return np.unique(np.clip(np.array([0, r - 1, r, r + 1, M - 1]), 0, M - 1))


def _check_rows(C, A, B, rows, K):
    import torch
    N = B.shape[1]
    rr = np.repeat(rows, N)
    cc = np.tile(np.arange(N), len(rows))
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy().reshape(-1).astype(np.float64)
    ref, S = oracle.gemm_f64_entries(A, B, rr, cc)
    return oracle.normalised_error(got, ref, S, K)


@pytest.mark.parametrize("variant", [g.VARIANT_TCGEN05, g.VARIANT_SIMT], ids=["tcgen05", "simt"])
def test_result_past_2_31_elements(variant):
    import torch
    M, N, K = 65543, 40003, 40          # C: 2.62e9 elements (10.5 GB); ragged M and N
    A = inputs.uniform_pm1(1901, M, K)
    B = inputs.uniform_pm1(1902, K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    buf = torch.full((M * N + GUARD,), SENTINEL, dtype=torch.float32, device="cuda")
    C = buf[:M * N].view(M, N)
    C.fill_(float("nan"))
    try:
        with g.Plan(M, N, K, variant=variant) as p:
            assert p.run_ptr(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 0) == g.OK
            assert p.check(0) == g.OK
            desc = p.describe()
        torch.cuda.synchronize()
        assert not torch.isnan(C).any().item(), f"{desc}: unwritten elements"
        assert (buf[M * N:] == SENTINEL).all().item(), f"{desc}: wrote past C"
        err = _check_rows(C, A, B, _rows_around(2 ** 31, N, M), K)
        assert err <= 2, f"{desc}: max normalised error {err}"
    finally:
        del buf, C, dA, dB
        torch.cuda.empty_cache()


def test_operand_past_2_31_elements():
    import torch
    # B: 2.62e9 elements (10.5 GB); its transposed hi/lo pieces as many each.
    # B is generated in 64-row chunks (seeded per chunk) straight into the
    # device buffer; the columns the check samples are kept on the host.
    M, N, K = 200, 40003, 65536
    A = inputs.uniform_pm1(1903, M, K)
    cols = np.array([0, 1, 20000, 40001, 40002])
    dA = torch.from_numpy(A).cuda()
    dB = torch.empty((K, N), dtype=torch.float32, device="cuda")
    Bcols = np.empty((K, len(cols)), dtype=np.float32)
    CH = 64
    for k0 in range(0, K, CH):
        chunk = inputs.uniform_pm1(1904 + k0 // CH, CH, N)
        dB[k0:k0 + CH].copy_(torch.from_numpy(chunk))
        Bcols[k0:k0 + CH] = chunk[:, cols]
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    try:
        with g.Plan(M, N, K, variant=g.VARIANT_TCGEN05, operand_split=1) as p:
            assert p.run_ptr(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 0) == g.OK
            assert p.check(0) == g.OK
            desc = p.describe()
        torch.cuda.synchronize()
        rows = np.array([0, 99, 199])
        rr, ci = np.repeat(rows, len(cols)), np.tile(np.arange(len(cols)), len(rows))
        got = C[torch.from_numpy(rr).cuda(), torch.from_numpy(cols[ci]).cuda()].cpu().numpy().astype(np.float64)
        ref, S = oracle.gemm_f64_entries(A, Bcols, rr, ci)
        err = oracle.normalised_error(got, ref, S, K)
        assert err <= 2, f"{desc}: max normalised error {err}"
        assert not torch.isnan(C).any().item(), desc
    finally:
        del C, dA, dB
        torch.cuda.empty_cache()
