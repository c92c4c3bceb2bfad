"""Helpers for the GPU parity tests: device buffers with canaries, runs through
the C-ABI binding, and comparison with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
import software_pipelined_gb300 as g

SENTINEL = 12345.0
GUARD = 64  # floats of canary before and after C


def device_matrix(host: np.ndarray, ld: int, offset: int = 0):
    """Copy a rows x cols float32 host matrix to a device buffer with leading
    dimension ld, starting `offset` floats into the allocation (offset 1 gives
    a base address that is not 16-byte aligned).  Padding holds NaN."""
    import torch
    rows, cols = host.shape
    n = offset + (rows * ld if rows else 0) + 4
    buf = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    if rows and cols:
        full = np.full((rows, ld), np.nan, dtype=np.float32)
        full[:, :cols] = host
        buf[offset:offset + rows * ld] = torch.from_numpy(full.reshape(-1)).cuda()
    view = buf[offset:offset + rows * ld].view(rows, ld)[:, :cols] if rows else buf[offset:offset].view(0, cols)
    return buf, view


class GuardedC:
    """C (M x N, ldc) inside a buffer whose margins and padding hold a sentinel;
    C itself starts as NaN so that every element must be written."""

    def __init__(self, M, N, ldc, offset=0):
        import torch
        self.M, self.N, self.ldc, self.offset = M, N, ldc, offset
        self.total = GUARD + offset + M * ldc + GUARD
        self.buf = torch.full((self.total,), SENTINEL, dtype=torch.float32, device="cuda")
        start = GUARD + offset
        self.mat = self.buf[start:start + M * ldc].view(M, ldc) if M else None
        if M and N:
            self.mat[:, :N] = float("nan")
        self.C = self.mat[:, :N] if M else self.buf[start:start].view(0, N)

    def ptr(self) -> int:
        return self.buf.data_ptr() + 4 * (GUARD + self.offset)

    def result(self) -> np.ndarray:
        return self.C.cpu().numpy().astype(np.float64)

    def canaries_intact(self) -> bool:
        h = self.buf.cpu().numpy()
        start = GUARD + self.offset
        if not (h[:start] == SENTINEL).all() or not (h[start + self.M * self.ldc:] == SENTINEL).all():
            return False
        if self.M and self.ldc > self.N:
            pad = h[start:start + self.M * self.ldc].reshape(self.M, self.ldc)[:, self.N:]
            return bool((pad == SENTINEL).all())
        return True


def run_gemm(A: np.ndarray, B: np.ndarray, lda=None, ldb=None, ldc=None, a_off=0, b_off=0, c_off=0,
             repeat=1, **plan_kwargs):
    """Run C = A*B on the GPU through the C-ABI.  Returns (C as float64, plan
    description, canaries intact, list of every repeat's result)."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)
    _, dA = device_matrix(A, lda, a_off)
    _, dB = device_matrix(B, ldb, b_off)
    gc = GuardedC(M, N, ldc, c_off)
    plan = g.Plan(M, N, K, lda, ldb, ldc, **plan_kwargs)
    try:
        outs = []
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(repeat):
            s = plan.run_ptr(dA.data_ptr() if M and K else 0, dB.data_ptr() if K and N else 0,
                             gc.ptr(), stream)
            assert s == g.OK, g.gemm_f32_status_string(s)
            s = plan.check()
            assert s == g.OK, g.gemm_f32_status_string(s)
            outs.append(gc.result())
        return outs[-1], plan.describe(), gc.canaries_intact(), outs
    finally:
        plan.close()


def check_against_oracle(C_gpu, A, B, factor=2.0):
    C, S = oracle.gemm_f64(A, B)
    K = A.shape[1]
    err = oracle.normalised_error(C_gpu, C, S, K)
    return err, err <= factor
