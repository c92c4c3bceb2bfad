"""Seeded random plans against the oracle: shapes, leading dimensions, base
offsets and forced options drawn from the ranges every kernel form accepts,
each checked element by element at the bound, the canaries intact and the
result the same bits on a second run.  The draws come from a fixed seed, so
a failure names its case and reproduces."""
import numpy as np
import pytest

import software_pipelined_gb300 as g
from software_pipelined_gb300 import inputs

from gpu_util import check_against_oracle, run_gemm

pytestmark = pytest.mark.gpu


def _cases(n=96, seed=20261202):
    rng = np.random.default_rng(seed)
    forms = [
        dict(variant=g.VARIANT_SIMT),
        dict(variant=g.VARIANT_TCGEN05, operand_split=1),
        dict(variant=g.VARIANT_TCGEN05, operand_split=2),
        dict(variant=g.VARIANT_TCGEN05, operand_split=3),
        dict(variant=g.VARIANT_TCGEN05, operand_split=4),
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=256, operand_split=2),
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=256, operand_split=3),
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=256, operand_split=4),
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=128, operand_split=4),
        dict(variant=g.VARIANT_AUTO),
        # the other ways of summing K-slices, and A split into tensor memory
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=256, operand_split=5),
        dict(variant=g.VARIANT_TCGEN05, tile_m=256, tile_n=256, operand_split=4, split_reduce=4),
        dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=128, operand_split=2, split_reduce=2),
        dict(variant=g.VARIANT_TCGEN05, tile_m=128, tile_n=128, operand_split=1, split_reduce=3),
    ]
    out = []
    for i in range(n):
        form = dict(forms[i % len(forms)])
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 700))
        K = int(rng.integers(32, 600))
        # tensor-core forms that read A (or B) by TMA need rows of whole 16-byte
        # chunks; the others take any leading dimension
        tma_a = form.get("operand_split", 0) >= 2 or form.get("tile_m") == 256
        tma_b = form.get("operand_split") == 2
        lda = K + (int(rng.integers(0, 3)) * 4 if tma_a else int(rng.integers(0, 5)))
        ldb = N + (int(rng.integers(0, 3)) * 4 if tma_b else int(rng.integers(0, 5)))
        ldc = N + int(rng.integers(0, 5))
        sk = int(rng.choice([0, 1, 2, 3]))
        if sk and form.get("variant") != g.VARIANT_AUTO:
            form["split_k"] = sk
        out.append((i, M, N, K, lda, ldb, ldc, form))
    return out


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}_{c[1]}x{c[2]}x{c[3]}" for c in CASES])
def test_fuzz_against_the_oracle(case):
    i, M, N, K, lda, ldb, ldc, form = case
    A = inputs.uniform_pm1(7000 + 2 * i, M, K)
    B = inputs.normal(7001 + 2 * i, K, N)
    try:
        C, desc, canaries, outs = run_gemm(A, B, lda=lda, ldb=ldb, ldc=ldc, repeat=2, **form)
    except g.GemmError as e:
        # a forced form that cannot take this shape must say so at plan time
        assert e.status == g.ERR_UNSUPPORTED, (form, str(e))
        return
    assert canaries, desc
    assert np.array_equal(outs[0], outs[1]), desc
    err, ok = check_against_oracle(C, A, B)
    assert ok, f"{desc}: {err}"
