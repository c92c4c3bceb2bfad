"""The seeded input generators: pinned to the published SplitMix64 vector."""
import os

import numpy as np

from software_pipelined_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vector():
    vals = []
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and not line.startswith("seed"):
                vals.append(int(line))
    got = inputs.splitmix64(1234567, len(vals))
    assert [int(x) for x in got] == vals


def test_splitmix64_stream_offsets_and_chunks():
    full = inputs.splitmix64(99, (1 << 22) + 5)
    assert np.array_equal(full[-5:], inputs.splitmix64(99, 5, start=1 << 22))


def test_uniform_grid_and_range():
    U = inputs.uniform_pm1(1001, 64, 64)
    assert U.dtype == np.float32
    assert U.min() >= -1.0 and U.max() < 1.0
    q = U.astype(np.float64) * 2.0 ** 23
    assert np.array_equal(q, np.round(q))
    assert abs(float(U.mean())) < 0.05
    assert abs(float(U.var()) - 1.0 / 3.0) < 0.02


def test_normal_moments():
    Z = inputs.normal(3001, 256, 256)
    assert Z.dtype == np.float32 and np.isfinite(Z).all()
    assert abs(float(Z.mean())) < 0.01
    assert abs(float(Z.std()) - 1.0) < 0.01


def test_deterministic_and_seed_dependent():
    assert np.array_equal(inputs.uniform_pm1(7, 9, 11), inputs.uniform_pm1(7, 9, 11))
    assert not np.array_equal(inputs.uniform_pm1(7, 9, 11), inputs.uniform_pm1(8, 9, 11))


def test_padded_view():
    A = inputs.uniform_pm1(5, 6, 7, ld=12)
    assert A.shape == (6, 7) and A.strides == (48, 4)
    assert np.array_equal(A, inputs.uniform_pm1(5, 6, 7))
    base = np.lib.stride_tricks.as_strided(A, shape=(6, 12), strides=(48, 4))
    assert np.isnan(base[:, 7:]).all()


def test_small_int_range():
    I = inputs.small_int(3, 50, 50)
    assert I.min() >= -8 and I.max() <= 8
    assert np.array_equal(I, np.round(I))


def test_top_of_range_values():
    T = inputs.top_of_range(41, 64, 64)
    bits = np.abs(T).view(np.uint32)
    assert np.isfinite(T).all()
    assert bits.min() >= 0x7F7FE000 and bits.max() <= 0x7F7FFFFF
    # about half would round up into the Inf exponent at 10 mantissa bits
    assert 0.4 < float((bits >= 0x7F7FF000).mean()) < 0.6
    assert 0.4 < float((T < 0).mean()) < 0.6


def test_subnormal_values():
    S = inputs.subnormal(42, 64, 64)
    a = np.abs(S).astype(np.float64)
    assert (a > 0).all() and (a < 2.0 ** -126).all()
    assert a.min() >= 2.0 ** -149
    assert 0.4 < float((S < 0).mean()) < 0.6


def test_scaled_exponents_span_and_exactness():
    X = inputs.scaled_exponents(43, 128, 128, -100, 100)
    u = inputs.uniform_pm1(43, 128, 128).astype(np.float64)
    r = X.astype(np.float64) / np.where(u == 0, 1.0, u)
    e = np.log2(np.abs(r[u != 0]))
    assert np.array_equal(e, np.round(e))       # an exact power of two per element
    assert e.min() == -100 and e.max() == 100
    assert np.array_equal(X, inputs.scaled_exponents(43, 128, 128, -100, 100))
