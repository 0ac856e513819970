"""Pins for the oracle's random stream and exponential (CPU only).

Philox4x64-10 is pinned to numpy's own implementation of the same generator
(numpy.random.Philox, which advances its counter by one before each block);
vexp is pinned to libm's exp by an error bound and to exact special values.
"""
import math
import struct
from decimal import Decimal, getcontext

import numpy as np
import pytest
from scipy import stats

from oracle import philox, vexp as vx

CASES = [
    ((0, 0, 0, 0), (0, 0)),
    ((5, 0, 1, 2), (1234, 0)),
    ((2**64 - 1, 7, 0, 0), (99, 3)),          # carry into counter word 1
    ((2**64 - 1, 2**64 - 1, 2**63, 9), (2**64 - 1, 2**62 + 17)),
    ((123456789, 42, 1, 0), (0xDEADBEEFCAFEF00D, 0)),
]


def _next_counter(c):
    """numpy's Philox increments the 256-bit counter before generating."""
    v = (c[0] | c[1] << 64 | c[2] << 128 | c[3] << 192) + 1
    v &= (1 << 256) - 1
    return tuple((v >> (64 * i)) & philox.MASK64 for i in range(4))


@pytest.mark.parametrize("counter,key", CASES)
def test_philox_matches_numpy(counter, key):
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array(counter, dtype=np.uint64))
    st = bg.state["state"]
    assert [int(x) for x in st["counter"]] == list(counter)
    assert [int(x) for x in st["key"]] == list(key)
    ref = [int(x) for x in bg.random_raw(4)]
    assert list(philox.philox4x64_10(_next_counter(counter), key)) == ref


def test_philox_array_matches_scalar():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 2**63, size=(4, 50), dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    k = rng.integers(0, 2**63, size=(2, 50), dtype=np.uint64)
    out = philox.philox4x64_10_array(c[0], c[1], c[2], c[3], k[0], k[1])
    for i in range(50):
        ref = philox.philox4x64_10([int(x) for x in c[:, i]], [int(x) for x in k[:, i]])
        assert tuple(int(o[i]) for o in out) == ref


def test_uniform_array_matches_scalar():
    seeds = np.arange(40, dtype=np.uint64) * np.uint64(977) + np.uint64(5)
    arr = philox.uniform_array(seeds, 4096, 3, philox.PURPOSE_EMIT)
    for s, u in zip(seeds, arr):
        assert philox.uniform(int(s), 4096, 3, philox.PURPOSE_EMIT) == u


def test_uniform_is_uniform():
    u = philox.uniform_array(np.arange(200_000, dtype=np.uint64), 17, 1, 1)
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    counts, _ = np.histogram(u, bins=100, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-4
    # different (row, purpose) addresses give unrelated streams
    v = philox.uniform_array(np.arange(200_000, dtype=np.uint64), 17, 1, 2)
    assert abs(np.corrcoef(u, v)[0, 1]) < 0.01


def _ulp32(x):
    x = np.float32(abs(x))
    return float(np.nextafter(x, np.float32(np.inf)) - x)


def test_vexp_special_values():
    assert vx.vexp(0.0) == 1.0 and isinstance(vx.vexp(0.0), np.float32)
    assert vx.vexp(-0.0) == 1.0
    assert vx.vexp(float("nan")) == 0.0
    assert vx.vexp(-87.5) == 0.0
    assert vx.vexp(-math.inf) == 0.0
    assert vx.vexp(np.float32(math.log(2.0))) == pytest.approx(2.0, rel=2**-22)
    assert vx.vexp(-87.0) > 0.0 and vx.vexp(-87.0) >= np.finfo(np.float32).tiny


def test_vexp_within_two_float32_ulp_of_libm():
    rng = np.random.default_rng(1)
    zs = np.concatenate([rng.uniform(-87.0, 0.0, 200_000), rng.uniform(-2.0, 0.0, 100_000),
                         -np.arange(0, 126) * math.log(2.0),           # reduction boundaries
                         -(np.arange(0, 125) + 0.5) * math.log(2.0)]).astype(np.float32)
    worst = 0.0
    for z in zs:
        ref = math.exp(float(z))                                      # exact input, libm result
        err = abs(float(vx.vexp(z)) - ref) / _ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_vexp_against_high_precision():
    getcontext().prec = 50
    rng = np.random.default_rng(2)
    for z in rng.uniform(-87.0, 0.0, 500).astype(np.float32):
        exact = Decimal(float(z)).exp()
        got = Decimal(float(vx.vexp(z)))
        assert abs(got - exact) <= Decimal(_ulp32(float(exact))) * Decimal(1.5)


def test_vexp_reduction_constants():
    getcontext().prec = 60
    ln2 = Decimal(2).ln()
    c1_bits = int(np.float32(vx.LN2_C1).view(np.uint32))
    assert c1_bits & 0xFF == 0                            # n*C1 exact for |n| < 256
    assert abs(Decimal(float(vx.LN2_C1)) + Decimal(float(vx.LN2_C2)) - ln2) < Decimal("1e-13")
    assert abs(Decimal(float(vx.INV_LN2)) - 1 / ln2) <= Decimal(_ulp32(float(vx.INV_LN2))) / 2
    from fractions import Fraction
    for j, c in enumerate(vx.TAYLOR):
        exact = Fraction(1, math.factorial(j))
        assert abs(Fraction(float(c)) - exact) <= Fraction(_ulp32(float(c))) / 2, j
