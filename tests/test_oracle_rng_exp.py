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
    assert u.min() >= 0.0 and u.max() < 1.0
    counts, _ = np.histogram(u, bins=100, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-4
    # different (row, purpose) addresses give unrelated streams
    v = philox.uniform_array(np.arange(200_000, dtype=np.uint64), 17, 1, 2)
    assert abs(np.corrcoef(u, v)[0, 1]) < 0.01


def _ulp(x):
    return math.ulp(x)


def test_vexp_special_values():
    assert vx.vexp(0.0) == 1.0
    assert vx.vexp(-0.0) == 1.0
    assert vx.vexp(float("nan")) == 0.0
    assert vx.vexp(-708.5) == 0.0
    assert vx.vexp(-math.inf) == 0.0
    assert vx.vexp(math.log(2.0)) == pytest.approx(2.0, rel=2**-51)
    assert vx.vexp(-708.0) > 0.0


def test_vexp_within_two_ulp_of_libm():
    rng = np.random.default_rng(1)
    zs = np.concatenate([rng.uniform(-708.0, 0.0, 100_000), rng.uniform(-2.0, 0.0, 50_000),
                         -np.arange(0, 1022) * math.log(2.0),          # reduction boundaries
                         -(np.arange(0, 1021) + 0.5) * math.log(2.0)])  # ties of the rounding
    worst = 0.0
    for z in zs:
        ref = math.exp(z)
        err = abs(vx.vexp(z) - ref) / _ulp(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_vexp_against_high_precision():
    getcontext().prec = 50
    rng = np.random.default_rng(2)
    for z in rng.uniform(-700.0, 0.0, 300):
        exact = Decimal(float(z)).exp()
        got = Decimal(vx.vexp(z))
        assert abs(got - exact) <= Decimal(_ulp(float(exact))) * Decimal(1.5)


def test_vexp_reduction_constants():
    getcontext().prec = 60
    ln2 = Decimal(2).ln()
    c1_bits = struct.unpack("<Q", struct.pack("<d", vx.LN2_C1))[0]
    assert c1_bits & 0xFFFFFFFF == 0                      # n*C1 exact for |n| < 2**32
    assert abs(Decimal(vx.LN2_C1) + Decimal(vx.LN2_C2) - ln2) < Decimal("1e-22")
    assert abs(Decimal(vx.INV_LN2) - 1 / ln2) <= Decimal(_ulp(vx.INV_LN2)) / 2
