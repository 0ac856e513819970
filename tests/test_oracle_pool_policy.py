"""Pins for the oracle's pool order, policy and draw rule (CPU only)."""
import itertools
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import verify as ov

VALUES = [1.0, -1.0, 0.0, -0.0, float("inf"), float("-inf"), float("nan")]


def value_rank(x):
    """The pool's total order, written on values rather than bits: every NaN
    lowest, then ordinary float order, with -0.0 just below +0.0."""
    if math.isnan(x):
        return (0, 0.0, 0)
    return (1, x, 1 if math.copysign(1.0, x) > 0 else 0)


def test_pool_order_matches_value_sort_on_every_tie_pattern():
    for combo in itertools.product(VALUES, repeat=5):
        row = np.array(combo, dtype=np.float32)
        ids, vals = ov.target_pool(row)
        ref = sorted(range(5), key=lambda i: (tuple(-c if isinstance(c, float) else -c
                                                      for c in value_rank(float(row[i]))), i))
        assert list(ids) == ref, combo
        assert np.array_equal(vals.view(np.uint32), row[ref].view(np.uint32))


def test_pool_width():
    rng = np.random.default_rng(0)
    assert len(ov.target_pool(rng.standard_normal(10).astype(np.float32))[0]) == 10
    row = rng.standard_normal(1000).astype(np.float32)
    ids, vals = ov.target_pool(row)
    assert len(ids) == 64
    assert set(ids) == set(np.argsort(-row, kind="stable")[:64])
    # a NaN with a negative sign bit is still the lowest class
    row = np.float32([np.nan, -np.nan, -np.inf, 0.0])
    row[1] = np.frombuffer(np.uint32(0xFFC00001).tobytes(), np.float32)[0]
    assert list(ov.target_pool(row)[0]) == [3, 2, 0, 1]


def test_candidate_pool_breaks_ties_by_id_then_slot():
    ids, vals = ov.candidate_pool([9, 3, 9, 5, 1, 7, 2, 4],
                                  np.float32([1, 1, 1, 2, np.nan, -np.inf, 2, 0]))
    assert list(ids) == [2, 5, 3, 9, 9, 4, 7, 1]


def test_greedy_and_topk_one_are_argmax():
    vals = np.float32([3.0, 2.0, 1.0])
    assert ov.policy_weights(vals, ov.Policy(temperature=0.0)) == (1, [1.0], 1.0)
    m, e, S = ov.policy_weights(vals, ov.Policy(temperature=1.0, top_k=1))
    assert (m, e, S) == (1, [1.0], 1.0)
    assert isinstance(S, np.float32) and isinstance(e[0], np.float32)


def _probs(vals, pol):
    m, e, S = ov.policy_weights(np.float32(vals), pol)
    return np.array([float(x) / float(S) for x in e])


def test_full_pool_is_softmax():
    rng = np.random.default_rng(1)
    for T in (0.3, 0.7, 1.0, 2.5):
        vals = np.sort(rng.standard_normal(64).astype(np.float32) * 3)[::-1]
        p = _probs(vals, ov.Policy(temperature=T, top_k=0))
        ref = softmax(vals.astype(np.float64) / np.float64(np.float32(T)))
        # float32 policy: each weight within a few float32 ulps of the softmax
        np.testing.assert_allclose(p, ref, rtol=1e-5, atol=1e-30)   # z itself is rounded to float32


def test_topk_absent_is_twenty():
    vals = np.sort(np.random.default_rng(2).standard_normal(64).astype(np.float32))[::-1]
    assert ov.policy_weights(vals, ov.Policy(temperature=1.0))[0] == 20
    assert ov.policy_weights(vals, ov.Policy(temperature=1.0, top_k=0))[0] == 64
    assert ov.policy_weights(vals, ov.Policy(temperature=1.0, top_k=200))[0] == 64
    assert ov.policy_weights(vals[:8], ov.Policy(temperature=1.0))[0] == 8


def test_min_p_keeps_tokens_above_fraction_of_max():
    rng = np.random.default_rng(3)
    for trial in range(50):
        vals = np.sort(rng.standard_normal(64).astype(np.float32) * 2)[::-1]
        T, mp = 0.8, float(rng.uniform(0.01, 0.5))
        ref = softmax(vals.astype(np.float64) / np.float64(np.float32(T)))
        ratio = ref / ref[0]
        mp32 = float(np.float32(mp))
        if np.min(np.abs(ratio - mp32)) < 1e-5:
            continue
        p = _probs(vals, ov.Policy(temperature=T, top_k=0, min_p=mp))
        assert len(p) == int(np.sum(ratio >= mp32))


def test_top_p_keeps_the_smallest_prefix_reaching_the_mass():
    rng = np.random.default_rng(4)
    for trial in range(50):
        vals = np.sort(rng.standard_normal(64).astype(np.float32) * 2)[::-1]
        T, tp = 0.7, float(rng.uniform(0.05, 0.99))
        ref = softmax(vals.astype(np.float64) / np.float64(np.float32(T)))
        cum = np.cumsum(ref)
        tp32 = float(np.float32(tp))
        if np.min(np.abs(cum - tp32)) < 1e-5:
            continue
        p = _probs(vals, ov.Policy(temperature=T, top_k=0, top_p=tp))
        assert len(p) == int(np.argmax(cum >= tp32)) + 1
        np.testing.assert_allclose(p, ref[:len(p)] / ref[:len(p)].sum(), rtol=1e-5)


def test_low_temperature_tends_to_argmax():
    vals = np.float32([2.0, 1.9, 1.0])
    p = _probs(vals, ov.Policy(temperature=0.001, top_k=0))
    assert p[0] == 1.0 and p[1] == 0.0          # e_1 = exp(-100) is below the float32 range


def test_nan_and_minus_inf_get_no_mass():
    vals = np.float32([1.0, 0.5, -np.inf, np.nan])
    m, e, S = ov.policy_weights(vals, ov.Policy(temperature=1.0, top_k=0))
    assert e[2] == 0.0 and e[3] == 0.0 and e[1] > 0


def test_draw_matches_weights():
    """The draw rule maps u-intervals to entries with lengths e_j / S."""
    e = [np.float32(x) for x in (1.0, 0.5, 0.0, 0.25, 0.125)]
    S = ov.seq_sum(e)
    N = 100_000
    counts = np.zeros(len(e))
    for i in range(N):
        counts[ov.draw_index(e, S, (i + 0.5) / N)] += 1
    np.testing.assert_allclose(counts / N, np.array(e, np.float64) / float(S), atol=2.0 / N)
    assert ov.draw_index(e, S, np.float32(1.0 - 2**-24)) == 4


def test_top_k_entries_is_a_prefix_of_the_sorted_row():
    """Top-K by brute force: Python's sort on (order key desc, id asc)."""
    rng = np.random.default_rng(70)
    for trial in range(200):
        V = int(rng.integers(1, 40))
        x = rng.choice(np.float32([np.nan, -np.inf, np.inf, 0.0, -0.0, 1.0, -2.5, 7.0]), V)
        k = int(rng.integers(1, 70))
        def key(i):
            b = int(x[i:i + 1].view(np.uint32)[0])
            if np.isnan(x[i]):
                return (-1, -i)
            return ((b ^ 0xFFFFFFFF) if b >> 31 else (b | 0x80000000), -i)
        want = sorted(range(V), key=key, reverse=True)[:k]
        ids, vals = ov.top_k_entries(x, k)
        assert list(ids) == want
        assert np.array_equal(vals.view(np.uint32), x[want].view(np.uint32))
