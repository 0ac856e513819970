"""Host-side draft proposal and window pricing (CPU only): the library's C
functions against the oracle, and the oracle against hand-worked cases, the
pages' own cost table and closed forms ("Speculative decoding on RDNA"
§05-§07; "One RDNA4 verify pass has slack for about two dozen speculative
tokens", "Spend the budget on a tree")."""
import json
import math
import os

import numpy as np
import pytest

from oracle import draft_policy as od
from speculative_decoding_verify_row_gb300 import build as vbuild


@pytest.fixture(scope="module")
def vb():
    vbuild.build()
    from speculative_decoding_verify_row_gb300 import binding
    binding.lib()
    return binding


# ---------------------------------------------------------------------------
# n-gram proposal: oracle pins

def test_most_recent_match_for_one_branch():
    #          0  1  2  3  4  5  6  7  8  9 10 11 12 13 14
    ctx = [1, 2, 3, 4, 9, 9, 1, 2, 3, 5, 7, 1, 2, 3]
    # key (1 2 3) occurs at 0 (-> 4 9) and 6 (-> 5 7): both once, 6 is later
    assert od.ngram_propose(ctx, 3, 2, 1, 63) == ([5, 7], [-1, 0])
    assert od.ngram_propose(ctx, 3, 2, 2, 63) == ([5, 7, 4, 9], [-1, 0, -1, 2])


def test_frequent_continuation_ranks_first_and_prefixes_are_shared():
    ctx = [8, 6, 5, 7, 8, 6, 5, 7, 8, 6, 5, 3, 0, 8, 6]
    # key (8 6) at 0, 4 (-> 5 7) and 8 (-> 5 3): (5 7) twice beats the later (5 3)
    toks, par = od.ngram_propose(ctx, 2, 2, 2, 63)
    assert (toks, par) == ([5, 7, 3], [-1, 0, 0])
    # a third branch does not exist: same tree
    assert od.ngram_propose(ctx, 2, 2, 3, 63) == (toks, par)
    # node budget: stops after two nodes
    assert od.ngram_propose(ctx, 2, 2, 2, 2) == ([5, 7], [-1, 0])


def test_no_match_and_short_contexts():
    assert od.ngram_propose([1, 2, 3, 4], 2, 3, 1, 63) == ([], [])
    assert od.ngram_propose([1, 2], 2, 3, 1, 63) == ([], [])
    # a continuation cut by the end of the context is shorter
    assert od.ngram_propose([4, 4, 4], 2, 3, 1, 63) == ([4], [-1])


def _paths(tokens, parent):
    out = []
    for j in range(len(tokens)):
        path, node = [], j
        while node >= 0:
            path.append(tokens[node])
            node = parent[node]
        out.append(tuple(path[::-1]))
    return out


def test_proposal_tree_invariants():
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(0, 200))
        ctx = list(rng.integers(0, 4, n))
        match, propose = int(rng.integers(1, 4)), int(rng.integers(1, 9))
        branches, cap = int(rng.integers(1, 5)), int(rng.integers(0, 30))
        toks, par = od.ngram_propose(ctx, match, propose, branches, cap)
        assert len(toks) <= min(cap, branches * propose)
        conts = set()
        if n > match:
            key = ctx[n - match:]
            for s in range(n - match):
                if ctx[s:s + match] == key:
                    conts.add(tuple(ctx[s + match:s + match + propose]))
        for j, p in enumerate(par):
            assert -1 <= p < j
        # every node spells a prefix of a real continuation; siblings differ
        for path in _paths(toks, par):
            assert any(c[:len(path)] == path for c in conts)
        assert len(set(zip(par, toks))) == len(toks)
        if conts and cap > 0:
            assert len(toks) > 0


# ---------------------------------------------------------------------------
# n-gram proposal: library against the oracle

def test_library_ngram_matches_oracle(vb):
    rng = np.random.default_rng(6)
    for trial in range(400):
        n = int(rng.integers(0, 400))
        ctx = rng.integers(0, int(rng.integers(2, 12)), n).astype(np.int32)
        match, propose = int(rng.integers(1, 6)), int(rng.integers(1, 10))
        branches, cap = int(rng.integers(1, 6)), int(rng.integers(0, 64))
        toks, par = vb.ngram_propose(ctx, match, propose, branches, cap)
        rt, rp = od.ngram_propose(ctx, match, propose, branches, cap)
        assert list(toks) == rt and list(par) == rp, trial


def test_library_ngram_defaults_give_a_chain_of_three(vb):
    ctx = np.int32([0, 1, 2, 3, 4, 8, 7, 6, 9, 0, 1, 2, 3, 4])
    toks, par = vb.ngram_propose(ctx)            # match 5, propose 3
    assert list(toks) == [8, 7, 6] and list(par) == [-1, 0, 1]


# ---------------------------------------------------------------------------
# window cost model (§05)

def test_break_even_table_from_the_fits(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sec05_window_cost.json")))
    for card, (a, b) in g["fits_ms"].items():
        for rows, tokens in g["break_even_tokens"][card].items():
            rows = int(rows)
            assert round((a + b * (rows - 1)) / a, 2) == tokens, (card, rows)


def test_fit_recovers_the_pages_fits(vb, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "sec05_window_cost.json")))
    for a, b in g["fits_ms"].values():
        rows = np.arange(1, 9)
        ms = a + b * (rows - 1)
        for fa, fb in (od.cost_fit(rows, ms), vb.cost_fit(rows, ms)):
            assert abs(fa - a) < 1e-9 and abs(fb - b) < 1e-9


def test_library_fit_matches_oracle_on_noisy_samples(vb):
    rng = np.random.default_rng(7)
    for trial in range(100):
        n = int(rng.integers(2, 40))
        rows = rng.integers(1, 26, n)
        if len(set(rows)) < 2:
            rows[0], rows[1] = 1, 2
        ms = 0.18 + 0.002 * (rows - 1) + rng.normal(0, 0.01, n)
        a, b = vb.cost_fit(rows, ms)
        ra, rb = od.cost_fit(rows, ms)
        assert math.isclose(a, ra, rel_tol=1e-9, abs_tol=1e-12)
        assert math.isclose(b, rb, rel_tol=1e-7, abs_tol=1e-12)


# ---------------------------------------------------------------------------
# expected emitted tokens and the depth choice (§05)

def test_expected_emitted_closed_forms():
    for alpha in (0.0, 0.3, 0.77, 1.0):
        for k in range(0, 9):
            want = k + 1.0 if alpha == 1.0 else (1 - alpha ** (k + 1)) / (1 - alpha)
            assert math.isclose(od.expected_emitted([alpha] * k, k), want, rel_tol=1e-12)
    # the first draft never accepted: one token whatever the depth
    assert od.expected_emitted([0.0, 1.0, 1.0], 3) == 1.0


def test_expected_emitted_by_simulation():
    rng = np.random.default_rng(8)
    alpha = [0.9, 0.6, 0.8, 0.3]
    u = rng.random((200_000, 4))
    accepted = np.cumprod(u < np.array(alpha), axis=1).sum(axis=1)
    assert abs((accepted + 1).mean() - od.expected_emitted(alpha, 4)) < 0.01


def test_depth_choice_at_the_pages_break_even(vb, golden_dir):
    """Halo fit: one draft pays once 1 + alpha exceeds 37.4 / 30.5 = 1.226."""
    a, b = json.load(open(os.path.join(golden_dir, "sec05_window_cost.json")))["fits_ms"][
        "strix_halo_gfx1151"]
    for fn in (lambda al: od.choose_depth(al, 1, a, b), lambda al: vb.choose_depth(al, a, b)):
        assert fn([0.22])[0] == 0
        assert fn([0.23])[0] == 1
    # exactly at break-even (1.25 tokens for 1.25x the cost, all exact in binary)
    # the plain step is kept: a window must be strictly better
    for fn in (lambda al: od.choose_depth(al, 1, 32.0, 8.0), lambda al: vb.choose_depth(al, 32.0, 8.0)):
        assert fn([0.25]) == (0, 1 / 32.0)
        assert fn([0.2500001])[0] == 1


def test_depth_choice_special_cases(vb):
    assert vb.choose_depth([0.0] * 7, 30.0, 7.0) == (0, 1 / 30.0)
    k, _ = vb.choose_depth([1.0] * 7, 30.0, 7.0)
    assert k == 7
    assert vb.choose_depth([], 30.0, 7.0, kmax=0) == (0, 1 / 30.0)
    # nearly flat cost: every extra draft still pays, so the deepest window
    k, _ = vb.choose_depth([0.8] * 24, 0.2, 1e-6)
    assert k == 24
    # a steeper slope stops where the next draft's expected token no longer
    # pays for its row: E(k) = 5 (1 - 0.8^(k+1)), cost 0.2 + 0.0005 k
    k, _ = vb.choose_depth([0.8] * 24, 0.2, 0.0005)
    rates = [5 * (1 - 0.8 ** (j + 1)) / (0.2 + 0.0005 * j) for j in range(25)]
    assert k == int(np.argmax(rates)) and 0 < k < 24


def test_library_depth_choice_matches_oracle(vb):
    rng = np.random.default_rng(9)
    for trial in range(500):
        kmax = int(rng.integers(0, 25))
        alpha = rng.random(kmax) ** rng.uniform(0.1, 3)
        a, b = float(rng.uniform(0.1, 40)), float(rng.uniform(0, 20))
        k, rate = vb.choose_depth(alpha, a, b)
        rk, rrate = od.choose_depth(alpha, kmax, a, b)
        assert math.isclose(rate, rrate, rel_tol=1e-12)
        rates = sorted(od.expected_emitted(alpha, j) / (a + b * j) for j in range(kmax + 1))
        if len(rates) < 2 or rates[-1] - rates[-2] > 1e-9 * rates[-1]:
            assert k == rk


# ---------------------------------------------------------------------------
# takeover (§06) and the AR floor (§07)

def test_takeover(vb):
    # equal pricing takes over (the n-gram rate only has to match the native one)
    assert vb.takeover([0.7, 0.7], [0.7, 0.7], 30.0, 7.0) and od.takeover([0.7] * 2, 2, [0.7] * 2, 2, 30.0, 7.0)
    rng = np.random.default_rng(10)
    for trial in range(300):
        kn, kg = int(rng.integers(0, 9)), int(rng.integers(1, 9))
        an, ag = rng.random(kn), rng.random(kg)
        a, b = float(rng.uniform(1, 40)), float(rng.uniform(0, 20))
        assert vb.takeover(an, ag, a, b) == od.takeover(an, kn, ag, kg, a, b)


def test_ar_floor(vb):
    for fn in (lambda ar, w, e: vb.ar_floor(ar, w, e), od.ar_floor):
        assert fn(25.0, [40.0, 60.0], [2, 2])                 # 20 ms per token < 25
        assert not fn(25.0, [50.0, 75.0], [2, 3])             # ties retire
        assert not fn(25.0, [80.0, 90.0, 70.0], [1, 2, 2])    # nothing cheaper
        assert not fn(25.0, [10.0, float("nan")], [1, 1])     # invalid timing
        assert not fn(25.0, [10.0, 20.0], [1, 0])             # a probe emitting nothing
        assert not fn(0.0, [10.0], [2])
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(1, 4))
        w = rng.uniform(10, 100, n)
        e = rng.integers(1, 5, n)
        ar = float(rng.uniform(10, 40))
        assert vb.ar_floor(ar, w, e) == od.ar_floor(ar, list(w), list(e))


def test_host_entry_points_reject_bad_arguments(vb):
    with pytest.raises(vb.VerifyRowError):
        vb.ngram_propose([1, 2, 3], match=0)
    with pytest.raises(vb.VerifyRowError):
        vb.ngram_propose([1, 2, 3], max_nodes=64)
    with pytest.raises(vb.VerifyRowError):
        vb.cost_fit([4, 4, 4], [1.0, 2.0, 3.0])
    with pytest.raises(vb.VerifyRowError):
        vb.cost_fit([1], [1.0])
    with pytest.raises(vb.VerifyRowError):
        vb.choose_depth([1.5], 30.0, 7.0)
    with pytest.raises(vb.VerifyRowError):
        vb.choose_depth([0.5], 0.0, 7.0)
    with pytest.raises(vb.VerifyRowError):
        vb.choose_depth([0.5] * 64, 30.0, 7.0)
    with pytest.raises(vb.VerifyRowError):
        vb.choose_depth([0.5, 0.5], 1.0, -0.6)                # cost turns negative
    with pytest.raises(vb.VerifyRowError):
        vb.takeover([0.5], [], 30.0, 7.0)
