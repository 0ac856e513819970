"""Pins for the oracle's acceptance rules (CPU only)."""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

from oracle import verify as ov
from oracle.philox import PURPOSE_ACCEPT, PURPOSE_EMIT


def test_figure_01_window(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "fig01_window.json")))
    vid = {w: i for i, w in enumerate(g["vocab"])}
    res = ov.verify_window(np.float32(g["logits"]), [vid[w] for w in g["drafts"]],
                           hist=[vid[w] for w in g["emitted_so_far"]], pol=ov.Policy())
    assert [g["vocab"][t] for t in res.emitted] == g["expected_emitted"]
    assert res.accept == g["expected_accept"]


def _logits_with_argmax(argmax, V, rng):
    x = rng.standard_normal((len(argmax), V)).astype(np.float32)
    for r, t in enumerate(argmax):
        x[r, t] = x[r].max() + 1.0
    return x


def test_greedy_accepts_the_targets_own_chain():
    rng = np.random.default_rng(0)
    for k in range(0, 9):
        am = list(rng.integers(0, 50, k + 1))
        res = ov.verify_window(_logits_with_argmax(am, 50, rng), am[:k], pol=ov.Policy())
        assert res.accept == k and res.n_emitted == k + 1 and res.emitted == am


def test_greedy_stops_at_the_first_mismatch():
    rng = np.random.default_rng(1)
    am = [4, 7, 9, 11]
    drafts = [4, 7, 3]                      # row 2 perturbed
    res = ov.verify_window(_logits_with_argmax(am, 20, rng), drafts, pol=ov.Policy())
    assert res.accept == 2 and res.n_emitted == 3 and res.emitted == [4, 7, 9]


def _brute_force_tree(argmax, tokens, parent):
    """Longest agreeing branch, by walking every node's ancestor path."""
    best, best_depth = -1, 0
    for j in range(len(tokens)):
        path, ok, node = [], True, j
        while node >= 0:
            p = parent[node]
            prow = 0 if p < 0 else 1 + p
            ok &= tokens[node] == argmax[prow]
            path.append(node)
            node = p
        if ok and len(path) > best_depth:
            best, best_depth = j, len(path)
    path = []
    node = best
    while node >= 0:
        path.append(tokens[node])
        node = parent[node]
    return path[::-1] + [argmax[0 if best < 0 else 1 + best]], best_depth


def test_tree_greedy_matches_brute_force():
    rng = np.random.default_rng(2)
    for trial in range(3000):
        n = int(rng.integers(0, 9))
        parent = [int(rng.integers(-1, j)) if j else -1 for j in range(n)]
        tokens = [int(t) for t in rng.integers(0, 3, n)]
        argmax = [int(t) for t in rng.integers(0, 3, n + 1)]
        assert ov.accept_greedy(argmax, tokens, parent) == _brute_force_tree(argmax, tokens, parent)


def test_single_branch_tree_is_the_chain_rule():
    rng = np.random.default_rng(3)
    for trial in range(500):
        k = int(rng.integers(0, 7))
        drafts = [int(t) for t in rng.integers(0, 2, k)]
        argmax = [int(t) for t in rng.integers(0, 2, k + 1)]
        a = next((i for i in range(k) if drafts[i] != argmax[i]), k)
        emitted, acc = ov.accept_greedy(argmax, drafts, ov.chain_parents(k))
        assert acc == a and emitted == drafts[:a] + [argmax[a]]


def _dist(ids, probs):
    probs = [np.float32(x) for x in probs]
    return ov.RowDist(list(ids), probs, ov.seq_sum(probs))


def test_accept_predicate_is_min_one_p_over_q():
    p = [_dist([0, 1], [0.3, 0.7]), _dist([0], [1.0])]
    q = [_dist([0, 1], [0.6, 0.4])]
    # p(0)/q(0) = 0.5: u1 just below accepts, just above rejects
    for u1, acc in ((0.4999, 1), (0.5001, 0)):
        res, a = ov.accept_rejection_chain(p, q, [0], lambda r, k: u1 if k == PURPOSE_ACCEPT else 0.1)
        assert a == acc
    # p(1) > q(1): always accepted
    res, a = ov.accept_rejection_chain(p, q, [1], lambda r, k: 0.999999 if k == PURPOSE_ACCEPT else 0.1)
    assert a == 1
    # on rejection the residual (p - q)+ is {1: 0.3}: token 1 whatever u2
    res, a = ov.accept_rejection_chain(p, q, [0], lambda r, k: 0.9 if k == PURPOSE_ACCEPT else 0.01)
    assert res == [1] and a == 0


class _Need(Exception):
    def __init__(self, key):
        self.key = key


def _explore(run, breakpoints):
    """Exact distribution of run(uniforms) over independent uniforms, for a
    run that is piecewise constant in each uniform with jumps only at the
    given breakpoints: evaluate at interval midpoints, weight by length."""
    out = {}

    def go(fixed, weight):
        def uniforms(row, purpose):
            key = (row, purpose)
            if key in fixed:
                return fixed[key]
            raise _Need(key)
        try:
            result = run(uniforms)
        except _Need as need:
            pts = sorted(set([0.0, 1.0] + [b for b in breakpoints(need.key) if 0.0 < b < 1.0]))
            for lo, hi in zip(pts[:-1], pts[1:]):
                if hi > lo:
                    go({**fixed, need.key: 0.5 * (lo + hi)}, weight * (hi - lo))
            return
        out[result] = out.get(result, 0.0) + weight
    go({}, 1.0)
    return out


def _chain_case(V, k, T, seed, qids=None):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    if qids is None:
        qids = np.stack([rng.permutation(V)[:8] if V >= 8 else
                         np.concatenate([rng.permutation(V), rng.integers(0, V, 8 - V)])
                         for _ in range(k)]).astype(np.int64)
    qlog = (rng.standard_normal((k, 8)) * 2.0).astype(np.float32)
    return logits, qids, qlog


@pytest.mark.parametrize("V,k,T,seed", [(6, 1, 1.0, 10), (6, 2, 0.7, 11), (5, 2, 1.6, 12)])
def test_rejection_sampling_is_exact_by_enumeration(V, k, T, seed):
    """Exact law of the emitted tokens, integrated over every draft outcome
    and every accept / residual / bonus uniform: the first token follows the
    target softmax of row 0, and the token at depth j, given the window got
    there, follows the softmax of row j (full pool: p is a plain softmax)."""
    logits, qids, qlog = _chain_case(V, k, T, seed)
    pol = ov.Policy(temperature=T, top_k=0)
    prep = ov.prepare_rows(logits, [0] * k, ov.chain_parents(k), qids, qlog, [], pol)
    p_ref = [softmax(logits[r].astype(np.float64) / np.float64(np.float32(T))) for r in range(k + 1)]
    q_ref = []
    for i in range(k):
        w = softmax(qlog[i].astype(np.float64) / np.float64(np.float32(T)))
        q_ref.append(np.bincount(qids[i], weights=w, minlength=V))

    def breakpoints_for(drafts):
        def bp(key):
            row, purpose = key
            if purpose == PURPOSE_ACCEPT:
                x = drafts[row]
                return [p_ref[row][x] / q_ref[row][x]] if q_ref[row][x] > 0 else []
            pts = list(np.cumsum(np.sort(p_ref[row])[::-1]))
            pd = prep.pdists[row]
            order = [pd.ids[j] for j in range(pd.m)]
            pts += list(np.cumsum(p_ref[row][order]))
            if row < k:
                r = np.maximum(p_ref[row][order] - q_ref[row][order], 0.0)
                if r.sum() > 0:
                    pts += list(np.cumsum(r) / r.sum())
            return pts
        return bp

    first = np.zeros(V)
    reach = np.zeros(k + 1)
    at_depth = np.zeros((k + 1, V))
    for drafts in np.ndindex(*([V] * k)):
        pd = np.prod([q_ref[i][drafts[i]] for i in range(k)]) if k else 1.0
        if pd == 0.0:
            continue

        def run(uniforms, drafts=drafts):
            em, _ = ov.accept_rejection_chain(prep.pdists, prep.qdists, list(drafts), uniforms)
            return tuple(em)
        for em, w in _explore(run, breakpoints_for(drafts)).items():
            first[em[0]] += pd * w
            for d, t in enumerate(em):
                reach[d] += pd * w
                at_depth[d, t] += pd * w
    # exact up to the float32 rounding of the policy (a few 1e-7)
    assert abs(first.sum() - 1.0) < 1e-9
    np.testing.assert_allclose(first, p_ref[0], atol=2e-6)
    for d in range(1, k + 1):
        if reach[d] > 1e-3:
            np.testing.assert_allclose(at_depth[d] / reach[d], p_ref[d], atol=2e-5)


def test_naive_descent_is_exact_for_a_deterministic_tree():
    """Sampled token tree: the first token follows p of the root row and the
    token after a taken child follows that child's row."""
    rng = np.random.default_rng(20)
    V, T = 5, 0.9
    tokens, parent = [0, 1, 2, 3, 4, 1], [-1, -1, 0, 0, 1, 4]
    logits = rng.standard_normal((7, V)).astype(np.float32)
    pol = ov.Policy(temperature=T, top_k=0)
    prep = ov.prepare_rows(logits, tokens, parent, None, None, [], pol)
    p_ref = [softmax(logits[r].astype(np.float64) / np.float64(np.float32(T))) for r in range(7)]

    def bp(key):
        row, _ = key
        pd = prep.pdists[row]
        return list(np.cumsum(p_ref[row][pd.ids]))

    law = _explore(lambda u: tuple(ov.accept_naive_descent(prep.pdists, tokens, parent, u)[0]), bp)
    first = np.zeros(V)
    second_after_0 = np.zeros(V)
    for em, w in law.items():
        first[em[0]] += w
        if em[0] == 0 and len(em) > 1:
            second_after_0[em[1]] += w
    np.testing.assert_allclose(first, p_ref[0], atol=2e-6)
    # token 0 at the root is node 0 (the lowest index); its row is 1
    np.testing.assert_allclose(second_after_0 / second_after_0.sum(), p_ref[1], atol=2e-5)


def test_every_window_emits_at_least_one_token():
    rng = np.random.default_rng(30)
    for trial in range(300):
        V = int(rng.integers(2, 90))
        n = int(rng.integers(0, 6))
        chain = trial % 2 == 0
        parent = ov.chain_parents(n) if chain else [int(rng.integers(-1, j)) if j else -1 for j in range(n)]
        tokens = list(rng.integers(0, V, n))
        logits = (rng.standard_normal((n + 1, V)) * 2).astype(np.float32)
        pol = ov.Policy(temperature=float(rng.choice([0.0, 0.5, 1.0])), top_k=int(rng.integers(-1, 70)),
                        min_p=float(rng.uniform(0, 0.2)), top_p=float(rng.uniform(0.5, 1.0)),
                        presence=1.5, window=int(rng.integers(0, 10)))
        qids = rng.integers(0, V, (n, 8)) if chain else None
        qlog = rng.standard_normal((n, 8)).astype(np.float32) if chain else None
        res = ov.verify_window(logits, tokens, parent, qids, qlog, list(rng.integers(0, V, 12)),
                               pol, seed=trial, position=7)
        assert 1 <= res.n_emitted <= n + 1 and res.n_emitted == res.accept + 1
        assert all(0 <= t < V for t in res.emitted)


def test_invalid_trees_are_rejected():
    logits = np.zeros((3, 4), np.float32)
    with pytest.raises(ValueError):
        ov.verify_window(logits, [1, 2], [-1, 1])       # parent is not an earlier node
    with pytest.raises(ValueError):
        ov.verify_window(logits, [1, 9], [-1, 0])       # token outside the vocabulary


def _point_mass_breakpoints(prep, p_ref, drafts, k):
    """Jumps of the point-mass chain rule: u1 at p(x); u2 at the running sums
    of p and of p with the draft removed, both in pool order."""
    def bp(key):
        row, purpose = key
        pd = prep.pdists[row]
        order = [pd.ids[j] for j in range(pd.m)]
        if purpose == PURPOSE_ACCEPT:
            return [p_ref[row][drafts[row]]]
        pts = list(np.cumsum(p_ref[row][order]))
        if row < k:
            r = np.where(np.array(order) == drafts[row], 0.0, p_ref[row][order])
            if r.sum() > 0:
                pts += list(np.cumsum(r) / r.sum())
        return pts
    return bp


@pytest.mark.parametrize("V,k,T,seed", [(6, 2, 1.0, 40), (5, 3, 0.6, 41), (7, 2, 1.4, 42)])
def test_point_mass_drafts_are_exact_by_enumeration(V, k, T, seed):
    """Drafts proposed without probabilities ("Speculative decoding on RDNA"
    §06, n-gram takeovers): accept d_i with probability p_i(d_i), else draw
    from p_i without d_i.  Exact law over every uniform: the first token
    follows p_0 and, given the window reached depth j, the token there
    follows p_j."""
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    drafts = [int(np.argmax(logits[i])) if i % 2 == 0 else int(rng.integers(0, V)) for i in range(k)]
    pol = ov.Policy(temperature=T, top_k=0)
    prep = ov.prepare_rows(logits, drafts, ov.chain_parents(k), None, None, [], pol)
    p_ref = [softmax(logits[r].astype(np.float64) / np.float64(np.float32(T))) for r in range(k + 1)]
    q = [ov.point_mass(d) for d in drafts]

    def run(u):
        return tuple(ov.accept_rejection_chain(prep.pdists, q, drafts, u)[0])
    law = _explore(run, _point_mass_breakpoints(prep, p_ref, drafts, k))
    first = np.zeros(V)
    reach = np.zeros(k + 1)
    at_depth = np.zeros((k + 1, V))
    for em, w in law.items():
        first[em[0]] += w
        for d, t in enumerate(em):
            reach[d] += w
            at_depth[d, t] += w
    assert abs(first.sum() - 1.0) < 1e-9
    np.testing.assert_allclose(first, p_ref[0], atol=2e-6)
    # depth d is reached exactly when d_0..d_{d-1} were all accepted
    for d in range(1, k + 1):
        np.testing.assert_allclose(reach[d], np.prod([p_ref[i][drafts[i]] for i in range(d)]),
                                   atol=2e-6)
        if reach[d] > 1e-3:
            np.testing.assert_allclose(at_depth[d] / reach[d], p_ref[d], atol=2e-5)


def test_point_mass_chain_has_the_law_of_naive_descent():
    """For a fixed chain the point-mass rejection rule and naive sampling
    descent (exact when the draft is deterministic) emit every sequence with the
    same probability, though from different uniforms."""
    rng = np.random.default_rng(43)
    V, k, T = 5, 3, 0.8
    logits = (rng.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    drafts = [int(np.argmax(logits[0])), int(np.argsort(logits[1])[-2]), int(np.argmax(logits[2]))]
    pol = ov.Policy(temperature=T, top_k=0)
    parent = ov.chain_parents(k)
    prep = ov.prepare_rows(logits, drafts, parent, None, None, [], pol)
    p_ref = [softmax(logits[r].astype(np.float64) / np.float64(np.float32(T))) for r in range(k + 1)]
    q = [ov.point_mass(d) for d in drafts]
    bp = _point_mass_breakpoints(prep, p_ref, drafts, k)
    law_pm = _explore(lambda u: tuple(ov.accept_rejection_chain(prep.pdists, q, drafts, u)[0]), bp)
    law_nd = _explore(lambda u: tuple(ov.accept_naive_descent(prep.pdists, drafts, parent, u)[0]), bp)
    keys = set(law_pm) | set(law_nd)
    assert len(keys) > 10
    for s in keys:
        assert abs(law_pm.get(s, 0.0) - law_nd.get(s, 0.0)) < 2e-6, s


def test_point_mass_equals_candidates_with_one_finite_logit():
    """q given as 8 candidates of which only the draft has a finite logit is
    the point mass: same emitted tokens from the same uniforms, under
    truncating policies and penalties."""
    rng = np.random.default_rng(44)
    for trial in range(400):
        V = int(rng.integers(2, 60))
        k = int(rng.integers(1, 7))
        logits = (rng.standard_normal((k + 1, V)) * 2).astype(np.float32)
        drafts = [int(np.argmax(logits[i])) if rng.random() < 0.5 else int(rng.integers(0, V))
                  for i in range(k)]
        pol = ov.Policy(temperature=float(rng.choice([0.3, 0.7, 1.0, 1.5])),
                        top_k=int(rng.integers(-1, 70)), min_p=float(rng.choice([0.0, 0.05])),
                        top_p=float(rng.choice([1.0, 0.9])), repeat=1.1, presence=1.5,
                        frequency=0.2, window=int(rng.integers(0, 8)))
        hist = list(rng.integers(0, V, 10))
        qids = rng.integers(0, V, (k, 8))
        qids[:, 0] = drafts
        qlog = np.full((k, 8), -np.inf, np.float32)
        qlog[:, 0] = rng.standard_normal(k).astype(np.float32)
        a = ov.verify_window(logits, drafts, None, None, None, hist, pol, seed=trial, position=3)
        b = ov.verify_window(logits, drafts, None, qids, qlog, hist, pol, seed=trial, position=3)
        assert (a.emitted, a.accept) == (b.emitted, b.accept)


def test_point_mass_accepts_with_probability_p_and_never_redraws_the_draft():
    p = [_dist([0, 1, 2], [0.5, 0.3, 0.2]), _dist([0], [1.0])]
    q = [ov.point_mass(1)]
    S = float(p[0].total)
    # accepted iff u1 < p(1) = 0.3
    for u1, acc in ((0.2999, 1), (0.3001, 0)):
        _, a = ov.accept_rejection_chain(p, q, [1], lambda r, k: u1 if k == PURPOSE_ACCEPT else 0.5)
        assert a == acc
    # on rejection the replacement is never the draft
    for u2 in np.linspace(0.0, 0.999, 101):
        em, a = ov.accept_rejection_chain(p, q, [1], lambda r, k: 0.9 if k == PURPOSE_ACCEPT else u2)
        assert a == 0 and em[0] in (0, 2)
    # a draft outside the kept set is rejected and p is drawn unchanged
    em, a = ov.accept_rejection_chain(p, [ov.point_mass(7)], [7],
                                      lambda r, k: 0.0 if k == PURPOSE_ACCEPT else 0.95)
    assert a == 0 and em == [2] and S > 0
