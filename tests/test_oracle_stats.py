"""The CPU statistical test that "Speculative decoding on RDNA" §03 describes
for its losslessness claim: 200,000 sampled windows per case, emitted tokens
checked against p by a chi-square; a control that samples the rejection
replacement from p, not from the residual, must fail that test in each
control case."""
import numpy as np
import pytest
from scipy import stats

from oracle import verify as ov
from oracle.philox import uniform_array, PURPOSE_DRAFT, PURPOSE_ACCEPT, PURPOSE_EMIT

TRIALS = 200_000
POSITION = 4096


def _case(name):
    rng = np.random.default_rng({"disjoint": 1, "policy": 2, "wide": 3}[name])
    if name == "disjoint":       # q favours tokens p dislikes: mostly residual draws
        V, k = 8, 2
        logits = np.tile(np.float32([3, 2.5, 2, 1, 0, -1, -1.5, -2]), (k + 1, 1))
        qids = np.tile(np.arange(8), (k, 1))
        qlog = np.tile(np.float32([-2, -1.5, -1, 0, 1, 2, 2.5, 3]), (k, 1))
        pol = ov.Policy(temperature=1.0, top_k=0)
        hist = []
    elif name == "policy":       # truncating policy and penalties on both p and q
        V, k = 40, 3
        logits = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
        qids = np.stack([rng.permutation(16)[:8] for _ in range(k)])
        qlog = (np.take_along_axis(logits[:k], qids, 1) + rng.standard_normal((k, 8))).astype(np.float32)
        pol = ov.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.9,
                        repeat=1.1, presence=1.5, frequency=0.2, window=6)
        hist = list(rng.integers(0, 16, 10))
    else:                        # wide vocabulary, top-k absent (20)
        V, k = 500, 2
        logits = (rng.standard_normal((k + 1, V)) * 2).astype(np.float32)
        order = np.argsort(-logits, axis=1)
        qids = np.stack([order[i, rng.permutation(24)[:8]] for i in range(k)])
        qlog = (rng.standard_normal((k, 8)) * 3).astype(np.float32)
        pol = ov.Policy(temperature=1.3)
        hist = []
    return logits, qids, qlog, pol, hist, k


def _simulate(name, replacement):
    logits, qids, qlog, pol, hist, k = _case(name)
    # drafts are placeholders for preparation; only q matters for drawing them
    prep = ov.prepare_rows(logits, [int(qids[i, 0]) for i in range(k)], ov.chain_parents(k),
                           qids, qlog, hist, pol)
    seeds = np.arange(TRIALS, dtype=np.uint64)
    u = {(r, pu): uniform_array(seeds, POSITION, r, pu)
         for r in range(k + 1) for pu in (PURPOSE_DRAFT, PURPOSE_ACCEPT, PURPOSE_EMIT)}
    first, second = [], []
    for t in range(TRIALS):
        drafts = []
        for i in range(k):
            q = prep.qdists[i]
            drafts.append(q.ids[ov.draw_index(q.e, q.total, u[(i, PURPOSE_DRAFT)][t])])
        em, _ = ov.accept_rejection_chain(prep.pdists, prep.qdists, drafts,
                                          lambda r, pu: u[(r, pu)][t], replacement)
        first.append(em[0])
        if len(em) > 1:
            second.append(em[1])
    return prep, np.array(first), np.array(second)


def _chi2_p(samples, dist):
    probs = {}
    for t, e in zip(dist.ids, dist.e):
        probs[t] = probs.get(t, 0.0) + float(e) / float(dist.total)
    ids = sorted(probs, key=lambda t: -probs[t])
    n = len(samples)
    if np.any(~np.isin(samples, ids)):
        return 0.0                                # a token outside p's support
    obs = np.array([np.sum(samples == t) for t in ids], dtype=np.float64)
    exp = np.array([probs[t] * n for t in ids])
    # merge categories whose expected count is below 5 into one
    small = exp < 5
    if small.any():
        obs = np.append(obs[~small], obs[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
    if len(obs) < 2:
        return 1.0
    return stats.chisquare(obs, exp * obs.sum() / exp.sum()).pvalue


@pytest.mark.parametrize("name", ["disjoint", "policy", "wide"])
def test_rejection_sampling_follows_p(name):
    prep, first, second = _simulate(name, "residual")
    assert _chi2_p(first, prep.pdists[0]) > 1e-4
    assert len(second) > 1000
    assert _chi2_p(second, prep.pdists[1]) > 1e-4


@pytest.mark.parametrize("name", ["disjoint", "policy", "wide"])
def test_replacement_from_p_control_fails(name):
    prep, first, second = _simulate(name, "p")
    assert _chi2_p(first, prep.pdists[0]) < 1e-9


def _simulate_point_mass(replacement):
    """Fixed drafts proposed without probabilities (an n-gram takeover,
    "Speculative decoding on RDNA" §06) through the rejection test with
    q = delta(draft)."""
    rng = np.random.default_rng(4)
    V, k = 30, 2
    logits = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.02, top_p=0.95)
    drafts = [int(np.argmax(logits[0])), int(np.argsort(logits[1])[-2])]
    prep = ov.prepare_rows(logits, drafts, ov.chain_parents(k), None, None, [], pol)
    q = [ov.point_mass(d) for d in drafts]
    seeds = np.arange(TRIALS, dtype=np.uint64)
    u = {(r, pu): uniform_array(seeds, POSITION, r, pu)
         for r in range(k + 1) for pu in (PURPOSE_ACCEPT, PURPOSE_EMIT)}
    first, second = [], []
    for t in range(TRIALS):
        em, _ = ov.accept_rejection_chain(prep.pdists, q, drafts, lambda r, pu: u[(r, pu)][t],
                                          replacement)
        first.append(em[0])
        if len(em) > 1:
            second.append(em[1])
    return prep, np.array(first), np.array(second)


def test_point_mass_rejection_follows_p():
    prep, first, second = _simulate_point_mass("residual")
    assert _chi2_p(first, prep.pdists[0]) > 1e-4
    assert len(second) > 1000
    assert _chi2_p(second, prep.pdists[1]) > 1e-4


def test_point_mass_replacement_from_p_control_fails():
    prep, first, _ = _simulate_point_mass("p")
    assert _chi2_p(first, prep.pdists[0]) < 1e-9
