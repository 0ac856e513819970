"""Pins for the oracle's batched form (CPU only): independent requests over
one stacked logits array, each with its own rows, policy, seed, position and
history (the batched serving workload of the verify step; the pages verify
one request at a time, and a batch is read as requests that do not
interact)."""
import numpy as np
import pytest

from oracle import verify as ov


def _logits_with_argmax(argmax, V, rng):
    x = rng.standard_normal((len(argmax), V)).astype(np.float32)
    for r, t in enumerate(argmax):
        x[r, t] = x[r].max() + 1.0
    return x


def _mixed_batch(seed):
    """Greedy chains with planted argmax paths, sampled chains with and
    without draft candidates, a penalised request and a sampled tree."""
    rng = np.random.default_rng(seed)
    V = 60
    blocks, reqs, want_accept = [], [], []
    for b, k in enumerate([3, 0, 5, 2, 4, 3]):
        am = [int(t) for t in rng.integers(0, V, k + 1)]
        blocks.append(_logits_with_argmax(am, V, rng))
        stop = int(rng.integers(0, k + 1))           # first draft that disagrees (k: none)
        drafts = am[:k]
        if stop < k:
            drafts[stop] = (am[stop] + 1 + int(rng.integers(0, V - 1))) % V
        reqs.append(dict(tokens=drafts, pol=ov.Policy(), seed=b, position=10 + b))
        want_accept.append(stop)
    for b in range(4):
        k = 3
        x = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
        blocks.append(x)
        req = dict(tokens=[int(t) for t in rng.integers(0, V, k)], seed=100 + b, position=7 * b,
                   pol=ov.Policy(temperature=0.8, top_k=0, min_p=0.02, top_p=0.95,
                                 presence=1.0 if b == 2 else 0.0, window=8 if b == 2 else 0),
                   hist=[int(t) for t in rng.integers(0, V, 12)])
        if b % 2:
            req["q_ids"] = rng.integers(0, V, (k, 8)).astype(np.int32)
            req["q_logits"] = rng.standard_normal((k, 8)).astype(np.float32)
        reqs.append(req)
        want_accept.append(None)
    blocks.append((rng.standard_normal((5, V)) * 1.5).astype(np.float32))
    reqs.append(dict(tokens=[int(t) for t in rng.integers(0, V, 4)], parent=[-1, 0, -1, 2],
                     pol=ov.Policy(temperature=0.7, top_k=20), seed=9, position=3))
    want_accept.append(None)
    return np.concatenate(blocks), reqs, want_accept


def test_greedy_requests_accept_their_own_argmax_prefix():
    # every greedy request walks its own rows: the planted argmax chain is
    # accepted up to the first disagreeing draft, whatever the other rows hold
    logits, reqs, want = _mixed_batch(0)
    out = ov.verify_batched(logits, reqs)
    for res, req, w in zip(out, reqs, want):
        if w is not None:
            assert res.accept == w and res.n_emitted == w + 1
            assert res.emitted[:w] == req["tokens"][:w]


def test_each_request_is_the_window_on_its_own_rows():
    logits, reqs, _ = _mixed_batch(1)
    out = ov.verify_batched(logits, reqs)
    r0 = 0
    for res, req in zip(out, reqs):
        r = len(req["tokens"]) + 1
        alone = ov.verify_window(logits[r0:r0 + r].copy(), req["tokens"], req.get("parent"),
                                 req.get("q_ids"), req.get("q_logits"), req.get("hist", ()),
                                 req["pol"], req["seed"], req["position"])
        assert res.emitted == alone.emitted and res.accept == alone.accept
        assert np.array_equal(res.pen_logits.view(np.uint32), alone.pen_logits.view(np.uint32))
        r0 += r


def test_requests_do_not_interact():
    # reversing the batch, and changing one request's seed, history and
    # rows, leaves every other request's result unchanged
    logits, reqs, _ = _mixed_batch(2)
    base = ov.verify_batched(logits, reqs)
    rows = [len(q["tokens"]) + 1 for q in reqs]
    starts = np.cumsum([0] + rows[:-1])
    order = list(range(len(reqs)))[::-1]
    rev_logits = np.concatenate([logits[starts[i]:starts[i] + rows[i]] for i in order])
    rev = ov.verify_batched(rev_logits, [reqs[i] for i in order])
    for j, i in enumerate(order):
        assert rev[j].emitted == base[i].emitted and rev[j].accept == base[i].accept
    victim = 7                                   # a sampled request
    changed = [dict(q) for q in reqs]
    changed[victim]["seed"] = 12345
    changed[victim]["hist"] = list(range(30))
    logits2 = logits.copy()
    logits2[starts[victim]:starts[victim] + rows[victim]] *= -1
    moved = ov.verify_batched(logits2, changed)
    for i in range(len(reqs)):
        if i != victim:
            assert moved[i].emitted == base[i].emitted and moved[i].accept == base[i].accept


def test_rows_must_cover_the_logits():
    logits, reqs, _ = _mixed_batch(3)
    with pytest.raises(ValueError):
        ov.verify_batched(logits[:-1], reqs)
    with pytest.raises(ValueError):
        ov.verify_batched(np.concatenate([logits, logits[:1]]), reqs)
