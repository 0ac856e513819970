"""Pins for the oracle's projection, histories and penalties (CPU only)."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import verify as ov


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint16)
    ours = ov.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_projection_is_the_exact_dot_product():
    """logits[r, v] = sum_h W[v, h] A[r, h]: checked against exact rational
    arithmetic on a non-square case (a transposed operand cannot pass)."""
    rng = np.random.default_rng(3)
    V, H, R = 7, 5, 3
    w = rng.standard_normal((V, H)).astype(np.float32)
    wbits = (w.view(np.uint32) >> 16).astype(np.uint16)            # truncated to bf16
    a = rng.standard_normal((R, H)).astype(np.float32)
    got = ov.project(wbits, a)
    assert got.shape == (R, V)
    wf = ov.bf16_bits_to_f32(wbits)
    for r in range(R):
        for v in range(V):
            exact = sum(Fraction(float(wf[v, h])) * Fraction(float(a[r, h])) for h in range(H))
            assert abs(Fraction(got[r, v]) - exact) <= abs(exact) * Fraction(1, 2**50) + Fraction(1, 2**80)
    cols = ov.project_columns(wbits, a, [6, 2])
    assert np.array_equal(cols, got[:, [6, 2]])


def test_histories_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "fig04_histories.json")))
    k = len(g["drafts"])
    for case in g["cases"]:
        H = ov.row_histories(g["hist"], g["drafts"], ov.chain_parents(k), case["W"])
        assert H == case["expected"]


def test_tree_histories_follow_ancestors():
    # two branches from the root: nodes 0->1 and 2->3
    tokens, parent = [5, 6, 7, 8], [-1, 0, -1, 2]
    H = ov.row_histories([1, 2], tokens, parent, 3)
    assert H == [[1, 2], [1, 2, 5], [2, 5, 6], [1, 2, 7], [2, 7, 8]]


def _pol(**kw):
    base = dict(temperature=0.7, window=8)
    base.update(kw)
    return ov.Policy(**base)


SPECIAL = np.array([3.5, -2.25, 0.0, -0.0, np.inf, -np.inf, np.nan, 1e-30, -7.0, 0.5,
                    2.0, -0.5, 100.0, -100.0, 1.0, -1.0], dtype=np.float32)


def test_neutral_policy_is_identity():
    for pol in (ov.Policy(temperature=1.0, window=0, repeat=1.3, presence=2.0),
                ov.Policy(temperature=1.0, window=16)):
        out = ov.penalize_row(SPECIAL, [0, 1, 2, 3, 4, 5, 6, 6], pol)
        assert np.array_equal(out.view(np.uint32), SPECIAL.view(np.uint32))


def test_only_history_tokens_change_and_all_decrease():
    rng = np.random.default_rng(4)
    row = rng.standard_normal(64).astype(np.float32) * 3
    H = [3, 9, 9, 40, 3, 3, 63]
    pol = _pol(repeat=1.3, presence=0.4, frequency=0.25)
    out = ov.penalize_row(row, H, pol)
    touched = sorted(set(H))
    for t in range(64):
        if t in touched:
            assert out[t] < row[t]
        else:
            assert out[t].view(np.uint32) == row[t].view(np.uint32)


def test_penalty_components():
    """Each component on its own, checked against its defining property."""
    row = np.array([2.0, -2.0, 0.0, 5.0], dtype=np.float32)
    H = [0, 1, 2, 3, 3, 3]
    # presence: one fixed amount per distinct token, whatever its count
    out = ov.penalize_row(row, H, _pol(presence=1.5))
    assert np.array_equal(row - out, np.float32([1.5, 1.5, 1.5, 1.5]))
    # frequency: proportional to the count
    out = ov.penalize_row(row, H, _pol(frequency=0.5))
    assert np.array_equal(row - out, np.float32([0.5, 0.5, 0.5, 1.5]))
    # repeat: positive logits shrink toward 0, negative ones move away from 0
    out = ov.penalize_row(row, H, _pol(repeat=2.0))
    assert np.array_equal(out, np.float32([1.0, -4.0, 0.0, 2.5]))


def test_penalty_is_permutation_invariant_and_windowed():
    rng = np.random.default_rng(5)
    row = rng.standard_normal(32).astype(np.float32)
    H = list(rng.integers(0, 32, 20))
    pol = _pol(repeat=1.1, presence=1.5, frequency=0.2, window=20)
    a = ov.penalize_row(row, H, pol)
    b = ov.penalize_row(row, list(reversed(H)), pol)
    assert np.array_equal(a, b)
    # tokens further back than W do not count
    hist = [31] * 50 + H
    Hw = ov.row_histories(hist, [], [], 20)[0]
    assert Hw == [int(t) for t in H]


def test_history_tokens_outside_vocab_are_ignored():
    row = np.float32([1.0, 2.0])
    out = ov.penalize_row(row, [5, -1, 1], _pol(presence=1.0))
    assert np.array_equal(out, np.float32([1.0, 1.0]))


def test_draft_candidates_use_the_same_history():
    row = np.float32([4.0, 3.0, 2.0, 1.0])
    H = [1, 1, 3]
    pol = _pol(repeat=1.1, presence=1.5, frequency=0.2)
    full = ov.penalize_row(row, H, pol)
    ids = [3, 1, 0]
    cand = ov.penalize_candidates(ids, row[ids], H, pol)
    assert np.array_equal(cand, full[ids])


def test_rejected_drafts_never_enter_the_next_history():
    """Two windows; the first rejects its second and third drafts.  The next
    window's histories contain the emitted ids only."""
    V = 16
    logits0 = np.zeros((4, V), np.float32)
    for r, t in enumerate([3, 4, 5, 6]):
        logits0[r, t] = 5.0
    seen = []

    def logits_fn(w, hist):
        seen.append(list(hist))
        return logits0

    windows = [dict(tokens=[3, 9, 10]), dict(tokens=[6, 7, 8])]
    res, hist = ov.run_windows(logits_fn, windows, [1, 2], ov.Policy(window=8, presence=1.0), 0, 2)
    assert res[0].emitted == [3, 4] and res[0].accept == 1
    assert seen[1] == [1, 2, 3, 4]
    assert 9 not in seen[1] and 10 not in seen[1]
    assert hist == [1, 2, 3, 4] + res[1].emitted
