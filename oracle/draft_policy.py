"""Oracle (test infrastructure only): the host-side draft proposal and window
pricing, written plainly from the pages.

  * ngram_propose -- prompt lookup over an n-gram index of the request's own
    context ("Speculative decoding on RDNA" §06, N-gram takeovers: match 5,
    propose 3); several matches become the branches of one token tree ("One
    RDNA4 verify pass has slack for about two dozen speculative tokens",
    "Spend the budget on a tree").
    Readings: matches are all earlier occurrences of the last `match`
    tokens; identical continuations are merged and ordered by how many
    occurrences propose them (the page ranks matches by recurrence), then
    by recency (plain prompt lookup uses the latest occurrence); branches
    sharing a prefix share its nodes.
  * cost_fit, expected_emitted, choose_depth -- §05 of the first page:
    window cost = one-row cost + a per-row increment (measured fits); the
    chosen depth maximises the expected number of emitted tokens (one, plus
    the sum over depths of the product of the acceptances up to that depth)
    divided by the window's cost, and k = 0 (a plain step) is kept unless
    some window is strictly better.
  * takeover -- §06: an n-gram window takes over when its tokens per unit
    of cost are at least the native window's.
  * ar_floor -- §07: keep speculating only if some probe window is strictly
    cheaper per emitted token than the timed plain step; equal cost, or a
    timing that is not a positive finite number, means retiring.
The CUDA library has its own implementation; nothing here is shared with it.
"""
import math
from collections import Counter

import numpy as np


def ngram_propose(context, match, propose, branches, max_nodes):
    """Returns (tokens, parent) lists describing the proposal tree."""
    ctx = [int(t) for t in context]
    n = len(ctx)
    if n <= match:
        return [], []
    key = ctx[n - match:]
    proposals = []                              # (start, continuation)
    for s in range(0, n - match):
        if ctx[s:s + match] == key:
            proposals.append((s, tuple(ctx[s + match:s + match + propose])))
    counts = Counter(c for _, c in proposals)
    latest = {}
    for s, c in proposals:
        latest[c] = max(latest.get(c, -1), s)
    ranked = sorted(counts, key=lambda c: (-counts[c], -latest[c]))
    tokens, parent = [], []
    for cont in ranked[:branches]:
        cur = -1
        for t in cont:
            child = None
            for j in range(len(tokens)):
                if parent[j] == cur and tokens[j] == t:
                    child = j
                    break
            if child is None:
                if len(tokens) == max_nodes:
                    break
                tokens.append(t)
                parent.append(cur)
                child = len(tokens) - 1
            cur = child
    return tokens, parent


def cost_fit(rows, ms):
    """Least squares ms = a + b (rows - 1): (a, b)."""
    x = np.asarray(rows, dtype=np.float64) - 1.0
    y = np.asarray(ms, dtype=np.float64)
    b, a = np.polyfit(x, y, 1)
    return float(a), float(b)


def expected_emitted(alpha, k):
    """E[emitted] of a k-draft window, from its definition: the window
    accepts exactly m drafts with probability alpha_1..alpha_m (1 -
    alpha_{m+1}) (no last factor for m = k) and then emits m + 1 tokens."""
    total = 0.0
    for m in range(k + 1):
        p = 1.0
        for i in range(m):
            p *= float(alpha[i])
        if m < k:
            p *= 1.0 - float(alpha[m])
        total += (m + 1) * p
    return total


def choose_depth(alpha, kmax, a, b):
    """(k, tokens per unit cost): the best k in [0, kmax], k = 0 unless a
    window is strictly better, the smaller k among equal rates."""
    rates = [expected_emitted(alpha, k) / (a + b * k) for k in range(kmax + 1)]
    best = 0
    for k in range(1, kmax + 1):
        if rates[k] > rates[best]:
            best = k
    return best, rates[best]


def takeover(alpha_native, k_native, alpha_ngram, k_ngram, a, b):
    native = expected_emitted(alpha_native, k_native) / (a + b * k_native)
    ngram = expected_emitted(alpha_ngram, k_ngram) / (a + b * k_ngram)
    return ngram >= native


def ar_floor(ar_ms, window_ms, emitted):
    """True to keep speculating, False to retire to plain steps."""
    if not math.isfinite(ar_ms) or ar_ms <= 0.0:
        return False
    for ms, e in zip(window_ms, emitted):
        if not math.isfinite(ms) or ms <= 0.0 or e < 1:
            return False
    return any(ms / e < ar_ms for ms, e in zip(window_ms, emitted))
