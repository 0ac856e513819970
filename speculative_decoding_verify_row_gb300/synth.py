"""Seeded synthetic inputs for the verify step (shared by the tests, the
benchmark and the smoke check).

This module only draws random numbers and assembles arrays; it computes
nothing of the verify step itself.  Where a workload needs something derived
from the target's logits (its argmax chain, its top-32), the caller passes
it in.  All generators use numpy's PCG64 with explicit seeds.

Workloads (hidden H, vocab V, drafts k, rows k + 1):
  tiny greedy chain   H 256,  V 4096,   k 3, weights N(0, 0.02), acts N(0, 1)
  sampled chain       H 4096, V 151936, k 3   (a Qwen3-8B-shaped LM head)
  penalised chain     H 4096, V 151936, k 8, 4096-token Zipf(1.1) history
  token tree          H 4096, V 151936, 3 branches x depth 8 (24 nodes)
  batched serving     H 5120, V 151936, 64 requests x k 3 (256 rows)
"""
import numpy as np

WEIGHT_SEED = 1234
WEIGHT_STD = 0.02
ACT_SEED_OFFSET = 1_000_000
CHUNK_ROWS = 4096          # weights are drawn in independently seeded row chunks
PERM_SEED = 7


def f32_to_bf16_bits(x):
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.
    Finite inputs only (the generators never produce NaN or inf)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def _chunk_rng(seed, chunk):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, chunk])))


def weight_chunk(chunk, hidden, vocab, seed=WEIGHT_SEED):
    r0 = chunk * CHUNK_ROWS
    n = min(CHUNK_ROWS, vocab - r0)
    w = _chunk_rng(seed, chunk).standard_normal((n, hidden), dtype=np.float32)
    w *= np.float32(WEIGHT_STD)
    return f32_to_bf16_bits(w)


def weights(vocab, hidden, seed=WEIGHT_SEED):
    """bf16 LM-head weights [V, H] (uint16 bits), N(0, 0.02) rounded to bf16."""
    out = np.empty((vocab, hidden), dtype=np.uint16)
    for c in range((vocab + CHUNK_ROWS - 1) // CHUNK_ROWS):
        r0 = c * CHUNK_ROWS
        out[r0:r0 + CHUNK_ROWS] = weight_chunk(c, hidden, vocab, seed)
    return out


def weight_rows(vocab, hidden, rows, seed=WEIGHT_SEED):
    """The same weights, only the requested vocab rows (regenerates just the
    chunks that hold them)."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), hidden), dtype=np.uint16)
    for c in np.unique(rows // CHUNK_ROWS):
        sel = np.nonzero(rows // CHUNK_ROWS == c)[0]
        chunk = weight_chunk(int(c), hidden, vocab, seed)
        out[sel] = chunk[rows[sel] - c * CHUNK_ROWS]
    return out


def activations(rows, hidden, window_seed):
    """Row activations [R, H] float32 ~ N(0, 1); seed = window seed + 10^6."""
    rng = np.random.default_rng(window_seed + ACT_SEED_OFFSET)
    return rng.standard_normal((rows, hidden), dtype=np.float32)


def zipf_history(length, vocab, seed, s=1.1):
    """Prompt || emitted history: ranks drawn from Zipf(s) truncated to
    1..V, rank r mapped to token perm[r - 1] (a fixed permutation)."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** -s)
    cdf /= cdf[-1]
    u = np.random.default_rng(seed).random(length)
    r = np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1)
    perm = np.random.default_rng(PERM_SEED).permutation(vocab)
    return perm[r].astype(np.int32)


def draft_candidates(top32_ids, top32_vals, seed):
    """Draft head candidates for k draft rows: each row's 8 ids drawn without
    replacement from the target's top 32 (uniformly), each logit = the
    target's logit + N(0, 1).  top32_ids/vals: [k, 32] from the caller."""
    top32_ids = np.asarray(top32_ids)
    top32_vals = np.asarray(top32_vals, dtype=np.float32)
    k = top32_ids.shape[0]
    rng = np.random.default_rng(seed)
    q_ids = np.empty((k, 8), np.int32)
    q_log = np.empty((k, 8), np.float32)
    for i in range(k):
        pick = rng.choice(32, size=8, replace=False)
        q_ids[i] = top32_ids[i, pick]
        q_log[i] = top32_vals[i, pick] + rng.standard_normal(8).astype(np.float32)
    return q_ids, q_log


def draft_choice(q_logits, temperature, seed):
    """A stand-in draft model's choice among its 8 candidates: index drawn
    with weights exp(l / T) (numpy RNG), or the largest logit when T == 0.
    Returns slot indices [k]."""
    q_logits = np.asarray(q_logits, dtype=np.float64)
    if temperature == 0:
        return np.argmax(q_logits, axis=1)
    rng = np.random.default_rng(seed)
    z = q_logits / temperature
    z -= z.max(axis=1, keepdims=True)
    w = np.exp(z)
    w /= w.sum(axis=1, keepdims=True)
    return np.array([rng.choice(8, p=wi) for wi in w])


def tree_parents(branches=3, depth=8):
    """Parent array of `branches` chains of `depth` nodes hanging from the
    root; branch b's nodes are b*depth .. b*depth+depth-1."""
    parent = []
    for b in range(branches):
        for j in range(depth):
            parent.append(-1 if j == 0 else b * depth + j - 1)
    return np.array(parent, dtype=np.int32)


def tree_tokens(argmax_rows, top32_rows, seed, branches=3, depth=8, agree=5):
    """Node tokens of the tree workload: branch 0 follows the target argmax
    of its parent row for `agree` nodes and then takes a random token that
    differs from it; branches 1.. take random tokens from the parent row's
    top 32.  argmax_rows [R], top32_rows [R, 32] come from the caller."""
    rng = np.random.default_rng(seed)
    parent = tree_parents(branches, depth)
    tok = np.empty(len(parent), np.int32)
    for n, p in enumerate(parent):
        prow = 0 if p < 0 else 1 + p
        b, j = divmod(n, depth)
        if b == 0 and j < agree:
            tok[n] = argmax_rows[prow]
        elif b == 0:
            choices = [t for t in top32_rows[prow] if t != argmax_rows[prow]]
            tok[n] = choices[rng.integers(len(choices))]
        else:
            tok[n] = top32_rows[prow][rng.integers(32)]
    return tok


def perturb_draft(argmax_rows, k, pos, vocab, seed):
    """The target's own argmax chain d_i = argmax(row i), i < k, with d_pos
    replaced by a uniform token that differs from it."""
    d = np.array(argmax_rows[:k], dtype=np.int32)
    rng = np.random.default_rng(seed)
    t = int(rng.integers(vocab - 1))
    d[pos] = t if t < d[pos] else t + 1
    return d


def ngram_context(length, vocab, seed, match=5, plants=(2, 1, 1), cont_len=8):
    """A context for prompt lookup: a Zipf(1.1) token stream whose last
    `match` tokens also occur earlier, once per entry of `plants` groups;
    group g plants the key plants[g] times, each followed by the same
    cont_len random tokens (so group 0's continuation recurs most often).
    Returns int32 [length]."""
    rng = np.random.default_rng(seed)
    ctx = zipf_history(length, vocab, seed)
    key = ctx[length - match:].copy()
    conts = [rng.integers(0, vocab, cont_len).astype(np.int32) for _ in plants]
    span = match + cont_len
    slots = rng.permutation((length - match - span) // span)[:sum(plants)] * span
    i = 0
    for g, times in enumerate(plants):
        for _ in range(times):
            s = int(slots[i])
            ctx[s:s + match] = key
            ctx[s + match:s + span] = conts[g]
            i += 1
    return ctx
