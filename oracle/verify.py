"""The verify step, restated plainly on the CPU.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Nothing here is blocked,
fused or reordered beyond what the definitions below state; sequential sums
are Python loops in pool order.

Notation: V vocab, H hidden, R verify rows, k drafts, P = 64 pool width,
C = 8 draft candidates, W penalty window.

Rows and nodes.  A window verifies n draft nodes.  A chain of k drafts is the
tree whose node i has parent i-1 (node 0 hangs from the root).  Row 0 scores
the root (the current position); row 1+j scores the position after node j.
Node j is therefore checked against row(parent(j)), with row(-1) = 0
("Speculative decoding on RDNA" §01 figure: k drafts, k+1 verify rows; token
trees: "One RDNA4 verify pass has slack ...", "Spend the budget on a tree").
"""
from dataclasses import dataclass, field
import math

import numpy as np

from .philox import uniform as philox_uniform, PURPOSE_ACCEPT, PURPOSE_EMIT
from .vexp import vexp, Z_MIN

POOL = 64          # the 64-wide candidate pool ("Speculative decoding on RDNA" §03)
QCAND = 8          # candidates per draft node, re-scored by the draft head (same section)
TOPK_ABSENT = 20   # top-k when the request gives none (same section)


# ---------------------------------------------------------------------------
# policy record

def _f32(x):
    return float(np.float32(x))


@dataclass
class Policy:
    """Per-request sampler and penalty settings.  Float fields hold float32
    values, as the C struct does."""
    temperature: float = 0.0     # 0 => greedy
    top_k: int = -1              # <0 absent (=> 20); 0 => all 64 pool entries
    min_p: float = 0.0           # <=0 disables
    top_p: float = 1.0           # >=1 disables
    repeat: float = 1.0          # 1 disables
    presence: float = 0.0        # 0 disables
    frequency: float = 0.0       # 0 disables
    window: int = 0              # W; 0 disables every penalty

    def __post_init__(self):
        for name in ("temperature", "min_p", "top_p", "repeat", "presence", "frequency"):
            setattr(self, name, _f32(getattr(self, name)))
        self.top_k = int(self.top_k)
        self.window = int(self.window)

    @property
    def greedy(self):
        return self.temperature == 0.0


# ---------------------------------------------------------------------------
# (a1) projection -- "Speculative decoding on RDNA" §01 (one pass scores all
# k+1 rows against one read of the weights) and §02 (bf16-weight x
# fp32-activation verify projection).  bf16 -> f64 and f32 -> f64 are exact,
# and each product of a bf16 and an f32 is exact in f64, so this is the exact
# logit up to the rounding of one f64 dot product.

def bf16_bits_to_f32(bits):
    """bf16 bit patterns (uint16) -> float32, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def project(weight_bits, act):
    """logits[r, v] = sum_h W[v, h] * A[r, h], in f64.  W: [V, H] bf16 bits,
    A: [R, H] float32.  Returns [R, V] float64."""
    w = bf16_bits_to_f32(weight_bits).astype(np.float64)
    a = np.asarray(act, dtype=np.float32).astype(np.float64)
    return a @ w.T


def project_columns(weight_bits, act, vocab_ids):
    """The same definition for a chosen subset of vocab rows: [R, len(ids)]."""
    w = bf16_bits_to_f32(np.asarray(weight_bits)[np.asarray(vocab_ids)]).astype(np.float64)
    a = np.asarray(act, dtype=np.float32).astype(np.float64)
    return a @ w.T


# ---------------------------------------------------------------------------
# tree bookkeeping

def chain_parents(k):
    """Parent array of a k-draft chain: node i hangs from node i-1."""
    return [i - 1 for i in range(k)]


def row_of(node):
    return 0 if node < 0 else 1 + node


def validate_tree(tokens, parent, vocab):
    n = len(tokens)
    if len(parent) != n:
        raise ValueError("parent array length differs from the node count")
    for j in range(n):
        if not (-1 <= parent[j] < j):
            raise ValueError(f"node {j}: parent {parent[j]} is not -1 or an earlier node")
        if not (0 <= tokens[j] < vocab):
            raise ValueError(f"node {j}: token {tokens[j]} outside the vocabulary")


def path_tokens(tokens, parent, node):
    """Tokens on the path root -> node, node included, in root-first order."""
    out = []
    while node >= 0:
        out.append(int(tokens[node]))
        node = parent[node]
    out.reverse()
    return out


# ---------------------------------------------------------------------------
# (a2) penalty histories -- "Speculative decoding on RDNA" §04 and its figure:
# row i is penalised against H_i, the W most recent tokens of the prompt, the
# tokens emitted so far and drafts 0..i-1.  For a tree the same rule is read along the node's
# ancestor path (each branch sees only its own ancestors, as in the masked
# tree pass of "One RDNA4 verify pass ...").  Fewer than W tokens: use all.

def row_histories(hist, tokens, parent, window):
    """H for every row: row 0 -> last W of hist; row 1+j -> last W of
    (hist || path tokens root -> node j)."""
    hist = [int(t) for t in hist]
    rows = len(tokens) + 1
    out = []
    for r in range(rows):
        seq = hist + ([] if r == 0 else path_tokens(tokens, parent, r - 1))
        out.append(seq[max(0, len(seq) - window):] if window > 0 else [])
    return out


# ---------------------------------------------------------------------------
# (a2) penalties -- "Speculative decoding on RDNA" §04 names repeat, presence
# and frequency penalties and says both p and q are penalised by the same
# H_i; it gives no formula.  Reading: the CTRL repetition penalty followed by
# the OpenAI presence/frequency form, each step one float32 operation rounded
# to nearest, applied once per distinct token t of H_i with count c:
#     x = l[t]
#     x = x / repeat   if x > 0 else x * repeat        (skipped if repeat == 1)
#     x = x - float32(c) * frequency                    (skipped if frequency == 0)
#     x = x - presence                                  (skipped if presence == 0)

def penalties_active(pol):
    return pol.window > 0 and (pol.repeat != 1.0 or pol.presence != 0.0 or pol.frequency != 0.0)


def penalize_value(x, count, pol):
    x = np.float32(x)
    if pol.repeat != 1.0:
        rep = np.float32(pol.repeat)
        x = np.float32(x / rep) if x > 0 else np.float32(x * rep)
    if pol.frequency != 0.0:
        x = np.float32(x - np.float32(np.float32(count) * np.float32(pol.frequency)))
    if pol.presence != 0.0:
        x = np.float32(x - np.float32(pol.presence))
    return x


def history_counts(H):
    counts = {}
    for t in H:
        counts[t] = counts.get(t, 0) + 1
    return counts


def penalize_row(row, H, pol):
    """Penalised copy of one target row (float32 [V]).  History tokens
    outside [0, V) have no logit and are ignored."""
    out = np.array(row, dtype=np.float32, copy=True)
    if not penalties_active(pol):
        return out
    with np.errstate(all="ignore"):
        for t, c in history_counts(H).items():
            if 0 <= t < out.shape[0]:
                out[t] = penalize_value(out[t], c, pol)
    return out


def penalize_candidates(ids, vals, H, pol):
    """Penalised copy of a draft row's candidate logits (float32 [C])."""
    out = np.array(vals, dtype=np.float32, copy=True)
    if not penalties_active(pol):
        return out
    counts = history_counts(H)
    with np.errstate(all="ignore"):
        for j, t in enumerate(ids):
            c = counts.get(int(t), 0)
            if c:
                out[j] = penalize_value(out[j], c, pol)
    return out


# ---------------------------------------------------------------------------
# (a3) pool -- "Speculative decoding on RDNA" §03: the sampler works on a
# pool of 64 entries whose ties are broken in one fixed way.  Reading: order by value descending under the total order of
# float32 that puts every NaN below -inf and -0.0 below +0.0, equal values by
# ascending token id ("feat(dflash) ...": the top-K selector is held to byte
# identity with ties, NaN and -inf).  The order is computed on the usual
# order-preserving map of float bits.

def order_keys(vals):
    """uint32 keys whose unsigned order is the value order above (NaN -> 0)."""
    v = np.asarray(vals, dtype=np.float32)
    bits = v.view(np.uint32)
    neg = (bits >> np.uint32(31)).astype(bool)
    keys = np.where(neg, ~bits, bits | np.uint32(0x80000000)).astype(np.uint32)
    keys[np.isnan(v)] = 0
    return keys


def top_k_entries(row, k):
    """The first min(k, V) entries of a row in pool order: (ids int64,
    values float32).  With k = 16 this is the batched top-K of "feat(dflash):
    developer-only online draft tuning" (ties, NaN and -inf under one fixed
    order)."""
    row = np.asarray(row, dtype=np.float32)
    keys = order_keys(row).astype(np.int64)
    ids = np.arange(row.shape[0], dtype=np.int64)
    order = np.lexsort((ids, -keys))[:min(k, row.shape[0])]
    return order, row[order]


def target_pool(row):
    """Top-min(64, V) of a row: (ids int64, values float32) in pool order."""
    return top_k_entries(row, POOL)


def candidate_pool(cand_ids, cand_vals):
    """The draft's C candidates in pool order (value desc, id asc, slot asc)."""
    cand_ids = np.asarray(cand_ids, dtype=np.int64)
    cand_vals = np.asarray(cand_vals, dtype=np.float32)
    keys = order_keys(cand_vals).astype(np.int64)
    order = np.lexsort((np.arange(len(cand_ids)), cand_ids, -keys))
    return cand_ids[order], cand_vals[order]


# ---------------------------------------------------------------------------
# (a4) policy -- "Speculative decoding on RDNA" §03 ("how hipfire does it"):
# temperature, top-k (20 when absent, all 64 pool entries when 0), min-p and
# top-p, on the AR sampler's pool, tie-breaking and summation.  Reading of
# the order and arithmetic (the pages fix neither): every step is one
# float32 operation rounded to nearest, sums run sequentially in pool order,
#   K = 20 if top_k absent, 64 if 0, else min(top_k, 64); K <= pool size
#   T == 0: greedy, p = point mass on pool[0]
#   e_0 = 1; e_j = vexp((v_j - v_0) / T) for j < K (0 if v_j is NaN or -inf,
#        or the exponent is below -87 or NaN)
#   min-p: cut the prefix at the first j >= 1 with e_j < min_p (e_j/e_0 is
#          p_j/p_max, so this keeps p_j >= min_p * p_max)
#   top-p: with S the sum of the survivors, keep the shortest prefix whose
#          running sum reaches top_p * S
#   S = sum of the kept e; p_j = e_j / S

F32 = np.float32


@dataclass
class RowDist:
    """A policy applied to one pool: the kept ids and unnormalised weights
    (float32)."""
    ids: list
    e: list
    total: np.float32

    @property
    def m(self):
        return len(self.ids)


def topk_limit(top_k):
    if top_k < 0:
        return TOPK_ABSENT
    if top_k == 0:
        return POOL
    return min(top_k, POOL)


def seq_sum(xs):
    s = F32(0.0)
    for x in xs:
        s = F32(s + F32(x))
    return s


def policy_weights(pool_vals, pol):
    """(m, e[:m], S) for one pool (values in pool order), all float32."""
    n = len(pool_vals)
    if n == 0:
        raise ValueError("empty pool")
    K = min(topk_limit(pol.top_k), n)
    if pol.greedy:
        return 1, [F32(1.0)], F32(1.0)
    T = F32(pol.temperature)
    v0 = F32(pool_vals[0])
    e = [F32(1.0)]
    with np.errstate(all="ignore"):
        for j in range(1, K):
            v = F32(pool_vals[j])
            if np.isnan(v) or v == -np.inf:
                e.append(F32(0.0))
                continue
            z = F32(F32(v - v0) / T)
            e.append(vexp(z) if z >= Z_MIN else F32(0.0))
        m = K
        if pol.min_p > 0.0:
            mp = F32(pol.min_p)
            j = 1
            while j < m and e[j] >= mp:
                j += 1
            m = j
        if pol.top_p < 1.0:
            thr = F32(F32(pol.top_p) * seq_sum(e[:m]))
            c = F32(0.0)
            for j in range(m):
                c = F32(c + e[j])
                if c >= thr:
                    m = j + 1
                    break
    e = e[:m]
    return m, e, seq_sum(e)


def row_dist(pool_ids, pool_vals, pol):
    m, e, S = policy_weights(pool_vals, pol)
    return RowDist([int(t) for t in pool_ids[:m]], e, S)


def prob_of(dist, x):
    """p(x) = e_j / S for the kept entry holding x (summed over repeats)."""
    acc = F32(0.0)
    for t, ej in zip(dist.ids, dist.e):
        if t == x:
            acc = F32(acc + F32(ej / dist.total))
    return acc


# ---------------------------------------------------------------------------
# draws -- one uniform u, t = u * S, the first j whose running sum exceeds t.
# Reading for the rounding corner where no running sum exceeds t: the last
# entry with a positive weight.

def draw_index(weights, total, u):
    t = F32(F32(u) * F32(total))
    c = F32(0.0)
    for j, w in enumerate(weights):
        c = F32(c + F32(w))
        if c > t:
            return j
    for j in range(len(weights) - 1, -1, -1):
        if weights[j] > 0.0:
            return j
    return 0


# ---------------------------------------------------------------------------
# (a5) acceptance

def accept_greedy(argmax, tokens, parent):
    """Greedy verify.  Chain: the longest prefix of drafts equal to the
    target's argmax, then the argmax at the first mismatch or the bonus after
    the last row ("Speculative decoding on RDNA" §02 and the §01 figure).
    Tree: the longest branch every node of which equals the argmax of its
    parent's row ("One RDNA4 verify pass ...", "Spend the budget on a tree");
    reading: equal depths go to the smaller node index, no agreeing node
    means the root.  Returns (emitted ids, accepted count)."""
    n = len(tokens)
    ok = [False] * n
    depth = [0] * n
    best, best_depth = -1, 0
    for j in range(n):
        p = parent[j]
        ok[j] = int(tokens[j]) == argmax[row_of(p)] and (p < 0 or ok[p])
        depth[j] = 1 if p < 0 else depth[p] + 1
        if ok[j] and depth[j] > best_depth:
            best, best_depth = j, depth[j]
    emitted = path_tokens(tokens, parent, best) + [argmax[row_of(best)]]
    return emitted, best_depth


def accept_rejection_chain(pdists, qdists, drafts, uniforms, replacement="residual"):
    """Speculative rejection sampling ("Speculative decoding on RDNA" §03,
    steps 1-4; Leviathan et al.; Chen et al.):
      for each draft x = d_i: accept with probability min(1, p_i(x)/q_i(x)),
      tested as u1 * q(x) < p(x) (reading: q(x) = 0 accepts iff p(x) > 0);
      a rejected draft is replaced by a sample of (p_i - q_i)+ renormalised
      (reading: of p_i when that residual is all zero), which ends the window;
      k accepted drafts are followed by a bonus token sampled from p_k.
    uniforms(row, purpose) gives the window's uniforms.  replacement="p" is
    the deliberately wrong control of the same section's CPU test, which
    samples the replacement from p rather than from the residual)."""
    emitted = []
    for i, x in enumerate(drafts):
        x = int(x)
        p, q = pdists[i], qdists[i]
        px, qx = prob_of(p, x), prob_of(q, x)
        u1 = F32(uniforms(i, PURPOSE_ACCEPT))
        accepted = (F32(u1 * qx) < px) if qx > 0.0 else (px > 0.0)
        if accepted:
            emitted.append(x)
            continue
        u2 = uniforms(i, PURPOSE_EMIT)
        if replacement == "p":
            j = draw_index(p.e, p.total, u2)
            emitted.append(p.ids[j])
            return emitted, i
        resid = []
        for t, ej in zip(p.ids, p.e):
            d = F32(F32(ej / p.total) - prob_of(q, t))
            resid.append(d if d > 0.0 else F32(0.0))
        sr = seq_sum(resid)
        j = draw_index(resid, sr, u2) if sr > 0.0 else draw_index(p.e, p.total, u2)
        emitted.append(p.ids[j])
        return emitted, i
    k = len(drafts)
    p = pdists[k]
    j = draw_index(p.e, p.total, uniforms(k, PURPOSE_EMIT))
    emitted.append(p.ids[j])
    return emitted, k


def point_mass(token):
    """q = delta(token): the draft distribution of a candidate proposed
    without probabilities (an n-gram match).  Fed to the chain rejection test
    it accepts the token with probability p(token) and, on rejection, draws
    from p with the token removed ("Speculative decoding on RDNA" §06, N-gram
    takeovers: a sampled n-gram candidate is verified by the §03 rejection
    test with all of q's mass on that candidate)."""
    return RowDist([int(token)], [F32(1.0)], F32(1.0))


def accept_naive_descent(pdists, tokens, parent, uniforms):
    """Naive sampling verify, exact when the draft is deterministic ("feat(dflash)
    ...", notes under the spec-step listing): from the root, draw y from the
    current row's p; if a child of the current node carries y (reading: the
    lowest-index such child), move there and repeat; otherwise emit y and
    stop.  At a leaf the draw is the bonus token.  Used for sampled token
    trees."""
    children = {}
    for j, p in enumerate(parent):
        children.setdefault(int(p), []).append(j)
    emitted = []
    cur = -1
    while True:
        r = row_of(cur)
        d = pdists[r]
        y = d.ids[draw_index(d.e, d.total, uniforms(r, PURPOSE_EMIT))]
        emitted.append(y)
        nxt = None
        for c in children.get(cur, []):
            if int(tokens[c]) == y:
                nxt = c
                break
        if nxt is None:
            return emitted, len(emitted) - 1
        cur = nxt


# ---------------------------------------------------------------------------
# the window

@dataclass
class WindowResult:
    pen_logits: np.ndarray          # [R, V] float32 (penalised target rows)
    pool_ids: list                  # per row, int64 [min(64, V)]
    pool_vals: list                 # per row, float32
    pdists: list                    # per row RowDist
    qdists: list                    # per node RowDist (chain rejection only;
                                    # point masses when no candidates were given)
    q_pen: np.ndarray = None        # [n, C] penalised draft logits
    emitted: list = field(default_factory=list)
    accept: int = 0

    @property
    def n_emitted(self):
        return len(self.emitted)


def prepare_rows(logits, tokens, parent, q_ids, q_logits, hist, pol):
    """Penalise, pool and apply the policy to every row (and to q)."""
    logits = np.asarray(logits, dtype=np.float32)
    R, V = logits.shape
    n = len(tokens)
    if R != n + 1:
        raise ValueError("rows must equal nodes + 1")
    validate_tree(tokens, parent, V)
    H = row_histories(hist, tokens, parent, pol.window)
    pen = np.stack([penalize_row(logits[r], H[r], pol) for r in range(R)])
    pools = [target_pool(pen[r]) for r in range(R)]
    pdists = [row_dist(ids, vals, pol) for ids, vals in pools]
    qdists, q_pen = [], None
    if q_ids is not None:
        q_ids = np.asarray(q_ids, dtype=np.int64).reshape(n, QCAND)
        q_logits = np.asarray(q_logits, dtype=np.float32).reshape(n, QCAND)
        if n and (q_ids.min() < 0 or q_ids.max() >= V):
            raise ValueError("draft candidate id outside the vocabulary")
        q_pen = np.stack([penalize_candidates(q_ids[j], q_logits[j], H[row_of(parent[j])], pol)
                          for j in range(n)]) if n else np.zeros((0, QCAND), np.float32)
        for j in range(n):
            cid, cval = candidate_pool(q_ids[j], q_pen[j])
            qdists.append(row_dist(cid, cval, pol))
    return WindowResult(pen, [p[0] for p in pools], [p[1] for p in pools], pdists, qdists, q_pen)


def is_chain(parent):
    return all(p == j - 1 for j, p in enumerate(parent))


def verify_window(logits, tokens, parent=None, q_ids=None, q_logits=None, hist=(),
                  pol=None, seed=0, position=0, uniforms=None, replacement="residual"):
    """One speculative window on given target logits [R, V] (float32).

    tokens: draft tokens (chain) or node tokens (tree); parent None = chain.
    Greedy requests: accept_greedy.  Sampled chains: rejection sampling,
    against the draft candidates' q when given, else against the point mass
    on each draft (n-gram takeover).  Sampled trees: naive sampling descent.
    Every window emits at least one token ("Speculative decoding on RDNA"
    §01)."""
    pol = pol or Policy()
    tokens = [int(t) for t in tokens]
    parent = chain_parents(len(tokens)) if parent is None else [int(p) for p in parent]
    res = prepare_rows(logits, tokens, parent, q_ids, q_logits, hist, pol)
    if uniforms is None:
        def uniforms(row, purpose):
            return philox_uniform(seed, position, row, purpose)
    if pol.greedy:
        argmax = [int(ids[0]) for ids in res.pool_ids]
        res.emitted, res.accept = accept_greedy(argmax, tokens, parent)
    elif is_chain(parent):
        if q_ids is None:
            res.qdists = [point_mass(t) for t in tokens]
        res.emitted, res.accept = accept_rejection_chain(res.pdists, res.qdists, tokens,
                                                         uniforms, replacement)
    else:
        res.emitted, res.accept = accept_naive_descent(res.pdists, tokens, parent, uniforms)
    return res


def run_windows(logits_fn, windows, hist, pol, seed, position):
    """Multi-window driver: after each window the emitted ids (never the
    rejected drafts) are appended to the history and the position advances by
    the number emitted ("Speculative decoding on RDNA" §04 and its figure:
    the next window's history holds only emitted tokens, never a rejected
    draft).
    logits_fn(w, hist) -> logits of window w; windows[w] = dict of tokens,
    parent, q_ids, q_logits.  Returns the list of WindowResult and the final
    history."""
    hist = list(hist)
    out = []
    for w, win in enumerate(windows):
        res = verify_window(logits_fn(w, hist), win["tokens"], win.get("parent"),
                            win.get("q_ids"), win.get("q_logits"), hist, pol, seed, position)
        out.append(res)
        hist += res.emitted
        position += res.n_emitted
    return out, hist


def verify_batched(logits, requests):
    """Independent requests over one stacked logits array [sum R_b, V]: each
    request b has its own rows, policy, seed, position and history.
    requests[b] = dict(tokens, parent, q_ids, q_logits, hist, pol, seed,
    position)."""
    out, row0 = [], 0
    for req in requests:
        r = len(req["tokens"]) + 1
        out.append(verify_window(logits[row0:row0 + r], req["tokens"], req.get("parent"),
                                 req.get("q_ids"), req.get("q_logits"), req.get("hist", ()),
                                 req["pol"], req.get("seed", 0), req.get("position", 0)))
        row0 += r
    if row0 != len(logits):
        raise ValueError("request rows do not cover the logits")
    return out
