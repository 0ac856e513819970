"""The statistical test of "Speculative decoding on RDNA" §03 run on the GPU:
200,000 sampled windows per case through the library's own sampler, the
emitted tokens checked against the target distribution p by a chi-square.

Each window is one request of a batched call (vr_verify_window_batched,
called through the C ABI with a request table built in numpy), with its own
seed 0..199,999 and drafts drawn from the draft distribution q that the
verifier itself uses.  One-hot activations make the projection return chosen
bf16 logits exactly (logits[r][v] = W[v][r]), so the expected distributions
come from the oracle's policy on exactly the GPU's logits.

Speculative sampling is lossless: the token emitted at depth j, given the
tokens emitted before it, follows p_j of the row reached by that prefix.
With penalties p_j and q_j depend on the earlier drafts (H_j holds them), so
depth j is tested per prefix, and the per-prefix chi-square statistics are
summed (their degrees of freedom too) into one p-value per depth.  The
deliberately wrong control (the replacement drawn from p, not from the
residual) stays on the CPU (test_oracle_stats.py), where it fails.

Cases: the oracle test's three (disjoint q, truncating policy with
penalties, wide vocabulary with top-k absent), drafts proposed without
probabilities (q = a point mass on each draft, §06), and a sampled token
tree (naive descent, "feat(dflash) ..." notes under the spec-step listing)
with penalty histories along each node's path.  Paths: the tensor-core
projection, whose windows sample in the row kernel, and the CUDA-core
projection, whose windows run the penalty kernel and the segment sampler."""
import ctypes

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import verify as ov
from speculative_decoding_verify_row_gb300 import binding as vb, synth
from gpu_common import require_gpu, dev, dev_weight
from test_oracle_stats import _case as cpu_case

pytestmark = pytest.mark.gpu

TRIALS = 200_000
POSITION = 4096
HIDDEN = 64
P_MIN = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _bf16_round(x):
    return ov.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(x, np.float32)))


def _case(name):
    """(logits [R, V] float32 bf16-exact, tokens or None, parent list,
    q_ids, q_logits, policy, hist) of one case."""
    if name in ("disjoint", "policy", "wide"):
        logits, qids, qlog, pol, hist, k = cpu_case(name)
        return dict(logits=_bf16_round(logits), k=k, parent=ov.chain_parents(k),
                    q_ids=np.asarray(qids, np.int32), q_log=np.asarray(qlog, np.float32),
                    pol=pol, hist=np.asarray(hist, np.int32), tokens=None)
    rng = np.random.default_rng({"point_mass": 4, "tree": 5}[name])
    if name == "point_mass":
        V, k = 30, 2
        logits = _bf16_round(rng.standard_normal((k + 1, V)) * 1.5)
        pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.02, top_p=0.95)
        tokens = [int(np.argmax(logits[0])), int(np.argsort(logits[1])[-2])]
        return dict(logits=logits, k=k, parent=ov.chain_parents(k), q_ids=None, q_log=None,
                    pol=pol, hist=np.zeros(0, np.int32), tokens=tokens)
    # tree: three children of the root on row 0's top tokens, a second level
    # under the first two, a third under node 3, and a duplicate child of the
    # root (node 6 repeats node 0's token: descent takes the lower index)
    V = 30
    parent = [-1, -1, -1, 0, 1, 3, -1]
    logits = _bf16_round(rng.standard_normal((len(parent) + 1, V)) * 1.5)
    top0 = np.argsort(-logits[0])
    tokens = [int(top0[0]), int(top0[1]), int(top0[2]), int(np.argmax(logits[1])),
              int(np.argmax(logits[2])), int(np.argsort(logits[4])[-2]), int(top0[0])]
    pol = ov.Policy(temperature=0.7, top_k=20, presence=1.5, window=8)
    hist = rng.integers(0, V, 12).astype(np.int32)
    hist[-2:] = tokens[3], tokens[1]          # penalties that differ between paths
    return dict(logits=logits, k=len(parent), parent=parent, q_ids=None, q_log=None, pol=pol,
                hist=hist, tokens=tokens)


class _Expected:
    """The oracle's distributions of one case: p of the row reached by an
    emitted prefix, and (chain with candidates) q of the next draft."""

    def __init__(self, c):
        self.c = c
        self.memo = {}

    def _prep(self, drafts):
        key = tuple(drafts)
        if key not in self.memo:
            c = self.c
            self.memo[key] = ov.prepare_rows(c["logits"], list(key), c["parent"], c["q_ids"],
                                             c["q_log"], c["hist"], c["pol"])
        return self.memo[key]

    def _pad(self, prefix):
        c = self.c
        if c["tokens"] is not None:
            return list(c["tokens"])
        return list(prefix) + [int(c["q_ids"][j, 0]) for j in range(len(prefix), c["k"])]

    def p(self, prefix):
        c = self.c
        if c["tokens"] is not None and not ov.is_chain(c["parent"]):
            node = -1                    # naive descent: walk the emitted prefix down the tree
            for y in prefix:
                node = next(j for j, p in enumerate(c["parent"])
                            if p == node and c["tokens"][j] == y)
            return self._prep(c["tokens"]).pdists[ov.row_of(node)]
        return self._prep(self._pad(prefix)).pdists[len(prefix)]

    def q(self, prefix):
        return self._prep(self._pad(prefix)).qdists[len(prefix)]


def _probs(dist):
    ids = np.asarray(dist.ids, np.int64)
    w = np.asarray([float(e) for e in dist.e], np.float64)
    return ids, w / w.sum()


def _groups(prefix_rows):
    """(distinct rows, index of each row's group) of a 2-D int array, also
    when it has no columns."""
    if prefix_rows.shape[1] == 0:
        return prefix_rows[:1], np.zeros(len(prefix_rows), np.int64)
    uniq, inv = np.unique(prefix_rows, axis=0, return_inverse=True)
    return uniq, inv.reshape(-1)


def _draw_drafts(c, exp, rng):
    """[TRIALS, k] drafts, each drawn from the verifier's q given the drafts
    before it (numpy's generator: independent of the GPU's Philox stream)."""
    k = c["k"]
    d = np.zeros((TRIALS, k), np.int32)
    for j in range(k):
        prefixes, inv = _groups(d[:, :j])
        for g, pre in enumerate(prefixes):
            sel = np.nonzero(inv == g)[0]
            ids, pr = _probs(exp.q(tuple(int(t) for t in pre)))
            d[sel, j] = ids[rng.choice(len(ids), size=len(sel), p=pr)]
    return d


def _request_dtype():
    """numpy layout of vr_request, so a whole request table is one array."""
    to_np = {ctypes.c_int32: np.int32, ctypes.c_void_p: np.uint64, ctypes.c_uint64: np.uint64,
             ctypes.c_float: np.float32}
    names, formats, offsets = [], [], []
    for name, ct in vb.vr_request._fields_:
        off = getattr(vb.vr_request, name).offset
        if ct is vb.vr_policy:
            for pn, pt in vb.vr_policy._fields_:
                names.append("policy_" + pn)
                formats.append(to_np[pt])
                offsets.append(off + getattr(vb.vr_policy, pn).offset)
        else:
            names.append(name)
            formats.append(to_np[ct])
            offsets.append(off)
    return np.dtype({"names": names, "formats": formats, "offsets": offsets,
                     "itemsize": ctypes.sizeof(vb.vr_request)})


def _run_gpu(c, drafts, path):
    """All TRIALS windows as requests of batched calls; returns
    (ids [TRIALS, k+1], accept [TRIALS], n_emitted [TRIALS], logits of one
    request)."""
    logits, k, pol = c["logits"], c["k"], c["pol"]
    R1, V = logits.shape
    per_call = min(vb.VR_MAX_REQUESTS, vb.VR_MAX_ROWS // R1)
    rows = per_call * R1
    W = np.zeros((V, HIDDEN), np.uint16)
    W[:, :R1] = synth.f32_to_bf16_bits(logits.T.copy())
    A = np.zeros((rows, HIDDEN), np.float32)
    A[np.arange(rows), np.arange(rows) % R1] = 1.0
    Wd, Ad = dev_weight(W), dev(A)
    tok = dev(drafts.reshape(-1) if c["tokens"] is None else np.asarray(c["tokens"], np.int32))
    par = None if ov.is_chain(c["parent"]) else dev(np.asarray(c["parent"], np.int32))
    qid = None if c["q_ids"] is None else dev(c["q_ids"])
    qlg = None if c["q_log"] is None else dev(c["q_log"])
    hist = dev(c["hist"]) if len(c["hist"]) else None
    out = torch.full((TRIALS, R1), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((TRIALS,), -7, dtype=torch.int32, device="cuda")
    nem = torch.full((TRIALS,), -7, dtype=torch.int32, device="cuda")
    g_logits = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(g_logits) if ov.penalties_active(pol) else None
    ws = vb.workspace(rows, HIDDEN, V)

    t = np.arange(TRIALS, dtype=np.uint64)
    tab = np.zeros(TRIALS, _request_dtype())
    tab["n_nodes"] = k
    tab["tokens"] = tok.data_ptr() + (t * np.uint64(4 * k) if c["tokens"] is None else 0)
    tab["parent"] = 0 if par is None else par.data_ptr()
    tab["q_ids"] = 0 if qid is None else qid.data_ptr()
    tab["q_logits"] = 0 if qlg is None else qlg.data_ptr()
    tab["hist"] = 0 if hist is None else hist.data_ptr()
    tab["hist_len"] = len(c["hist"])
    for name, _ in vb.vr_policy._fields_:
        tab["policy_" + name] = getattr(pol, name)
    tab["seed"] = t
    tab["position"] = POSITION
    tab["out_ids"] = out.data_ptr() + t * np.uint64(4 * R1)
    tab["out_accept"] = acc.data_ptr() + t * np.uint64(4)
    tab["out_n_emitted"] = nem.data_ptr() + t * np.uint64(4)

    lib = vb.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    base = tab.ctypes.data
    for first in range(0, TRIALS, per_call):
        n_req = min(per_call, TRIALS - first)
        reqs = ctypes.cast(ctypes.c_void_p(base + first * tab.itemsize),
                           ctypes.POINTER(vb.vr_request))
        st = lib.vr_verify_window_batched(ctypes.c_void_p(Wd.data_ptr()),
                                          ctypes.c_void_p(Ad.data_ptr()), HIDDEN, V, path, reqs,
                                          n_req, ctypes.c_void_p(g_logits.data_ptr()),
                                          None if pen is None else ctypes.c_void_p(pen.data_ptr()),
                                          ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
        assert st == vb.VR_OK
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    return (out.cpu().numpy(), acc.cpu().numpy(), nem.cpu().numpy(),
            g_logits[:R1].cpu().numpy())


def _chi2_parts(samples, dist):
    """(statistic, degrees of freedom) of samples against a RowDist, with
    categories of expected count below 5 merged; None if a sample lies
    outside the distribution's support."""
    ids, pr = _probs(dist)
    n = len(samples)
    if np.any(~np.isin(samples, ids)):
        return None
    obs = np.array([np.sum(samples == i) for i in ids], np.float64)
    exp = pr * n
    small = exp < 5
    if small.any():
        obs = np.append(obs[~small], obs[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
    keep = exp > 0
    obs, exp = obs[keep], exp[keep]
    if len(obs) < 2:
        return 0.0, 0
    return float(np.sum((obs - exp) ** 2 / exp)), len(obs) - 1


def _depth_pvalue(ids, n_em, depth, exp):
    """One p-value for the tokens emitted at `depth`, per emitted prefix."""
    reach = n_em > depth
    sub = ids[reach]
    prefixes, inv = _groups(sub[:, :depth])
    stat, dof = 0.0, 0
    for g, pre in enumerate(prefixes):
        parts = _chi2_parts(sub[inv == g, depth], exp.p(tuple(int(t) for t in pre)))
        if parts is None:
            return 0.0, int(reach.sum())
        stat += parts[0]
        dof += parts[1]
    return (float(stats.chi2.sf(stat, dof)) if dof else 1.0), int(reach.sum())


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_FFMA])
@pytest.mark.parametrize("name", ["disjoint", "policy", "wide", "point_mass", "tree"])
def test_gpu_emission_follows_p(name, path):
    c = _case(name)
    exp = _Expected(c)
    drafts = (_draw_drafts(c, exp, np.random.default_rng(77)) if c["tokens"] is None
              else np.tile(np.asarray(c["tokens"], np.int32), (TRIALS, 1)))
    ids, acc, n_em, g_logits = _run_gpu(c, drafts, path)
    # the projection returned the chosen logits bit for bit
    assert np.array_equal(g_logits.view(np.uint32), c["logits"].view(np.uint32))
    # every window emits at least one token, accepted + 1 of them
    assert n_em.min() >= 1 and np.array_equal(n_em, acc + 1)
    # the first windows are the oracle's, id for id
    for t in range(64):
        ref = ov.verify_window(c["logits"], drafts[t], c["parent"], c["q_ids"], c["q_log"],
                               c["hist"], c["pol"], seed=t, position=POSITION)
        assert list(ids[t, :n_em[t]]) == ref.emitted and acc[t] == ref.accept, t
    # depth 0 and 1 always; deeper while enough windows reach it
    for depth in range(c["k"] + 1):
        pval, n = _depth_pvalue(ids, n_em, depth, exp)
        if depth >= 2 and n < 5000:
            break
        assert n > 1000, (depth, n)
        assert pval > P_MIN, (name, depth, n, pval)
