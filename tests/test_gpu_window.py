"""The fused window on the GPU against the oracle, on the workloads of the
benchmark suite: tiny greedy chain, sampled chain (k 3), penalised chain
(k 8), token tree (3 x 8), batched serving (64 requests), plus the
multi-window history rule and the host-buffer entry point.

Parity here is stage-wise, so that no oracle input comes from the CUDA path:
  * logits: GPU vs the fp64 oracle, |d| <= 1e-3 * max(1, |ref|);
  * sampling: GPU sample_accept and the oracle on the same float32 logits
    (float32 of the oracle's fp64 logits): penalised rows, pools, ids and
    accept counts bit for bit;
  * the fused window's ids equal the GPU's own sample_accept on the window's
    logits, and equal the oracle's ids whenever both sides' pools agree (a
    near-tie in float32 can legitimately reorder a pool; such a window is
    counted, not compared)."""
import numpy as np
import pytest
import torch

from oracle import draft_policy as od, verify as ov
from speculative_decoding_verify_row_gb300 import binding as vb, synth
from gpu_common import require_gpu, dev, dev_weight, assert_logits_close, same_bits_f32

pytestmark = pytest.mark.gpu

# fused windows compared id for id with the oracle, out of all checked (the
# terminal summary prints the ratio, so a projection change that reorders
# pools shows up even while each test's threshold holds)
END_TO_END = {"windows": 0, "compared": 0}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def bpol(p):
    return vb.Policy(**p.__dict__)


def run_window(wd, act, tokens, pol, seed, position, parent=None, q_ids=None, q_log=None,
               hist=None, path=vb.VR_PATH_AUTO, separate_pen=True):
    R, H = act.shape
    V = wd.shape[0]
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(logits) if separate_pen else None
    out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ne = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = vb.workspace(R, H, V)
    vb.verify_window(wd, dev(act), dev(tokens) if len(tokens) else None, bpol(pol), seed, position,
                     logits, out, acc, ne, ws, parent=None if parent is None else dev(parent),
                     q_ids=None if q_ids is None else dev(q_ids),
                     q_logits=None if q_log is None else dev(q_log),
                     hist=None if hist is None or len(hist) == 0 else dev(hist), pen_logits=pen,
                     path=path)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    penalised = pen if (pen is not None and ov.penalties_active(pol)) else logits
    return dict(logits=logits, pen=penalised, ids=out.cpu().numpy(), accept=int(acc.item()),
                n=int(ne.item()), ws=ws)


def gpu_sample(pen_np, tokens, pol, seed, position, parent=None, q_ids=None, q_pen=None):
    R, V = pen_np.shape
    out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ne = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = vb.workspace(R, 8, V)
    vb.verify_sample_accept(dev(pen_np), dev(tokens) if len(tokens) else None, bpol(pol), seed,
                            position, out, acc, ne, ws, parent=None if parent is None else dev(parent),
                            q_ids=None if q_ids is None else dev(q_ids),
                            q_logits=None if q_pen is None else dev(q_pen))
    torch.cuda.synchronize()
    return list(out.cpu().numpy()[:int(ne.item())]), int(acc.item())


def check_window(win, ref_logits64, tokens, pol, seed, position, parent=None, q_ids=None,
                 q_log=None, hist=(), stats=None, logit_cols=None):
    """All stage-wise checks of one fused GPU window (see module doc)."""
    g_logits = win["logits"]
    if logit_cols is None:
        assert_logits_close(g_logits.cpu().numpy(), ref_logits64)
    else:
        c = torch.from_numpy(logit_cols).cuda()
        assert_logits_close(g_logits[:, c].cpu().numpy(), ref_logits64[:, logit_cols])
    plist = ov.chain_parents(len(tokens)) if parent is None else [int(p) for p in parent]
    ref32 = ref_logits64.astype(np.float32)
    # (1) oracle and GPU sampler on the same float32 logits
    ref = ov.verify_window(ref32, tokens, plist, q_ids, q_log, hist, pol, seed, position)
    g_ids, g_acc = gpu_sample(ref.pen_logits, tokens, pol, seed, position, parent, q_ids, ref.q_pen)
    assert (g_ids, g_acc) == (ref.emitted, ref.accept)
    # (2) the fused window equals the GPU's own stages run one by one on its
    # raw logits (penalize, then sample_accept)
    R, V = g_logits.shape
    pen_again = g_logits.clone()
    q_again = None if q_log is None else dev(q_log)
    ws = vb.workspace(R, 8, V)
    vb.verify_penalize(pen_again, dev(tokens) if len(tokens) else None,
                       dev(np.asarray(hist, np.int32)) if len(hist) else None, bpol(pol), ws,
                       parent=None if parent is None else dev(parent),
                       q_ids=None if q_ids is None else dev(q_ids), q_logits=q_again)
    torch.cuda.synchronize()
    assert torch.equal(pen_again.view(torch.int32), win["pen"].view(torch.int32))
    g_pen = win["pen"].cpu().numpy()
    own_ids, own_acc = gpu_sample(g_pen, tokens, pol, seed, position, parent, q_ids,
                                  None if q_again is None else q_again.cpu().numpy())
    assert list(win["ids"][:win["n"]]) == own_ids and win["accept"] == own_acc
    assert 1 <= win["n"] == win["accept"] + 1
    # (3) end to end against the oracle when both sides' pools agree
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.verify_select(win["pen"].contiguous(), ids, vals, ws)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    same_pools = all(np.array_equal(ids[r, :len(ref.pool_ids[r])], ref.pool_ids[r]) for r in range(R))
    if stats is not None:
        stats["windows"] = stats.get("windows", 0) + 1
        stats["compared"] = stats.get("compared", 0) + int(same_pools)
    END_TO_END["windows"] += 1
    END_TO_END["compared"] += int(same_pools)
    if same_pools:
        assert list(win["ids"][:win["n"]]) == ref.emitted and win["accept"] == ref.accept
    return ref


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_FFMA])
def test_tiny_greedy_chain(path):
    """hidden 256, vocab 4096, k 3; drafts = the oracle's argmax chain with
    row 2 perturbed: two drafts accepted, three tokens emitted."""
    W = synth.weights(4096, 256)
    A = synth.activations(4, 256, 0)
    L64 = ov.project(W, A)
    am = [int(ov.target_pool(L64[r].astype(np.float32))[0][0]) for r in range(4)]
    drafts = synth.perturb_draft(am, 3, 2, 4096, seed=0)
    win = run_window(dev_weight(W), A, drafts, ov.Policy(), 0, 100, path=path)
    ref = check_window(win, L64, drafts, ov.Policy(), 0, 100)
    assert ref.accept == 2 and win["accept"] == 2 and win["n"] == 3
    assert list(win["ids"][:3]) == am[:2] + [am[2]]


def chain_inputs(bw, k, window_seed, pol_q_temp=0.7):
    A = synth.activations(k + 1, bw.hidden, window_seed)
    L64 = bw.oracle_logits(A)
    top = [ov.target_pool(L64[r].astype(np.float32)) for r in range(k + 1)]
    t32_ids = np.stack([t[0][:32] for t in top[:k]])
    t32_val = np.stack([t[1][:32] for t in top[:k]])
    q_ids, q_log = synth.draft_candidates(t32_ids, t32_val, seed=window_seed)
    slot = synth.draft_choice(q_log, pol_q_temp, seed=window_seed + 1)
    drafts = q_ids[np.arange(k), slot].astype(np.int32)
    return A, L64, q_ids, q_log, drafts


def cols_sample(V, seed, n=2000):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, V, n), [0, V - 1]]))


def test_sampled_chain_full_size(big_weights_4096):
    """hidden 4096, vocab 151936, k 3; T 0.7, top-k absent, min-p 0.05,
    top-p 0.95, no penalties; several window seeds."""
    bw = big_weights_4096
    pol = ov.Policy(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95)
    stats = {}
    for s in range(6):
        A, L64, q_ids, q_log, drafts = chain_inputs(bw, 3, s)
        win = run_window(bw.dev, A, drafts, pol, s, 4096 + s, q_ids=q_ids, q_log=q_log)
        check_window(win, L64, drafts, pol, s, 4096 + s, q_ids=q_ids, q_log=q_log, stats=stats)
    assert stats["compared"] >= 4


@pytest.mark.parametrize("mode", ["greedy", "sampled", "penalised"])
def test_window_over_stale_buffers(big_weights_4096, mode):
    """A 4-row window's row kernel starts while the projection runs and works
    once through the logits and group maxima as they stand, before its wait.
    Here both hold another window's values and the logits are then set to
    -inf, so that the stale maxima pick groups with no entry at their level
    (an empty pool in that pass).  The window must give exactly what it gives
    on fresh buffers.  The logits sit behind a 64-float guard inside their
    allocation."""
    bw = big_weights_4096
    R, V, H = 4, 151936, 4096
    pol = {"greedy": ov.Policy(),
           "sampled": ov.Policy(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95),
           "penalised": ov.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95, repeat=1.1,
                                  presence=1.5, frequency=0.2, window=64)}[mode]
    hist = synth.zipf_history(4096, V, seed=41) if mode == "penalised" else None
    A, L64, q_ids, q_log, drafts = chain_inputs(bw, 3, 40)
    fresh = run_window(bw.dev, A, drafts, pol, 40, 4096, q_ids=q_ids, q_log=q_log, hist=hist,
                       separate_pen=False)

    guard = torch.zeros(64 + R * V, dtype=torch.float32, device="cuda")
    logits = guard[64:].view(R, V)
    ws = vb.workspace(R, H, V)
    out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ne = torch.zeros(1, dtype=torch.int32, device="cuda")
    hd = None if hist is None else dev(hist)

    def window(act, tokens, qi, ql):
        vb.verify_window(bw.dev, dev(act), dev(tokens), bpol(pol), 40, 4096, logits, out, acc, ne,
                         ws, q_ids=dev(qi), q_logits=dev(ql), hist=hd)

    A2, _, q_ids2, q_log2, drafts2 = chain_inputs(bw, 3, 41)
    window(A2, drafts2, q_ids2, q_log2)           # another window's logits and maxima
    logits.fill_(-float("inf"))
    window(A, drafts, q_ids, q_log)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    assert torch.equal(logits.view(torch.int32), fresh["logits"].view(torch.int32))
    n = int(ne.item())
    assert (n, int(acc.item())) == (fresh["n"], fresh["accept"])
    assert list(out.cpu().numpy()[:n]) == list(fresh["ids"][:n])
    assert torch.all(guard[:64] == 0)


def test_penalised_chain_full_size(big_weights_4096):
    """k 8 (9 rows), 4096-token Zipf(1.1) history, W 64, repeat 1.1,
    presence 1.5, frequency 0.2, top-k 0 (the 64-wide pool).  The last
    window plants row 0's pool tokens in the last 64 history slots, so that
    the penalties reorder the pool."""
    bw = big_weights_4096
    pol = ov.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95, repeat=1.1, presence=1.5,
                    frequency=0.2, window=64)
    stats = {}
    for s in range(3):
        A, L64, q_ids, q_log, drafts = chain_inputs(bw, 8, 100 + s)
        hist = synth.zipf_history(4096, 151936, seed=100 + s)
        if s == 2:
            hist[-64:] = ov.target_pool(L64[0].astype(np.float32))[0][:64]
        win = run_window(bw.dev, A, drafts, pol, s, 4096, q_ids=q_ids, q_log=q_log, hist=hist)
        ref = check_window(win, L64, drafts, pol, s, 4096, q_ids=q_ids, q_log=q_log, hist=hist,
                           stats=stats, logit_cols=cols_sample(151936, s))
        # penalties applied in place (no separate buffer): same rows, same ids
        inplace = run_window(bw.dev, A, drafts, pol, s, 4096, q_ids=q_ids, q_log=q_log, hist=hist,
                             separate_pen=False)
        assert torch.equal(inplace["logits"].view(torch.int32), win["pen"].view(torch.int32))
        assert list(inplace["ids"][:inplace["n"]]) == list(win["ids"][:win["n"]])
        if s == 2:
            raw_pool = ov.target_pool(L64[0].astype(np.float32))[0]
            assert not np.array_equal(ref.pool_ids[0], raw_pool)
    assert stats["compared"] >= 2


@pytest.mark.parametrize("temperature", [0.0, 0.7])
def test_token_tree_full_size(big_weights_4096, temperature):
    """3 branches x depth 8 (24 nodes, 25 rows); branch 0 agrees with the
    target for 5 nodes.  Greedy: longest agreeing branch; sampled (T 0.7,
    top-k 20): naive descent with per-node penalty histories (W 64,
    presence 1.5)."""
    bw = big_weights_4096
    parent = synth.tree_parents(3, 8)
    pol = ov.Policy(temperature=temperature, top_k=20, presence=1.5, window=64)
    stats = {}
    for s in range(3):
        A = synth.activations(25, 4096, 200 + s)
        L64 = bw.oracle_logits(A)
        pools = [ov.target_pool(L64[r].astype(np.float32))[0] for r in range(25)]
        tokens = synth.tree_tokens([p[0] for p in pools], [p[:32] for p in pools], seed=200 + s)
        hist = synth.zipf_history(2048, 151936, seed=200 + s)
        win = run_window(bw.dev, A, tokens, pol, s, 2048, parent=parent, hist=hist)
        ref = check_window(win, L64, tokens, pol, s, 2048, parent=parent, hist=hist, stats=stats,
                           logit_cols=cols_sample(151936, 300 + s))
        if temperature == 0.0:
            assert ref.accept >= 5          # branch 0 agrees for 5 nodes at least
    assert stats["compared"] >= 2


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH])
def test_batched_serving(big_weights_5120, path):
    """64 requests x k 3 (256 rows), hidden 5120; even requests greedy, odd
    ones T 0.8 / top-k 20 / top-p 0.9 / presence 1.5; 2048-token Zipf
    histories, W 64, seeds 0..63.  Checked on 8 requests against the
    oracle, on all of them against the GPU's own per-request windows."""
    bw = big_weights_5120
    nreq, k, H, V = 64, 3, 5120, 151936
    A = synth.activations(nreq * (k + 1), H, 500)
    check = set(range(0, nreq, 8)) | {1, 63}
    rows = [r for b in sorted(check) for r in range(b * (k + 1), (b + 1) * (k + 1))]
    L64_rows = bw.oracle_logits(A[rows])
    L64 = {b: L64_rows[i * (k + 1):(i + 1) * (k + 1)] for i, b in enumerate(sorted(check))}
    reqs, keep, specs = [], [], []
    rng = np.random.default_rng(500)
    for b in range(nreq):
        greedy = b % 2 == 0
        pol = ov.Policy() if greedy else ov.Policy(temperature=0.8, top_k=20, top_p=0.9,
                                                   presence=1.5, window=64)
        hist = synth.zipf_history(2048, V, seed=1000 + b)
        # draft candidates around a plausible region (the top-32 is known
        # only for the checked requests; the rest use random ids)
        if b in L64:
            top = [ov.target_pool(L64[b][r].astype(np.float32)) for r in range(k)]
            q_ids, q_log = synth.draft_candidates(np.stack([t[0][:32] for t in top]),
                                                  np.stack([t[1][:32] for t in top]), seed=b)
        else:
            q_ids = rng.integers(0, V, (k, 8)).astype(np.int32)
            q_log = rng.standard_normal((k, 8)).astype(np.float32)
        slot = synth.draft_choice(q_log, 0.0 if greedy else 0.8, seed=b + 7)
        drafts = q_ids[np.arange(k), slot].astype(np.int32)
        t = dict(tok=dev(drafts), q=dev(q_ids), ql=dev(q_log), h=dev(hist),
                 out=torch.full((k + 1,), -7, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                 n=torch.zeros(1, dtype=torch.int32, device="cuda"))
        keep.append(t)
        specs.append((drafts, q_ids, q_log, hist, pol))
        reqs.append(vb.make_request(k, t["tok"], bpol(pol), b, 2048, t["out"], t["acc"], t["n"],
                                    q_ids=t["q"], q_logits=t["ql"], hist=t["h"]))
    R = nreq * (k + 1)
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(logits)
    ws = vb.workspace(R, H, V)
    vb.verify_window_batched(bw.dev, dev(A), reqs, logits, ws, pen_logits=pen, path=path)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    stats = {}
    for b in range(nreq):
        drafts, q_ids, q_log, hist, pol = specs[b]
        sl = slice(b * (k + 1), (b + 1) * (k + 1))
        penalised = pen if ov.penalties_active(pol) else logits
        win = dict(logits=logits[sl], pen=penalised[sl], ids=keep[b]["out"].cpu().numpy(),
                   accept=int(keep[b]["acc"].item()), n=int(keep[b]["n"].item()))
        if b in L64:
            check_window(win, L64[b], drafts, pol, b, 2048, q_ids=q_ids, q_log=q_log, hist=hist,
                         stats=stats, logit_cols=cols_sample(V, b, 500))
        else:
            scratch = win["logits"].clone()
            q_pen = dev(q_log)
            vb.verify_penalize(scratch, dev(drafts), dev(hist), bpol(pol), vb.workspace(k + 1, 8, V),
                               q_ids=dev(q_ids), q_logits=q_pen)
            torch.cuda.synchronize()
            own_ids, own_acc = gpu_sample(win["pen"].cpu().numpy(), drafts, pol, b, 2048, None,
                                          q_ids, q_pen.cpu().numpy())
            assert list(win["ids"][:win["n"]]) == own_ids and win["accept"] == own_acc
    assert stats["compared"] >= 6


def test_multi_window_history():
    """Four consecutive windows of one request: the next history is the old
    one plus the emitted ids only (never a rejected draft), and the
    position advances by the number emitted."""
    rng = np.random.default_rng(9)
    V, H, k = 5000, 256, 4
    W = synth.weights(V, H)
    wd = dev_weight(W)
    pol = ov.Policy(temperature=0.9, top_k=0, presence=1.5, frequency=0.3, window=16)
    hist = list(rng.integers(0, V, 40))
    position = len(hist)
    for w in range(4):
        A = synth.activations(k + 1, H, 700 + w)
        L64 = ov.project(W, A)
        top = [ov.target_pool(L64[r].astype(np.float32)) for r in range(k)]
        q_ids, q_log = synth.draft_candidates(np.stack([t[0][:32] for t in top]),
                                              np.stack([t[1][:32] for t in top]), seed=w)
        drafts = q_ids[np.arange(k), synth.draft_choice(q_log, 0.9, seed=w)].astype(np.int32)
        win = run_window(wd, A, drafts, pol, 42, position, q_ids=q_ids, q_log=q_log,
                         hist=np.array(hist, np.int32))
        ref = check_window(win, L64, drafts, pol, 42, position, q_ids=q_ids, q_log=q_log, hist=hist)
        emitted = [int(t) for t in win["ids"][:win["n"]]]
        rejected = [int(d) for d in drafts[win["accept"]:]]
        hist = hist + emitted
        position += len(emitted)
        assert hist[-len(emitted):] == emitted
        if rejected and win["accept"] < k:
            assert hist[len(hist) - len(emitted):] == emitted


@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_point_matches_device_entry_point(big_weights_4096, pinned):
    """Pinned host buffers are read and written by the kernels through their
    mapped addresses; pageable ones go through copies.  Both equal the
    device entry point."""
    bw = big_weights_4096
    pol = ov.Policy(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95, presence=1.5, window=64)
    A, L64, q_ids, q_log, drafts = chain_inputs(bw, 3, 77)
    hist = synth.zipf_history(4096, 151936, seed=77)
    win = run_window(bw.dev, A, drafts, pol, 77, 4096, q_ids=q_ids, q_log=q_log, hist=hist)
    if pinned:
        pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    else:
        pin = lambda x: torch.from_numpy(np.ascontiguousarray(x).copy())
    logits = torch.empty((4, 151936), dtype=torch.float32, device="cuda")
    out = pin(np.full(4, -7, np.int32))
    ws = vb.workspace(4, 4096, 151936)
    acc, n = vb.verify_window_host(bw.dev, pin(A), pin(drafts), bpol(pol), 77, 4096, logits, out, ws,
                                   q_ids_h=pin(q_ids), q_logits_h=pin(q_log), hist_h=pin(hist))
    assert (acc, n) == (win["accept"], win["n"])
    assert list(out.numpy()[:n]) == list(win["ids"][:n])
    # no separate penalised buffer was given, so the penalties went in place
    assert torch.equal(logits.view(torch.int32), win["pen"].view(torch.int32))


def test_async_host_entry_point_pipelined(big_weights_4096):
    """Several host-buffer windows enqueued back to back without waiting, each
    read after its event: every one equals the same window run alone."""
    bw = big_weights_4096
    pol = ov.Policy(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95)
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    logits = torch.empty((4, 151936), dtype=torch.float32, device="cuda")
    ws = vb.workspace(4, 4096, 151936)
    stream = torch.cuda.current_stream()
    cases, pending = [], []
    for w in range(4):
        A, L64, q_ids, q_log, drafts = chain_inputs(bw, 3, 300 + w)
        cases.append((A, q_ids, q_log, drafts))
        h = (pin(A), pin(drafts), pin(q_ids), pin(q_log))
        # the last window's result goes to pageable memory: one copy instead
        out = pin(np.full(6, -7, np.int32)) if w < 3 else torch.full((6,), -7, dtype=torch.int32)
        vb.verify_window_host_async(bw.dev, h[0], h[1], bpol(pol), 300 + w, 4096, logits, out, ws,
                                    q_ids_h=h[2], q_logits_h=h[3], stream=stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        pending.append((ev, out, h))
    for w, (ev, out, _) in enumerate(pending):
        ev.synchronize()
        A, q_ids, q_log, drafts = cases[w]
        win = run_window(bw.dev, A, drafts, pol, 300 + w, 4096, q_ids=q_ids, q_log=q_log)
        got = out.numpy()
        assert (int(got[0]), int(got[1])) == (win["accept"], win["n"])
        assert list(got[2:2 + win["n"]]) == list(win["ids"][:win["n"]])


@pytest.mark.parametrize("shape", ["chain", "tree_greedy", "tree_sampled"])
def test_ngram_drafted_windows_full_size(big_weights_4096, shape):
    """Drafts from prompt lookup over the request's own context ("Speculative
    decoding on RDNA" §06: match 5, propose 3, sampled candidates verified
    against a point-mass q; "Spend the budget on a tree": three matches at
    depth 8 as one tree).  The oracle's proposal feeds both sides; the
    library's own proposer must give the same tree."""
    bw = big_weights_4096
    V = 151936
    stats = {}
    for s in range(3):
        ctx = synth.ngram_context(2048, V, seed=900 + s)
        if shape == "chain":
            toks, par = od.ngram_propose(ctx, 5, 3, 1, 63)
            pol = ov.Policy(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95, presence=1.5,
                            window=64)
        else:
            toks, par = od.ngram_propose(ctx, 5, 8, 3, 24)
            pol = ov.Policy(temperature=0.0 if shape == "tree_greedy" else 0.7, top_k=20,
                            presence=1.5, window=64)
        lt, lp = vb.ngram_propose(ctx, 5, 3 if shape == "chain" else 8,
                                  1 if shape == "chain" else 3, 63 if shape == "chain" else 24)
        assert list(lt) == toks and list(lp) == par
        tokens = np.array(toks, np.int32)
        parent = None if shape == "chain" else np.array(par, np.int32)
        R = len(tokens) + 1
        A = synth.activations(R, 4096, 900 + s)
        L64 = bw.oracle_logits(A)
        win = run_window(bw.dev, A, tokens, pol, s, len(ctx), parent=parent, hist=ctx)
        check_window(win, L64, tokens, pol, s, len(ctx), parent=parent, hist=ctx, stats=stats,
                     logit_cols=cols_sample(V, 900 + s))
    assert stats["compared"] >= 2


def _bf16_column(values):
    """float32 values (NaN allowed) -> bf16 bits (finite values rounded to
    nearest even, NaN as the quiet NaN 0x7fc0)."""
    v = np.asarray(values, np.float32)
    bits = synth.f32_to_bf16_bits(np.where(np.isnan(v), 0.0, v).astype(np.float32))
    bits[np.isnan(v)] = 0x7FC0
    return bits


def _crafted_rows(V, seed):
    """Four logit rows that stress the group-maxima selection: all entries
    equal (every group ties, 2048 candidates); a top value shared by a block
    of 40 ids and ~30 scattered ids; four distinct values with NaNs; distinct
    values with 20 % NaN, a whole NaN group and a top cluster in bf16 ties."""
    rng = np.random.default_rng(seed)
    rows = np.empty((4, V), np.float32)
    rows[0] = 0.5
    r1 = rng.standard_normal(V).astype(np.float32)
    r1[rng.random(V) < 30.0 / V] = 3.0
    r1[64:104] = 3.0
    rows[1] = r1
    r2 = rng.choice(np.array([-1.0, 0.0, 0.25, 1.0], np.float32), V, p=[0.3, 0.2, 0.25, 0.25])
    r2[rng.random(V) < 0.05] = np.nan
    rows[2] = r2
    r3 = rng.standard_normal(V).astype(np.float32)
    r3[rng.random(V) < 0.2] = np.nan
    r3[32:96] = 5.0 + 0.01 * np.arange(64, dtype=np.float32)[:len(r3[32:96])]
    r3[160:192] = np.nan
    rows[3] = r3
    return rows


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH, vb.VR_PATH_FFMA])
@pytest.mark.parametrize("V", [1, 33, 100, 2047, 5000, 151936, 163840, 163841])
@pytest.mark.parametrize("mode", ["greedy", "sampled", "penalised"])
def test_row_pools_on_crafted_logits(V, mode, path):
    """With one-hot activations the projection returns chosen bf16 values
    exactly (logits[r][v] = W[v][r], NaN where W[v] holds a NaN), so the
    pool selection of the window
    path (group maxima from the projection epilogue, then the row kernel; the
    segment select and its merge past 5120 groups and on the CUDA-core path)
    meets ties across groups, gathers past its fast capacity, NaN and
    vocabularies with fewer than 64 groups.
    Pools must equal the oracle's pool of the same rows bit for bit, and the
    window's result the oracle's window on them."""
    _check_crafted_window(_crafted_rows(V, seed=V), V, mode, path)


def _tied_group_rows(V, seed):
    """Four rows whose top value fills whole 32-id groups: 96 groups (3072
    tied entries), 97 groups, exactly 64 groups (2048, all the gather can
    hold) and 64 groups plus one more top entry in a 65th.  The row kernel
    must pick the 64 lowest-index groups among more than 64 tied maxima and
    rank a full gather of tied candidates.  The rest are standard normal
    draws, far below the top value 8."""
    rng = np.random.default_rng(seed)
    rows = rng.standard_normal((4, V)).astype(np.float32)
    rows[0, :96 * 32] = 8.0
    rows[1, :97 * 32] = 8.0
    rows[2, :64 * 32] = 8.0
    rows[3, :64 * 32] = 8.0
    rows[3, 300 * 32 + 5] = 8.0
    return rows


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH])
@pytest.mark.parametrize("mode", ["greedy", "sampled", "penalised"])
def test_row_pools_on_tied_top_groups(mode, path):
    """Rows whose top value fills 64, 65, 96 or 97 whole groups: pools and the
    window's result equal the oracle's."""
    V = 151936
    _check_crafted_window(_tied_group_rows(V, seed=11), V, mode, path)


def _check_crafted_window(rows, V, mode, path):
    H, R = 64, 4
    rng = np.random.default_rng(V + 1)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * np.float32(0.1))
    for r in range(R):
        W[:, r] = _bf16_column(rows[r])
    A = np.zeros((R, H), np.float32)
    A[np.arange(R), np.arange(R)] = 1.0
    # W[v][r] exactly, except that a NaN anywhere in W[v] reaches every row
    # (NaN x 0); the fp64 oracle projection is exact here
    exact = ov.project(W, A).astype(np.float32)
    if mode == "greedy":
        pol = ov.Policy(temperature=0.0)
    elif mode == "sampled":
        pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.0, top_p=1.0)
    else:
        pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.0, top_p=1.0, presence=0.75,
                        frequency=0.25, window=64)
    argmax = [int(ov.target_pool(exact[r])[0][0]) for r in range(R)]
    drafts = np.array([argmax[0], argmax[1], int(rng.integers(0, V))], np.int32)
    hist = np.array([argmax[0], 64, 65, 32, 33, 7] * 3, np.int32) % V if mode == "penalised" else None
    win = run_window(dev_weight(W), A, drafts, pol, 5, 100, hist=hist, path=path)
    assert same_bits_f32(win["logits"].cpu().numpy(), exact)
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.window_pools(win["ws"], R, H, V, ids, vals)
    torch.cuda.synchronize()
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    pen = win["pen"].cpu().numpy()
    # only the argmax is defined for a greedy request
    n = 1 if mode == "greedy" else min(64, V)
    for r in range(R):
        want_ids, want_vals = ov.target_pool(pen[r])
        assert np.array_equal(ids[r, :n], want_ids[:n]), (mode, V, r)
        assert same_bits_f32(vals[r, :n], want_vals[:n]), (mode, V, r)
        if mode != "greedy":
            assert (ids[r, n:] == -1).all()
    ref = ov.verify_window(win["logits"].cpu().numpy(), drafts, hist=() if hist is None else hist,
                           pol=pol, seed=5, position=100)
    if mode == "penalised":
        assert same_bits_f32(pen, ref.pen_logits)
    assert list(win["ids"][:win["n"]]) == ref.emitted and win["accept"] == ref.accept


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH])
@pytest.mark.parametrize("V", [1000, 151936])
def test_batched_requests_on_crafted_logits(V, path):
    """One batched call over eight requests of different shapes and policies
    (chain of 4 rows, a single row, a 5-row tree, chain of 8 rows; greedy,
    sampled against draft candidates, sampled against the point mass,
    penalised) on crafted logits (one-hot activations: row r reads weight
    column r % 64, each column a tie/NaN pattern or random bf16 values).
    Every row's pool and every request's result must equal the oracle's on
    the GPU's own logits."""
    H = 64
    rng = np.random.default_rng(V + 7)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * np.float32(0.1))
    base = _crafted_rows(V, seed=V + 3)
    for c in range(H):
        if c % 4 == 0 and c // 4 < 4:
            W[:, c] = _bf16_column(base[c // 4])
        elif c % 3 == 0:
            # few distinct values: ties everywhere
            W[:, c] = _bf16_column(rng.choice(np.array([-0.5, 0.5, 1.0, 2.0], np.float32), V))
    shapes = [(3, None), (0, None), (4, [-1, 0, -1, 2]), (7, None)] * 2
    pols = [ov.Policy(temperature=0.0),
            ov.Policy(temperature=0.8, top_k=0, min_p=0.0, top_p=1.0),
            ov.Policy(temperature=0.7, top_k=20, min_p=0.05, top_p=0.9),
            ov.Policy(temperature=0.8, top_k=0, presence=0.75, frequency=0.25, window=64),
            ov.Policy(temperature=0.0, presence=1.5, window=16),
            ov.Policy(temperature=1.1, top_k=5, min_p=0.0, top_p=0.8),
            ov.Policy(temperature=0.5, top_k=64, min_p=0.2, top_p=1.0, repeat=1.3, window=8),
            ov.Policy(temperature=0.9, top_k=-1, min_p=0.0, top_p=0.95)]
    rows_of = []
    r0 = 0
    for n, _ in shapes:
        rows_of.append(list(range(r0, r0 + n + 1)))
        r0 += n + 1
    R = r0
    A = np.zeros((R, H), np.float32)
    A[np.arange(R), np.arange(R) % H] = 1.0
    exact = ov.project(W, A).astype(np.float32)
    reqs, keep, specs = [], [], []
    for b, ((n, parent), pol) in enumerate(zip(shapes, pols)):
        par = ov.chain_parents(n) if parent is None else parent
        am = [int(ov.target_pool(exact[rows_of[b][0] + (0 if p < 0 else 1 + p)])[0][0]) for p in par]
        tokens = np.array([am[j] if j % 2 == 0 else int(rng.integers(0, V)) for j in range(n)],
                          np.int32)
        with_q = parent is None and n > 0 and b % 2 == 1 and pol.temperature > 0
        q_ids = q_log = None
        if with_q:
            q_ids = rng.integers(0, V, (n, 8)).astype(np.int32)
            q_ids[:, 0] = tokens
            q_log = rng.standard_normal((n, 8)).astype(np.float32)
        hist = (rng.integers(0, V, 40).astype(np.int32) if ov.penalties_active(pol) else None)
        t = dict(tok=dev(tokens) if n else None,
                 par=None if parent is None else dev(np.array(parent, np.int32)),
                 q=None if q_ids is None else dev(q_ids), ql=None if q_log is None else dev(q_log),
                 h=None if hist is None else dev(hist),
                 out=torch.full((n + 1,), -7, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                 n=torch.zeros(1, dtype=torch.int32, device="cuda"))
        keep.append(t)
        specs.append((tokens, parent, q_ids, q_log, hist, pol))
        reqs.append(vb.make_request(n, t["tok"], bpol(pol), 40 + b, 300 + b, t["out"], t["acc"],
                                    t["n"], parent=t["par"], q_ids=t["q"], q_logits=t["ql"],
                                    hist=t["h"]))
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(logits)
    ws = vb.workspace(R, H, V)
    vb.verify_window_batched(dev_weight(W), dev(A), reqs, logits, ws, pen_logits=pen, path=path)
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.window_pools(ws, R, H, V, ids, vals)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    g_logits = logits.cpu().numpy()
    assert same_bits_f32(g_logits, exact)
    ids, vals, g_pen = ids.cpu().numpy(), vals.cpu().numpy(), pen.cpu().numpy()
    refs = ov.verify_batched(g_logits, [dict(tokens=tokens, parent=parent, q_ids=q_ids,
                                             q_logits=q_log, hist=() if hist is None else hist,
                                             pol=pol, seed=40 + b, position=300 + b)
                                        for b, (tokens, parent, q_ids, q_log, hist, pol)
                                        in enumerate(specs)])
    for b, (tokens, parent, q_ids, q_log, hist, pol) in enumerate(specs):
        rs = rows_of[b]
        ref = refs[b]
        rows_pen = g_pen[rs] if ov.penalties_active(pol) else g_logits[rs]
        if ov.penalties_active(pol):
            assert same_bits_f32(rows_pen, ref.pen_logits), b
        for i, r in enumerate(rs):
            want_ids, want_vals = ov.target_pool(rows_pen[i])
            n = 1 if pol.temperature == 0.0 else len(want_ids)   # greedy: the argmax only
            assert np.array_equal(ids[r, :n], want_ids[:n]), (b, i)
            assert same_bits_f32(vals[r, :n], want_vals[:n]), (b, i)
        n_em = int(keep[b]["n"].item())
        assert list(keep[b]["out"].cpu().numpy()[:n_em]) == ref.emitted, b
        assert int(keep[b]["acc"].item()) == ref.accept, b


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH, vb.VR_PATH_FFMA])
@pytest.mark.parametrize("shape", ["chain", "tree"])
def test_largest_window_and_penalty_window(shape, path):
    """The largest window (64 rows: 63 drafts in a chain, or a 63-node tree)
    with the largest penalty window (W 512 over a 600-token history), sampled,
    full vocabulary: the result equals the oracle's window on the GPU's own
    logits, and every pool equals the oracle's pool of the penalised rows."""
    H, V, R = 64, 151936, vb.VR_MAX_WINDOW_ROWS
    n = R - 1
    rng = np.random.default_rng(640 + path)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * np.float32(0.3))
    A = rng.standard_normal((R, H)).astype(np.float32)
    if shape == "chain":
        parent = None
        plist = ov.chain_parents(n)
    else:
        # 7 branches of 9 nodes from the root
        plist = [-1 if j % 9 == 0 else j - 1 for j in range(n)]
        parent = np.array(plist, np.int32)
    # drafts: the oracle's argmax of each parent row for most nodes, so the
    # acceptance walks deep
    L64 = ov.project(W, A)
    am = [int(ov.target_pool(L64[r].astype(np.float32))[0][0]) for r in range(R)]
    tokens = np.array([am[0 if p < 0 else 1 + p] if j % 11 else int(rng.integers(0, V))
                       for j, p in enumerate(plist)], np.int32)
    hist = rng.integers(0, V, 600).astype(np.int32)
    hist[-40:] = tokens[:40] if n >= 40 else hist[-40:]
    pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.0, top_p=0.97, repeat=1.2, presence=0.5,
                    frequency=0.1, window=vb.VR_MAX_PENALTY_WINDOW)
    win = run_window(dev_weight(W), A, tokens, pol, 9, 1000, parent=parent, hist=hist, path=path)
    g_logits = win["logits"].cpu().numpy()
    assert_logits_close(g_logits, L64)
    ref = ov.verify_window(g_logits, tokens, plist, None, None, hist, pol, 9, 1000)
    pen = win["pen"].cpu().numpy()
    assert same_bits_f32(pen, ref.pen_logits)
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.window_pools(win["ws"], R, H, V, ids, vals)
    torch.cuda.synchronize()
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    for r in range(R):
        want_ids, want_vals = ov.target_pool(pen[r])
        assert np.array_equal(ids[r], want_ids) and same_bits_f32(vals[r], want_vals), r
    assert list(win["ids"][:win["n"]]) == ref.emitted and win["accept"] == ref.accept
    assert win["n"] >= 1


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH])
def test_largest_batched_call(path):
    """The largest batched call: VR_MAX_REQUESTS requests of 4 rows each
    (VR_MAX_ROWS rows in one projection), greedy, sampled and penalised
    requests mixed; every request equals the oracle's window on the GPU's
    own logits."""
    H, V = 64, 5000
    nreq, k = vb.VR_MAX_REQUESTS, 3
    R = nreq * (k + 1)
    assert R == vb.VR_MAX_ROWS
    rng = np.random.default_rng(1024 + path)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * np.float32(0.3))
    A = rng.standard_normal((R, H)).astype(np.float32)
    pols = [ov.Policy(), ov.Policy(temperature=0.8, top_k=20, top_p=0.9),
            ov.Policy(temperature=0.7, top_k=0, min_p=0.05, presence=1.0, window=32),
            ov.Policy(temperature=0.0, repeat=1.3, window=8)]
    reqs, keep, specs = [], [], []
    for b in range(nreq):
        pol = pols[b % 4]
        tokens = rng.integers(0, V, k).astype(np.int32)
        hist = rng.integers(0, V, 50).astype(np.int32)
        t = dict(tok=dev(tokens), h=dev(hist),
                 out=torch.full((k + 1,), -7, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                 n=torch.zeros(1, dtype=torch.int32, device="cuda"))
        keep.append(t)
        specs.append((tokens, hist, pol))
        reqs.append(vb.make_request(k, t["tok"], bpol(pol), b, 77, t["out"], t["acc"], t["n"],
                                    hist=t["h"]))
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(logits)
    ws = vb.workspace(R, H, V)
    vb.verify_window_batched(dev_weight(W), dev(A), reqs, logits, ws, pen_logits=pen, path=path)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    g_logits = logits.cpu().numpy()
    g_pen = pen.cpu().numpy()
    assert_logits_close(g_logits[:64], ov.project(W, A[:64]))
    refs = ov.verify_batched(g_logits, [dict(tokens=tokens, hist=hist, pol=pol, seed=b,
                                             position=77)
                                        for b, (tokens, hist, pol) in enumerate(specs)])
    for b, (tokens, hist, pol) in enumerate(specs):
        rs = slice(b * (k + 1), (b + 1) * (k + 1))
        ref = refs[b]
        if ov.penalties_active(pol):
            assert same_bits_f32(g_pen[rs], ref.pen_logits), b
        n_em = int(keep[b]["n"].item())
        assert list(keep[b]["out"].cpu().numpy()[:n_em]) == ref.emitted, b
        assert int(keep[b]["acc"].item()) == ref.accept, b


@pytest.mark.parametrize("path", [vb.VR_PATH_TC, vb.VR_PATH_FFMA])
@pytest.mark.parametrize("rows", [31, 32, 33])
@pytest.mark.parametrize("mode", ["greedy", "sampled_q", "point_mass"])
def test_chains_at_the_acceptance_word_limit(rows, mode, path):
    """Chains of at most 32 rows end with one done/accept word per request,
    longer ones with the walk over the rows' decisions: at 31, 32 and 33 rows
    the result equals the oracle's window on the GPU's own logits, with drafts
    that agree with the argmax for a long prefix so that the acceptance walks
    deep."""
    H, V = 64, 5000
    n = rows - 1
    rng = np.random.default_rng(3100 + rows + 7 * path)
    W = synth.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * np.float32(0.3))
    A = rng.standard_normal((rows, H)).astype(np.float32)
    L64 = ov.project(W, A)
    am = [int(ov.target_pool(L64[r].astype(np.float32))[0][0]) for r in range(rows)]
    stop = n - 2 if rows % 2 else n                     # a late mismatch, or none
    tokens = np.array([am[j] if j != stop else (am[j] + 1) % V for j in range(n)], np.int32)
    q_ids = q_log = None
    if mode == "sampled_q":
        q_ids = rng.integers(0, V, (n, 8)).astype(np.int32)
        q_ids[:, 0] = tokens
        q_log = rng.standard_normal((n, 8)).astype(np.float32) + np.float32(4.0) * (
            np.arange(8) == 0).astype(np.float32)
    pol = ov.Policy() if mode == "greedy" else ov.Policy(temperature=0.3, top_k=0, top_p=0.99)
    for seed in range(3):
        win = run_window(dev_weight(W), A, tokens, pol, seed, 777, q_ids=q_ids, q_log=q_log,
                         path=path)
        g_logits = win["logits"].cpu().numpy()
        assert_logits_close(g_logits, L64)
        ref = ov.verify_window(g_logits, tokens, None, q_ids, q_log, (), pol, seed, 777)
        assert list(win["ids"][:win["n"]]) == ref.emitted and win["accept"] == ref.accept, seed
        if mode == "greedy":
            assert win["accept"] == min(stop, n)
