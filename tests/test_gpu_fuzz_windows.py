"""Seeded random windows against the oracle.  Each case draws its own shape,
projection path and policy: 1-33 rows as a chain or a random token tree,
vocabularies from 64 to 70001 (most not multiples of 32), hidden sizes from
64 to 520, greedy, sampled or penalised requests, drafts with their
re-scored candidates or as point masses.  Every window is checked stage-wise
as the full-size window tests check theirs (logits against the fp64 oracle;
the GPU sampler against the oracle on the same float32 logits, bit for bit;
the fused window against the GPU's own stages; the oracle end to end when
both sides' pools agree), so a fault that only some combination of shape,
path and policy reaches shows up here."""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verify_row_gb300 import binding as vb, synth
from gpu_common import require_gpu, dev, dev_weight, assert_logits_close, same_bits_f32
import test_gpu_window as tw

pytestmark = pytest.mark.gpu

PATHS = [vb.VR_PATH_AUTO, vb.VR_PATH_TC, vb.VR_PATH_TC_BATCH, vb.VR_PATH_FFMA]
VOCABS = [64, 100, 999, 4097, 12345, 32768, 70001]
HIDDENS = [64, 128, 200, 256, 520]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _policy(rng):
    kind = rng.choice(["greedy", "sampled", "penalised"], p=[0.3, 0.4, 0.3])
    if kind == "greedy":
        return ov.Policy()
    pol = dict(temperature=float(rng.choice([0.5, 0.7, 1.3])),
               top_k=int(rng.choice([-1, 0, 1, 5, 20, 64])),
               min_p=float(rng.choice([0.0, 0.05, 0.2])),
               top_p=float(rng.choice([1.0, 0.9, 0.5])))
    if kind == "penalised":
        pol.update(repeat=float(rng.choice([1.0, 1.1, 1.3])),
                   presence=float(rng.choice([0.0, 0.5, 1.5])),
                   frequency=float(rng.choice([0.0, 0.2])),
                   window=int(rng.choice([1, 8, 64, 200])))
    return ov.Policy(**pol)


def _case(seed):
    """Inputs of one random window, drawn from the case's seed."""
    rng = np.random.default_rng(10_000 + seed)
    V, H = int(rng.choice(VOCABS)), int(rng.choice(HIDDENS))
    k = int(rng.integers(0, 33))
    path = int(rng.choice(PATHS))
    pol = _policy(rng)
    W = synth.weights(V, H, seed=20_000 + seed)
    A = synth.activations(k + 1, H, 30_000 + seed)
    L64 = ov.project(W, A)
    pools = [ov.target_pool(L64[r].astype(np.float32)) for r in range(k + 1)]
    tree = k >= 2 and rng.random() < 0.3
    parent = q_ids = q_log = None
    if tree:
        parent = np.array([int(rng.integers(-1, j)) for j in range(k)], np.int32)
        # a node's token from the top of the row that scores it (its parent's
        # row; the root row for children of the root), so that some agree
        tokens = np.array([int(pools[p + 1][0][int(rng.integers(0, min(4, len(pools[p + 1][0]))))])
                           for p in parent], np.int32)
    elif k and pol.temperature > 0 and rng.random() < 0.6:
        ids = np.stack([pools[r][0][:32] for r in range(k)])      # every vocabulary has >= 64 ids
        vals = np.stack([pools[r][1][:32] for r in range(k)])
        q_ids, q_log = synth.draft_candidates(ids, vals, seed=seed)
        slot = synth.draft_choice(q_log, 0.7, seed=seed + 1)
        tokens = q_ids[np.arange(k), slot].astype(np.int32)
    else:
        tokens = np.array([int(pools[r][0][int(rng.integers(0, min(3, len(pools[r][0]))))])
                           for r in range(k)], np.int32)
    hist = synth.zipf_history(int(rng.choice([0, 10, 500])), V, seed=seed) \
        if pol.window > 0 else np.zeros(0, np.int32)
    return dict(W=W, A=A, L64=L64, tokens=tokens, parent=parent, q_ids=q_ids, q_log=q_log,
                hist=hist, pol=pol, seed=int(rng.integers(0, 2**63)),
                position=int(rng.integers(0, 10**6)), path=path)


@pytest.mark.parametrize("seed", range(200))
def test_random_window(seed):
    c = _case(seed)
    win = tw.run_window(dev_weight(c["W"]), c["A"], c["tokens"], c["pol"], c["seed"],
                        c["position"], parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"],
                        hist=c["hist"], path=c["path"])
    tw.check_window(win, c["L64"], c["tokens"], c["pol"], c["seed"], c["position"],
                    parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"], hist=c["hist"])
    assert 1 <= win["n"] <= len(c["tokens"]) + 1


def _batched_case(seed):
    """One random batched call: 1-24 requests of 1-9 rows (chains and random
    trees), each with its own policy, seed, position, drafts and history,
    on one random projection shape and path."""
    rng = np.random.default_rng(50_000 + seed)
    V, H = int(rng.choice(VOCABS)), int(rng.choice(HIDDENS))
    path = int(rng.choice(PATHS))
    n_req = int(rng.integers(1, 25))
    ks = [int(rng.integers(0, 9)) for _ in range(n_req)]
    R = sum(k + 1 for k in ks)
    W = synth.weights(V, H, seed=60_000 + seed)
    A = synth.activations(R, H, 70_000 + seed)
    L64 = ov.project(W, A)
    specs, r0 = [], 0
    for b, k in enumerate(ks):
        pol = _policy(rng)
        pools = [ov.target_pool(L64[r0 + r].astype(np.float32)) for r in range(k + 1)]
        parent = q_ids = q_log = None
        if k >= 2 and rng.random() < 0.3:
            parent = np.array([int(rng.integers(-1, j)) for j in range(k)], np.int32)
            tokens = np.array([int(pools[p + 1][0][int(rng.integers(0, 4))]) for p in parent],
                              np.int32)
        elif k and pol.temperature > 0 and rng.random() < 0.5:
            ids = np.stack([pools[r][0][:32] for r in range(k)])
            vals = np.stack([pools[r][1][:32] for r in range(k)])
            q_ids, q_log = synth.draft_candidates(ids, vals, seed=seed * 100 + b)
            tokens = q_ids[np.arange(k), synth.draft_choice(q_log, 0.7, seed=seed * 100 + b + 1)]
            tokens = tokens.astype(np.int32)
        else:
            tokens = np.array([int(pools[r][0][int(rng.integers(0, 3))]) for r in range(k)],
                              np.int32)
        hist = (synth.zipf_history(int(rng.choice([5, 300])), V, seed=seed * 100 + b)
                if ov.penalties_active(pol) else None)
        specs.append(dict(rows=list(range(r0, r0 + k + 1)), tokens=tokens, parent=parent,
                          q_ids=q_ids, q_log=q_log, hist=hist, pol=pol,
                          seed=int(rng.integers(0, 2**63)), position=int(rng.integers(0, 10**6))))
        r0 += k + 1
    return dict(W=W, A=A, L64=L64, R=R, H=H, V=V, path=path, specs=specs)


@pytest.mark.parametrize("seed", range(40))
def test_random_batched_call(seed):
    """Every request of a random batched call equals the oracle's window on
    the GPU's own logits rows (penalised rows, pools, emitted ids and accept
    counts bit for bit), and the logits match the fp64 oracle."""
    c = _batched_case(seed)
    R, H, V = c["R"], c["H"], c["V"]
    reqs, keep = [], []
    for s in c["specs"]:
        k = len(s["tokens"])
        t = dict(tok=dev(s["tokens"]) if k else None,
                 par=None if s["parent"] is None else dev(s["parent"]),
                 q=None if s["q_ids"] is None else dev(s["q_ids"]),
                 ql=None if s["q_log"] is None else dev(s["q_log"]),
                 h=None if s["hist"] is None else dev(s["hist"]),
                 out=torch.full((k + 1,), -7, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                 n=torch.zeros(1, dtype=torch.int32, device="cuda"))
        keep.append(t)
        reqs.append(vb.make_request(k, t["tok"], tw.bpol(s["pol"]), s["seed"], s["position"],
                                    t["out"], t["acc"], t["n"], parent=t["par"], q_ids=t["q"],
                                    q_logits=t["ql"], hist=t["h"]))
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(logits)
    ws = vb.workspace(R, H, V)
    vb.verify_window_batched(dev_weight(c["W"]), dev(c["A"]), reqs, logits, ws, pen_logits=pen,
                             path=c["path"])
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.window_pools(ws, R, H, V, ids, vals)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    g_logits = logits.cpu().numpy()
    assert_logits_close(g_logits, c["L64"])
    ids, vals, g_pen = ids.cpu().numpy(), vals.cpu().numpy(), pen.cpu().numpy()
    refs = ov.verify_batched(g_logits, [dict(tokens=s["tokens"], parent=s["parent"],
                                             q_ids=s["q_ids"], q_logits=s["q_log"],
                                             hist=() if s["hist"] is None else s["hist"],
                                             pol=s["pol"], seed=s["seed"],
                                             position=s["position"]) for s in c["specs"]])
    for b, (s, ref) in enumerate(zip(c["specs"], refs)):
        active = ov.penalties_active(s["pol"])
        rows = g_pen[s["rows"]] if active else g_logits[s["rows"]]
        if active:
            assert same_bits_f32(rows, ref.pen_logits), b
        for i, r in enumerate(s["rows"]):
            want_ids, want_vals = ov.target_pool(rows[i])
            n = 1 if s["pol"].temperature == 0.0 else len(want_ids)
            assert np.array_equal(ids[r, :n], want_ids[:n]), (b, i)
            assert same_bits_f32(vals[r, :n], want_vals[:n]), (b, i)
        n_em = int(keep[b]["n"].item())
        assert list(keep[b]["out"].cpu().numpy()[:n_em]) == ref.emitted, b
        assert int(keep[b]["acc"].item()) == ref.accept, b


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("seed", range(0, 200, 10))
def test_random_host_window(seed, pinned):
    """The host-buffer entry point on a random window (the shapes of
    test_random_window): pinned inputs read by the staging kernel, or pageable
    ones copied, give the device entry point's result and logits bit for
    bit."""
    c = _case(seed)
    wd = dev_weight(c["W"])
    win = tw.run_window(wd, c["A"], c["tokens"], c["pol"], c["seed"], c["position"],
                        parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"], hist=c["hist"],
                        path=c["path"], separate_pen=False)
    if pinned:
        host = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    else:
        host = lambda x: torch.from_numpy(np.ascontiguousarray(x).copy())
    opt = lambda x: None if x is None or len(x) == 0 else host(x)
    R, H = c["A"].shape
    V = c["W"].shape[0]
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    out = host(np.full(R, -7, np.int32))
    ws = vb.workspace(R, H, V)
    acc, n = vb.verify_window_host(wd, host(c["A"]), opt(c["tokens"]), tw.bpol(c["pol"]),
                                   c["seed"], c["position"], logits, out, ws,
                                   parent_h=opt(c["parent"]), q_ids_h=opt(c["q_ids"]),
                                   q_logits_h=opt(c["q_log"]), hist_h=opt(c["hist"]),
                                   path=c["path"])
    assert (acc, n) == (win["accept"], win["n"])
    assert list(out.numpy()[:n]) == list(win["ids"][:n])
    assert torch.equal(logits.view(torch.int32), win["logits"].view(torch.int32))


def test_random_windows_share_one_workspace():
    """Thirty random windows of different shapes and paths run one after
    another through one workspace sized for the largest (as a server keeps
    one): each gives what it gives on a fresh workspace, so no call depends
    on what an earlier call of another shape left behind (the control region
    is left zeroed, and every other region is written before it is read)."""
    cases = [_case(seed) for seed in range(300, 330)]
    Rm = max(c["A"].shape[0] for c in cases)
    Hm = max(c["A"].shape[1] for c in cases)
    Vm = max(c["W"].shape[0] for c in cases)
    shared = vb.workspace(Rm, Hm, Vm)
    for i, c in enumerate(cases):
        wd = dev_weight(c["W"])
        fresh = tw.run_window(wd, c["A"], c["tokens"], c["pol"], c["seed"], c["position"],
                              parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"],
                              hist=c["hist"], path=c["path"], separate_pen=False)
        R, H = c["A"].shape
        V = c["W"].shape[0]
        logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
        out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        ne = torch.zeros(1, dtype=torch.int32, device="cuda")
        opt = lambda x: None if x is None or len(x) == 0 else dev(x)
        vb.verify_window(wd, dev(c["A"]), opt(c["tokens"]), tw.bpol(c["pol"]), c["seed"],
                         c["position"], logits, out, acc, ne, shared, parent=opt(c["parent"]),
                         q_ids=opt(c["q_ids"]), q_logits=opt(c["q_log"]), hist=opt(c["hist"]),
                         path=c["path"])
        torch.cuda.synchronize()
        assert vb.device_status(shared) == 0, i
        n = int(ne.item())
        assert (n, int(acc.item())) == (fresh["n"], fresh["accept"]), i
        assert list(out.cpu().numpy()[:n]) == list(fresh["ids"][:n]), i
        assert torch.equal(logits.view(torch.int32), fresh["logits"].view(torch.int32)), i


def test_random_windows_on_concurrent_streams():
    """Pairs of random windows enqueued on two streams at once, each with its
    own buffers and workspace, give what they give alone: the library keeps
    no state between calls outside the workspace it is handed."""
    opt = lambda x: None if x is None or len(x) == 0 else dev(x)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for p in range(8):
        cs = [_case(400 + 2 * p), _case(401 + 2 * p)]
        alone, bufs = [], []
        for c in cs:
            wd = dev_weight(c["W"])
            alone.append(tw.run_window(wd, c["A"], c["tokens"], c["pol"], c["seed"], c["position"],
                                       parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"],
                                       hist=c["hist"], path=c["path"], separate_pen=False))
            R, H = c["A"].shape
            V = c["W"].shape[0]
            bufs.append(dict(wd=wd, a=dev(c["A"]), tok=opt(c["tokens"]), par=opt(c["parent"]),
                             q=opt(c["q_ids"]), ql=opt(c["q_log"]), h=opt(c["hist"]),
                             lg=torch.empty((R, V), dtype=torch.float32, device="cuda"),
                             out=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                             acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                             n=torch.zeros(1, dtype=torch.int32, device="cuda"),
                             ws=vb.workspace(R, H, V)))
        torch.cuda.synchronize()
        for c, b, s in zip(cs, bufs, streams):
            vb.verify_window(b["wd"], b["a"], b["tok"], tw.bpol(c["pol"]), c["seed"], c["position"],
                             b["lg"], b["out"], b["acc"], b["n"], b["ws"], parent=b["par"],
                             q_ids=b["q"], q_logits=b["ql"], hist=b["h"], path=c["path"],
                             stream=s)
        torch.cuda.synchronize()
        for i, (b, w) in enumerate(zip(bufs, alone)):
            n = int(b["n"].item())
            assert vb.device_status(b["ws"]) == 0, (p, i)
            assert (n, int(b["acc"].item())) == (w["n"], w["accept"]), (p, i)
            assert list(b["out"].cpu().numpy()[:n]) == list(w["ids"][:n]), (p, i)
            assert torch.equal(b["lg"].view(torch.int32), w["logits"].view(torch.int32)), (p, i)


def test_random_windows_captured_in_a_cuda_graph():
    """Six random windows captured into one CUDA graph (each with its own
    buffers and workspace) and replayed twice give their eager results: a
    window enqueues kernels only (no host work, no copy), so it can be
    captured."""
    opt = lambda x: None if x is None or len(x) == 0 else dev(x)
    cases = [_case(s) for s in range(500, 506)]
    eager, bufs = [], []
    for c in cases:
        wd = dev_weight(c["W"])
        eager.append(tw.run_window(wd, c["A"], c["tokens"], c["pol"], c["seed"], c["position"],
                                   parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"],
                                   hist=c["hist"], path=c["path"], separate_pen=False))
        R, H = c["A"].shape
        V = c["W"].shape[0]
        bufs.append(dict(wd=wd, a=dev(c["A"]), tok=opt(c["tokens"]), par=opt(c["parent"]),
                         q=opt(c["q_ids"]), ql=opt(c["q_log"]), h=opt(c["hist"]),
                         lg=torch.empty((R, V), dtype=torch.float32, device="cuda"),
                         out=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                         acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                         n=torch.zeros(1, dtype=torch.int32, device="cuda"),
                         ws=vb.workspace(R, H, V)))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c, b in zip(cases, bufs):
            vb.verify_window(b["wd"], b["a"], b["tok"], tw.bpol(c["pol"]), c["seed"],
                             c["position"], b["lg"], b["out"], b["acc"], b["n"], b["ws"],
                             parent=b["par"], q_ids=b["q"], q_logits=b["ql"], hist=b["h"],
                             path=c["path"])
    for rep in range(2):
        for b in bufs:
            b["out"].fill_(-7)
            b["lg"].fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        for i, (b, w) in enumerate(zip(bufs, eager)):
            n = int(b["n"].item())
            assert vb.device_status(b["ws"]) == 0, (rep, i)
            assert (n, int(b["acc"].item())) == (w["n"], w["accept"]), (rep, i)
            assert list(b["out"].cpu().numpy()[:n]) == list(w["ids"][:n]), (rep, i)
            assert torch.equal(b["lg"].view(torch.int32), w["logits"].view(torch.int32)), (rep, i)


def test_random_batched_call_captured_in_a_cuda_graph():
    """A random batched call captured into a CUDA graph and replayed gives its
    eager result (the request table is captured with the call)."""
    c = _batched_case(7)
    R, H, V = c["R"], c["H"], c["V"]
    wd, a = dev_weight(c["W"]), dev(c["A"])

    def requests():
        reqs, keep = [], []
        for s in c["specs"]:
            k = len(s["tokens"])
            t = dict(tok=dev(s["tokens"]) if k else None,
                     par=None if s["parent"] is None else dev(s["parent"]),
                     q=None if s["q_ids"] is None else dev(s["q_ids"]),
                     ql=None if s["q_log"] is None else dev(s["q_log"]),
                     h=None if s["hist"] is None else dev(s["hist"]),
                     out=torch.full((k + 1,), -7, dtype=torch.int32, device="cuda"),
                     acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                     n=torch.zeros(1, dtype=torch.int32, device="cuda"))
            keep.append(t)
            reqs.append(vb.make_request(k, t["tok"], tw.bpol(s["pol"]), s["seed"], s["position"],
                                        t["out"], t["acc"], t["n"], parent=t["par"], q_ids=t["q"],
                                        q_logits=t["ql"], hist=t["h"]))
        return reqs, keep

    def outputs(keep):
        return [(int(t["n"].item()), int(t["acc"].item()),
                 list(t["out"].cpu().numpy()[:int(t["n"].item())])) for t in keep]

    lg = torch.empty((R, V), dtype=torch.float32, device="cuda")
    ws = vb.workspace(R, H, V)
    reqs, keep = requests()
    vb.verify_window_batched(wd, a, reqs, lg, ws, path=c["path"])
    torch.cuda.synchronize()
    want, want_lg = outputs(keep), lg.clone()
    reqs2, keep2 = requests()
    lg2 = torch.empty_like(lg)
    ws2 = vb.workspace(R, H, V)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vb.verify_window_batched(wd, a, reqs2, lg2, ws2, path=c["path"])
    for rep in range(2):
        for t in keep2:
            t["out"].fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert vb.device_status(ws2) == 0
        assert outputs(keep2) == want, rep
        assert torch.equal(lg2.view(torch.int32), want_lg.view(torch.int32)), rep


def test_random_async_host_windows_captured_in_a_cuda_graph():
    """Four random windows through the pipelined host-buffer entry point
    (pinned inputs and [accept, n, ids] outputs) captured into a CUDA graph:
    each replay reads the pinned inputs and writes the pinned outputs, which
    equal the device entry point's results."""
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    opt = lambda x: None if x is None or len(x) == 0 else pin(x)
    cases = [_case(s) for s in range(600, 604)]
    want, bufs = [], []
    for c in cases:
        wd = dev_weight(c["W"])
        w = tw.run_window(wd, c["A"], c["tokens"], c["pol"], c["seed"], c["position"],
                          parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"], hist=c["hist"],
                          path=c["path"], separate_pen=False)
        want.append((w["accept"], w["n"], list(w["ids"][:w["n"]])))
        R, H = c["A"].shape
        V = c["W"].shape[0]
        bufs.append(dict(wd=wd, a=pin(c["A"]), tok=opt(c["tokens"]), par=opt(c["parent"]),
                         q=opt(c["q_ids"]), ql=opt(c["q_log"]), h=opt(c["hist"]),
                         lg=torch.empty((R, V), dtype=torch.float32, device="cuda"),
                         out=torch.full((R + 2,), -7, dtype=torch.int32).pin_memory(),
                         ws=vb.workspace(R, H, V)))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c, b in zip(cases, bufs):
            vb.verify_window_host_async(b["wd"], b["a"], b["tok"], tw.bpol(c["pol"]), c["seed"],
                                        c["position"], b["lg"], b["out"], b["ws"],
                                        parent_h=b["par"], q_ids_h=b["q"], q_logits_h=b["ql"],
                                        hist_h=b["h"], path=c["path"])
    for rep in range(2):
        for b in bufs:
            b["out"].fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for i, (b, w) in enumerate(zip(bufs, want)):
            o = b["out"].numpy()
            acc, n = int(o[0]), int(o[1])
            assert (acc, n, list(o[2:2 + n])) == w, (rep, i)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("what", ["token", "parent", "qid"])
def test_fused_window_flags_invalid_device_data(path, what):
    """Device data the host cannot check (a draft token past the vocabulary,
    a parent array that is not topological, a candidate id past the
    vocabulary) makes the fused window emit nothing and set the status word,
    on every path and with penalties active (the history walk meets the bad
    parent first); the next good window on the same workspace is unaffected."""
    V, H, k = 5000, 64, 3
    W = synth.weights(V, H, seed=77)
    A = synth.activations(k + 1, H, 78)
    wd = dev_weight(W)
    pol = ov.Policy(temperature=0.8, top_k=20, presence=0.5, window=16)
    tokens = np.array([5, 6, 7], np.int32)
    parent = q_ids = q_log = None
    if what == "token":
        tokens[1] = V + 3
    elif what == "parent":
        parent = np.array([-1, 2, 1], np.int32)          # node 1 names a later node
    else:
        q_ids = np.tile(np.arange(8, dtype=np.int32), (k, 1))
        q_ids[0, 0] = tokens[0]
        q_ids[2, 5] = V + 100
        q_log = np.zeros((k, 8), np.float32)
    hist = np.arange(20, dtype=np.int32)
    ws = vb.workspace(k + 1, H, V)
    lg = torch.empty((k + 1, V), dtype=torch.float32, device="cuda")
    out = torch.full((k + 1,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ne = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    opt = lambda x: None if x is None else dev(x)
    vb.verify_window(wd, dev(A), dev(tokens), tw.bpol(pol), 1, 2, lg, out, acc, ne, ws,
                     parent=opt(parent), q_ids=opt(q_ids), q_logits=opt(q_log), hist=dev(hist),
                     path=path)
    torch.cuda.synchronize()
    st = vb.device_status(ws)
    flag = {"token": vb.VR_DEV_BAD_TOKEN, "parent": vb.VR_DEV_BAD_PARENT,
            "qid": vb.VR_DEV_BAD_QID}[what]
    assert st & flag, st
    assert int(ne.item()) == 0 and int(acc.item()) == 0
    # the status word was read and cleared: a good window runs clean
    good = np.array([5, 6, 7], np.int32)
    vb.verify_window(wd, dev(A), dev(good), tw.bpol(pol), 1, 2, lg, out, acc, ne, ws,
                     hist=dev(hist), path=path)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    assert 1 <= int(ne.item()) <= k + 1


@pytest.mark.parametrize("seed", range(6))
def test_batched_call_isolates_a_request_with_invalid_data(seed):
    """One request of a random batched call carries a draft token past the
    vocabulary: that request emits nothing and the status word is set, while
    every other request still equals the oracle's window on the GPU's own
    logits."""
    c = _batched_case(100 + seed)
    specs = c["specs"]
    bad = next((b for b, s in enumerate(specs) if len(s["tokens"])), None)
    if bad is None:
        pytest.skip("no request with drafts in this draw")
    R, H, V = c["R"], c["H"], c["V"]
    reqs, keep = [], []
    for b, s in enumerate(specs):
        k = len(s["tokens"])
        tokens = s["tokens"].copy()
        if b == bad:
            tokens[k - 1] = V + 7
        t = dict(tok=dev(tokens) if k else None,
                 par=None if s["parent"] is None else dev(s["parent"]),
                 q=None if s["q_ids"] is None else dev(s["q_ids"]),
                 ql=None if s["q_log"] is None else dev(s["q_log"]),
                 h=None if s["hist"] is None else dev(s["hist"]),
                 out=torch.full((k + 1,), -7, dtype=torch.int32, device="cuda"),
                 acc=torch.zeros(1, dtype=torch.int32, device="cuda"),
                 n=torch.full((1,), -1, dtype=torch.int32, device="cuda"))
        keep.append(t)
        reqs.append(vb.make_request(k, t["tok"], tw.bpol(s["pol"]), s["seed"], s["position"],
                                    t["out"], t["acc"], t["n"], parent=t["par"], q_ids=t["q"],
                                    q_logits=t["ql"], hist=t["h"]))
    lg = torch.empty((R, V), dtype=torch.float32, device="cuda")
    pen = torch.empty_like(lg)
    ws = vb.workspace(R, H, V)
    vb.verify_window_batched(dev_weight(c["W"]), dev(c["A"]), reqs, lg, ws, pen_logits=pen,
                             path=c["path"])
    torch.cuda.synchronize()
    assert vb.device_status(ws) & vb.VR_DEV_BAD_TOKEN
    g_logits = lg.cpu().numpy()
    refs = ov.verify_batched(g_logits, [dict(tokens=s["tokens"], parent=s["parent"],
                                             q_ids=s["q_ids"], q_logits=s["q_log"],
                                             hist=() if s["hist"] is None else s["hist"],
                                             pol=s["pol"], seed=s["seed"],
                                             position=s["position"]) for s in specs])
    for b, ref in enumerate(refs):
        n_em = int(keep[b]["n"].item())
        if b == bad:
            assert n_em == 0 and int(keep[b]["acc"].item()) == 0
            continue
        assert list(keep[b]["out"].cpu().numpy()[:n_em]) == ref.emitted, b
        assert int(keep[b]["acc"].item()) == ref.accept, b


@pytest.mark.parametrize("H,path", [(16384, p) for p in PATHS] +
                         [(65536, vb.VR_PATH_TC), (32768, vb.VR_PATH_TC_BATCH)])
def test_wide_hidden_windows(H, path):
    """Hidden sizes far past the test workloads' (256 K blocks at 16384, the
    ABI's maximum 65536 on the default path): a sampled 5-row chain's window
    against the oracle stage by stage.  The tensor-core paths' logit error
    grows about linearly with hidden (fp32 accumulation over thousands of
    MMA steps); the batched path, whose two planes share one accumulator,
    stays within the tolerance up to 32768 (0.56 of the bound there, 1.35 at
    65536, measured), the default path up to 65536 (0.67)."""
    V, k = 1000, 4
    W = synth.weights(V, H, seed=H + 1)
    A = synth.activations(k + 1, H, H + 2)
    L64 = ov.project(W, A)
    pools = [ov.target_pool(L64[r].astype(np.float32)) for r in range(k + 1)]
    tokens = np.array([int(pools[r][0][r % 3]) for r in range(k)], np.int32)
    pol = ov.Policy(temperature=0.7, top_k=20, min_p=0.05, top_p=0.95)
    win = tw.run_window(dev_weight(W), A, tokens, pol, 5, 6, path=path)
    tw.check_window(win, L64, tokens, pol, 5, 6)


def test_cuda_core_path_rejects_hidden_past_its_shared_memory():
    """The CUDA-core projection keeps a pass's activations in shared memory
    (4 * hidden bytes per row): at hidden 65536 not even one row fits, and
    the call says so instead of running."""
    V, H = 64, 65536
    W = synth.weights(V, H, seed=3)
    lg = torch.empty((1, V), dtype=torch.float32, device="cuda")
    with pytest.raises(vb.VerifyRowError) as e:
        vb.verify_project(dev_weight(W), dev(synth.activations(1, H, 4)), lg,
                          vb.workspace(1, H, V), path=vb.VR_PATH_FFMA)
    assert e.value.status == vb.VR_ERR_UNSUPPORTED


def test_host_threads_run_windows_at_once():
    """Four host threads, each on its own stream with its own buffers and
    workspaces, run random windows through the device and the host-buffer
    entry points at the same time (the foreign calls release the
    interpreter's lock): every result equals the one computed alone."""
    import threading
    cases = [_case(s) for s in range(700, 716)]
    alone = []
    for c in cases:
        w = tw.run_window(dev_weight(c["W"]), c["A"], c["tokens"], c["pol"], c["seed"],
                          c["position"], parent=c["parent"], q_ids=c["q_ids"], q_log=c["q_log"],
                          hist=c["hist"], path=c["path"], separate_pen=False)
        alone.append((w["accept"], w["n"], list(w["ids"][:w["n"]])))
    results, errors = {}, []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            opt = lambda x: None if x is None or len(x) == 0 else torch.from_numpy(
                np.ascontiguousarray(x)).pin_memory()
            with torch.cuda.stream(stream):
                for i in range(t, len(cases), 4):
                    c = cases[i]
                    R, H = c["A"].shape
                    V = c["W"].shape[0]
                    wd = dev_weight(c["W"])
                    lg = torch.empty((R, V), dtype=torch.float32, device="cuda")
                    out = torch.full((R,), -7, dtype=torch.int32).pin_memory()
                    ws = vb.workspace(R, H, V, stream=stream)
                    acc, n = vb.verify_window_host(
                        wd, opt(c["A"]), opt(c["tokens"]), tw.bpol(c["pol"]), c["seed"],
                        c["position"], lg, out, ws, parent_h=opt(c["parent"]),
                        q_ids_h=opt(c["q_ids"]), q_logits_h=opt(c["q_log"]),
                        hist_h=opt(c["hist"]), path=c["path"], stream=stream)
                    results[i] = (acc, n, list(out.numpy()[:n]))
        except Exception as e:                  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i, want in enumerate(alone):
        assert results[i] == want, i
