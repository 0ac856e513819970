"""Benchmark of the verify step on one GB300 (or N replicas).

Workload: the sampled chain -- hidden 4096, vocab 151936, three drafts
and so four rows to verify, bf16 LM-head weights N(0, 0.02), fp32 activations N(0, 1),
draft q over 8 candidates drawn from the target top-32 with logit = target
logit + N(0, 1); temperature 0.7, top-k absent (20), min-p 0.05, top-p 0.95,
no penalties.  One step = one fused verify window (projection, pool,
policy, acceptance).  256 distinct windows (seeds 0..255) are resident in
HBM and cycled; the 1.24 GB weight stream is larger than L2, so no step
reuses another's weights from cache.

Prints one JSON line (see the repository's benchmark contract).  With
--impl reference it times the CPU oracle instead (bounded sample).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

V, H, K_DRAFTS = 151936, 4096, 3
ROWS = K_DRAFTS + 1
N_WINDOWS = 256
WEIGHT_BYTES = V * H * 2
METRIC = "verify windows/s (hidden 4096, V=151936, k+1 rows); HBM GB/s vs 8 TB/s peak"
WORKLOAD = "sampled chain: hidden 4096, vocab 151936, k=3 (4 rows), T 0.7, top-k 20, min-p 0.05, top-p 0.95"
POLICY = dict(temperature=0.7, top_k=-1, min_p=0.05, top_p=0.95)
# windows behind each breakdown of the line (stages, latency, other
# workloads, host-buffer paths); fixed so that a short --steps run still
# reports figures over large samples
STAGE_SAMPLES = 2000
LATENCY_SAMPLES = 500
EXTRA_SAMPLES = 1000
E2E_SAMPLES = 2000
E2E_SYNC_SAMPLES = 1000
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the penalised-chain, tree and batched workloads")
    p.add_argument("--mode", choices=["full", "window", "project", "project_batched", "batched",
                                      "topk", "penalize"],
                   default="full",
                   help="window: only the timed windows (for a profiler's launch list); "
                        "project: only the projection of one window (for a kernel capture); "
                        "project_batched: only the 256-row batched projection at hidden 5120; "
                        "topk: only the batched top-K (15 x 248320, K 16); "
                        "penalize: only the penalty entry point on the penalised chain's rows")
    p.add_argument("--path", choices=["tc", "ffma"], default="tc",
                   help="projection path of --mode project")
    p.add_argument("--rows", type=int, default=ROWS, help="rows of --mode project")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def traffic_record(kernel):
    """Per-launch DRAM bytes from a committed ncu summary, valid only while
    the kernel source is unchanged since it was taken."""
    path = os.path.join(HERE, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    src = os.path.join(HERE, rec["source"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec["bytes_per_launch"] if digest == rec["sha256"] else None


class ClockSampler:
    """nvidia-smi clock and throttle samples taken while the timed region runs."""

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_windows(torch, vb, synth, wd, dev):
    """N_WINDOWS resident windows: activations, draft candidates and drafts.
    The target top-32 that the draft recipe needs is taken from a cuBLAS
    bf16 product (input preparation only, outside any timed region)."""
    acts = np.stack([synth.activations(ROWS, H, s) for s in range(N_WINDOWS)])
    A = torch.from_numpy(acts).to(dev)
    w_bf16 = wd.view(torch.bfloat16)
    top_ids, top_vals = [], []
    for s in range(0, N_WINDOWS, 32):
        a = A[s:s + 32, :K_DRAFTS].reshape(-1, H).to(torch.bfloat16)
        lg = (a @ w_bf16.T).float()
        v, i = torch.topk(lg, 32, dim=1)
        top_ids.append(i.reshape(-1, K_DRAFTS, 32).cpu().numpy())
        top_vals.append(v.reshape(-1, K_DRAFTS, 32).cpu().numpy())
    top_ids = np.concatenate(top_ids)
    top_vals = np.concatenate(top_vals)
    q_ids, q_log, drafts = [], [], []
    for s in range(N_WINDOWS):
        qi, ql = synth.draft_candidates(top_ids[s], top_vals[s], seed=s)
        slot = synth.draft_choice(ql, POLICY["temperature"], seed=s + 1)
        q_ids.append(qi)
        q_log.append(ql)
        drafts.append(qi[np.arange(K_DRAFTS), slot].astype(np.int32))
    return dict(act_np=acts, act=A, q_ids_np=np.stack(q_ids), q_log_np=np.stack(q_log),
                drafts_np=np.stack(drafts), q_ids=torch.from_numpy(np.stack(q_ids)).to(dev),
                q_log=torch.from_numpy(np.stack(q_log)).to(dev),
                drafts=torch.from_numpy(np.stack(drafts)).to(dev))


def cpu_oracle_windows(W, win, n_windows, threads_note=True):
    """Time the oracle as it stands on n_windows full windows of the workload."""
    from oracle import verify as ov
    pol = ov.Policy(**POLICY)
    times = []
    for s in range(n_windows):
        t0 = time.perf_counter()
        L = ov.project(W, win["act_np"][s]).astype(np.float32)
        ov.verify_window(L, win["drafts_np"][s], None, win["q_ids_np"][s], win["q_log_np"][s], (),
                         pol, s, 4096)
        times.append(time.perf_counter() - t0)
    return times


def run_reference(args):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from speculative_decoding_verify_row_gb300 import synth
    W = synth.weights(V, H)
    win = {"act_np": np.stack([synth.activations(ROWS, H, s) for s in range(8)])}
    # the draft recipe needs the target top-32; the reference arm takes it
    # from the oracle's own projection of each window
    from oracle import verify as ov
    q_ids, q_log, drafts = [], [], []
    for s in range(8):
        L = ov.project(W, win["act_np"][s]).astype(np.float32)
        top = [ov.target_pool(L[r]) for r in range(K_DRAFTS)]
        qi, ql = synth.draft_candidates(np.stack([t[0][:32] for t in top]),
                                        np.stack([t[1][:32] for t in top]), seed=s)
        slot = synth.draft_choice(ql, POLICY["temperature"], seed=s + 1)
        q_ids.append(qi)
        q_log.append(ql)
        drafts.append(qi[np.arange(K_DRAFTS), slot].astype(np.int32))
    win.update(q_ids_np=np.stack(q_ids), q_log_np=np.stack(q_log), drafts_np=np.stack(drafts))
    warm = min(args.warmup, 1)
    steps = max(1, min(args.steps, 6))
    cpu_oracle_windows(W, win, warm)
    times = cpu_oracle_windows(W, win, steps)
    value = steps / sum(times)
    sample = (f"{steps} full oracle windows of the workload (fp64 projection of 4 x 151936 x 4096 "
              f"+ penalties/pool/policy/acceptance), {warm} warm-up")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "windows/s",
            "n_gpus": args.gpus, "steps": steps, "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": 1000.0 * sum(times) / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": "windows/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "windows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _event_time(torch, stream, fn, n):
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    for i in range(3):
        fn(i)
    t0.record(stream)
    for i in range(n):
        fn(i)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / 1000.0 / n


def batched_serving(torch, vb, synth, dev):
    """The batched-serving workload: 64 requests x k 3 (256 rows) at hidden
    5120; even requests greedy, odd ones T 0.8 / top-k 20 / top-p 0.9 /
    presence 1.5 over 2048-token Zipf histories (W 64)."""
    H5, nreq, k = 5120, 64, 3
    W5 = synth.weights(V, H5)
    wd5 = torch.from_numpy(W5.view(np.int16)).to(dev)
    del W5
    R = nreq * (k + 1)
    A = torch.from_numpy(synth.activations(R, H5, 500)).to(dev)
    rng = np.random.default_rng(500)
    keep, reqs = [], []
    for b in range(nreq):
        greedy = b % 2 == 0
        bpol = vb.Policy() if greedy else vb.Policy(temperature=0.8, top_k=20, top_p=0.9,
                                                     presence=1.5, window=64)
        qi = rng.integers(0, V, (k, 8)).astype(np.int32)
        ql = rng.standard_normal((k, 8)).astype(np.float32)
        t = dict(d=torch.from_numpy(qi[:, 0].copy()).to(dev), q=torch.from_numpy(qi).to(dev),
                 ql=torch.from_numpy(ql).to(dev),
                 h=torch.from_numpy(synth.zipf_history(2048, V, seed=1000 + b)).to(dev),
                 o=torch.empty(k + 1, dtype=torch.int32, device=dev),
                 a=torch.empty(1, dtype=torch.int32, device=dev),
                 n=torch.empty(1, dtype=torch.int32, device=dev))
        keep.append(t)
        reqs.append(vb.make_request(k, t["d"], bpol, b, 2048, t["o"], t["a"], t["n"], q_ids=t["q"],
                                    q_logits=t["ql"], hist=t["h"]))
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    return dict(H5=H5, nreq=nreq, R=R, wd5=wd5, A=A, reqs=reqs, keep=keep, lg=lg,
                pen=torch.empty_like(lg), ws=vb.workspace(R, H5, V, device=dev))


def extra_workloads(torch, vb, synth, wd, dev, stream, n_steps):
    """The other verify workloads on the same GPU: the penalised chain (k 8),
    the 3 x 8 token tree (greedy and sampled) and 64 batched requests at
    hidden 5120.  Per-window time of the fused call, events on the stream;
    inputs resident, 32 distinct windows cycled."""
    out = {}
    w_bf16 = wd.view(torch.bfloat16)
    nwin = 32

    def top32(a):                              # [R, H] -> cuBLAS bf16 top-32 (input prep)
        lg = (a.to(torch.bfloat16) @ w_bf16.T).float()
        v, i = torch.topk(lg, 32, dim=1)
        return i.cpu().numpy(), v.cpu().numpy()

    # penalised chain: k 8, W 64, repeat 1.1, presence 1.5, frequency 0.2, top-k 0
    k, R = 8, 9
    pol = vb.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95, repeat=1.1, presence=1.5,
                    frequency=0.2, window=64)
    wins = []
    for s in range(nwin):
        a = torch.from_numpy(synth.activations(R, H, 100 + s)).to(dev)
        ti, tv = top32(a[:k])
        qi, ql = synth.draft_candidates(ti, tv, seed=100 + s)
        slot = synth.draft_choice(ql, 0.7, seed=101 + s)
        wins.append(dict(a=a, q=torch.from_numpy(qi).to(dev), ql=torch.from_numpy(ql).to(dev),
                         d=torch.from_numpy(qi[np.arange(k), slot].astype(np.int32)).to(dev),
                         h=torch.from_numpy(synth.zipf_history(4096, V, seed=100 + s)).to(dev)))
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    pen = torch.empty_like(lg)
    o = torch.empty(R, dtype=torch.int32, device=dev)
    acc = torch.empty(1, dtype=torch.int32, device=dev)
    ne = torch.empty(1, dtype=torch.int32, device=dev)
    ws = vb.workspace(R, H, V, device=dev)

    def pen_window(i):
        w = wins[i % nwin]
        vb.verify_window(wd, w["a"], w["d"], pol, i, 4096, lg, o, acc, ne, ws, q_ids=w["q"],
                         q_logits=w["ql"], hist=w["h"], pen_logits=pen, stream=stream)
    t = _event_time(torch, stream, pen_window, n_steps)
    out["penalised_chain_k8"] = {"windows_per_s": 1.0 / t, "us_per_window": 1e6 * t, "rows": R}
    # the same windows through the stage entry points (projection, penalty
    # prepass, pool + policy + acceptance), events between the stages; the
    # fused call applies the penalties inside its row sampling kernel instead
    n_st = min(n_steps, 200)
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_st)]
    qpen = torch.empty((k, 8), dtype=torch.float32, device=dev)
    for i in range(n_st):
        w = wins[i % nwin]
        qpen.copy_(w["ql"])
        st_ev[i][0].record(stream)
        vb.verify_project(wd, w["a"], lg, ws, stream=stream)
        st_ev[i][1].record(stream)
        vb.verify_penalize(lg, w["d"], w["h"], pol, ws, q_ids=w["q"], q_logits=qpen, stream=stream)
        st_ev[i][2].record(stream)
        vb.verify_sample_accept(lg, w["d"], pol, i, 4096, o, acc, ne, ws, q_ids=w["q"],
                                q_logits=qpen, stream=stream)
        st_ev[i][3].record(stream)
    torch.cuda.synchronize()
    names = ("projection", "penalize", "pool_policy_accept")
    st_us = {nm: 1000.0 * statistics.fmean(e[j].elapsed_time(e[j + 1]) for e in st_ev)
             for j, nm in enumerate(names)}
    tot = sum(st_us.values())
    out["penalised_chain_k8"]["stages_us"] = st_us
    out["penalised_chain_k8"]["stages_pct"] = {nm: 100.0 * v / tot for nm, v in st_us.items()}

    # token tree: 3 branches x depth 8 (25 rows)
    parent = torch.from_numpy(synth.tree_parents(3, 8)).to(dev)
    R = 25
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    pen = torch.empty_like(lg)
    o = torch.empty(R, dtype=torch.int32, device=dev)
    ws = vb.workspace(R, H, V, device=dev)
    twins = []
    for s in range(nwin):
        a = torch.from_numpy(synth.activations(R, H, 200 + s)).to(dev)
        ti, _ = top32(a)
        toks = synth.tree_tokens(ti[:, 0], ti, seed=200 + s)
        twins.append(dict(a=a, t=torch.from_numpy(toks).to(dev),
                          h=torch.from_numpy(synth.zipf_history(2048, V, seed=200 + s)).to(dev)))
    for name, tpol in (("tree_3x8_greedy", vb.Policy()),
                       ("tree_3x8_sampled", vb.Policy(temperature=0.7, top_k=20, presence=1.5,
                                                      window=64))):
        def tree_window(i, tpol=tpol):
            w = twins[i % nwin]
            vb.verify_window(wd, w["a"], w["t"], tpol, i, 2048, lg, o, acc, ne, ws, parent=parent,
                             hist=w["h"], pen_logits=pen, stream=stream)
        t = _event_time(torch, stream, tree_window, n_steps)
        out[name] = {"windows_per_s": 1.0 / t, "us_per_window": 1e6 * t, "rows": R}
    del wins, twins, lg, pen, ws

    # batched serving: 64 requests x k 3 at hidden 5120
    bs = batched_serving(torch, vb, synth, dev)
    wd5, A, reqs, lg, pen, ws = bs["wd5"], bs["A"], bs["reqs"], bs["lg"], bs["pen"], bs["ws"]
    H5, nreq, R = bs["H5"], bs["nreq"], bs["R"]

    def batched(i):
        vb.verify_window_batched(wd5, A, reqs, lg, ws, pen_logits=pen, path=vb.VR_PATH_TC_BATCH,
                                 stream=stream)
    t = _event_time(torch, stream, batched, max(5, n_steps // 50))
    flops = 2.0 * R * H5 * V
    # the projection alone, for the tensor-pipe roofline (2 bf16 planes)
    tp = _event_time(torch, stream,
                     lambda i: vb.verify_project(wd5, A, lg, ws, path=vb.VR_PATH_TC_BATCH,
                                                 stream=stream), max(5, n_steps // 50))
    # the exact alternative: the same 256 rows through the three-plane path
    tx = _event_time(torch, stream,
                     lambda i: vb.verify_project(wd5, A, lg, ws, path=vb.VR_PATH_TC,
                                                 stream=stream), max(5, n_steps // 100))
    out["batched_64x4_h5120"] = {"windows_per_s": nreq / t, "us_per_call": 1e6 * t, "rows": R,
                                 "path": "tc_batch", "projection_us": 1e6 * tp,
                                 "algorithmic_tflops": flops / tp / 1e12,
                                 "executed_tflops": 2 * flops / tp / 1e12,
                                 "weight_gbs": V * H5 * 2 / tp / 1e9,
                                 "activations": "two exact bf16 planes: 16 significant bits of "
                                                "each fp32 activation (a lone window on the "
                                                "default path keeps all 24, so its logits' bits "
                                                "differ from the batched call's)",
                                 "exact_three_plane_projection_us": 1e6 * tx}
    del wd5
    out["topk_15x248320_k16"] = topk_workload(torch, vb, dev, stream, n_steps)
    return out


COST_ROWS = (1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 17, 21, 25)


def window_cost_model(torch, vb, synth, wd, dev, stream):
    """Window cost against rows, and what it implies for the draft depth
    ("Speculative decoding on RDNA" §05).  Sampled chain windows with k
    point-mass drafts (prompt-lookup style, no candidates) at 1..25 rows,
    events on the stream, 64 windows per row count over 8 distinct inputs;
    the library's cost fit ms = a + b (rows - 1) over those times; the
    break-even tokens per window (cost / one-row cost) and the depth the
    library's chooser picks for constant per-draft acceptance."""
    pol = vb.Policy(**POLICY)
    rows_ms = {}
    for R in COST_ROWS:
        k = R - 1
        acts = [torch.from_numpy(synth.activations(R, H, 7000 + 10 * R + j)).to(dev) for j in range(8)]
        rng = np.random.default_rng(R)
        drafts = [torch.from_numpy(rng.integers(0, V, k).astype(np.int32)).to(dev) if k else None
                  for _ in range(8)]
        lg = torch.empty((R, V), dtype=torch.float32, device=dev)
        o = torch.empty(R, dtype=torch.int32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        ne = torch.empty(1, dtype=torch.int32, device=dev)
        ws = vb.workspace(R, H, V, device=dev)

        def win(i):
            vb.verify_window(wd, acts[i % 8], drafts[i % 8], pol, i, 4096, lg, o, acc, ne, ws,
                             stream=stream)
        rows_ms[R] = 1000.0 * _event_time(torch, stream, win, 64)
    rows = list(rows_ms)
    a, b = vb.cost_fit(rows, [rows_ms[r] for r in rows])
    choose = {}
    for alpha in (0.3, 0.5, 0.7, 0.9):
        k, rate = vb.choose_depth([alpha] * 24, a, b)
        choose[str(alpha)] = {"k": k, "tokens_per_ms": rate}
    return {"window_us_by_rows": {str(r): round(1000.0 * t, 2) for r, t in rows_ms.items()},
            "fit_us": {"one_row": 1000.0 * a, "per_extra_row": 1000.0 * b},
            "break_even_tokens": {str(r): (a + b * (r - 1)) / a for r in (2, 3, 4, 9, 25)},
            "chosen_depth_kmax24": choose,
            "drafts": "point-mass (no candidates), T 0.7, top-k 20, min-p 0.05, top-p 0.95"}


TOPK_ROWS, TOPK_VOCAB, TOPK_K = 15, 248320, 16


def topk_inputs(torch, dev, n):
    """n distinct 15 x 248320 float rows with ties, NaN and -inf (seeded)."""
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    xs = []
    for i in range(n):
        x = torch.randn((TOPK_ROWS, TOPK_VOCAB), generator=g, device=dev)
        x = torch.round(x * 64) / 64                       # many exact ties
        m = torch.rand(x.shape, generator=g, device=dev)
        x[m < 0.01] = float("nan")
        x[(m >= 0.01) & (m < 0.02)] = float("-inf")
        xs.append(x)
    return xs


def topk_workload(torch, vb, dev, stream, n_steps):
    """The draft tuner's batched top-K: 15 rows x 248320, K 16.  16 distinct
    inputs (238 MB, above the L2) cycled.  One call is a single ~10 us
    launch, shorter than the Python binding's own per-call cost, so the 16
    calls are captured once in a CUDA graph and the graph is replayed; events
    on the stream.  Also reported: the same calls issued one by one from
    Python (host-bound)."""
    xs = topk_inputs(torch, dev, 16)
    ids = torch.empty((TOPK_ROWS, TOPK_K), dtype=torch.int32, device=dev)
    vals = torch.empty((TOPK_ROWS, TOPK_K), dtype=torch.float32, device=dev)
    ws = vb.workspace(TOPK_ROWS, 8, TOPK_VOCAB, device=dev)
    nbytes = TOPK_ROWS * TOPK_VOCAB * 4
    t_py = _event_time(torch, stream, lambda i: vb.topk(xs[i % 16], TOPK_K, ids, vals, ws,
                                                        stream=stream), max(200, n_steps // 10))
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(16):                      # warm-up outside the capture
            vb.topk(xs[i], TOPK_K, ids, vals, ws)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(16):
            vb.topk(xs[i], TOPK_K, ids, vals, ws)
    stream.wait_stream(side)
    n_rep = max(20, n_steps // 50)
    t_graph = _event_time(torch, stream, lambda i: g.replay(), n_rep) / 16
    return {"us_per_call": 1e6 * t_graph, "input_gbs": nbytes / t_graph / 1e9,
            "us_per_call_python_loop": 1e6 * t_py, "rows": TOPK_ROWS, "vocab": TOPK_VOCAB,
            "k": TOPK_K, "timing": "CUDA graph of 16 calls on 16 distinct inputs, replayed"}


def run_topk_only(torch, vb, dev, args):
    """Batched top-K (15 x 248320, K 16), warm-up + steps times."""
    xs = topk_inputs(torch, dev, 2)
    ids = torch.empty((TOPK_ROWS, TOPK_K), dtype=torch.int32, device=dev)
    vals = torch.empty((TOPK_ROWS, TOPK_K), dtype=torch.float32, device=dev)
    ws = vb.workspace(TOPK_ROWS, 8, TOPK_VOCAB, device=dev)
    for i in range(args.warmup):
        vb.topk(xs[i % 2], TOPK_K, ids, vals, ws)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.steps):
        vb.topk(xs[i % 2], TOPK_K, ids, vals, ws)
    torch.cuda.synchronize(dev)
    print(json.dumps({"mode": "topk", "steps": args.steps,
                      "us_per_call": 1e6 * (time.perf_counter() - t0) / max(1, args.steps)}))


def run_projection_only(torch, vb, synth, wd, dev, args):
    """The projection of one window (--rows rows, --path), warm-up + steps
    times."""
    R = args.rows
    path = vb.VR_PATH_FFMA if args.path == "ffma" else vb.VR_PATH_TC
    a = torch.from_numpy(synth.activations(R, H, 0)).to(dev)
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    ws = vb.workspace(R, H, V, device=dev)
    for _ in range(args.warmup):
        vb.verify_project(wd, a, lg, ws, path=path)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vb.verify_project(wd, a, lg, ws, path=path)
    torch.cuda.synchronize(dev)
    print(json.dumps({"mode": "project", "path": args.path, "rows": R, "steps": args.steps,
                      "us_per_call": 1e6 * (time.perf_counter() - t0) / max(1, args.steps)}))


def run_penalize_only(torch, vb, synth, wd, dev, args):
    """The penalty entry point on the penalised chain's rows (k 8, 9 rows,
    4096-token history, W 64, repeat 1.1, presence 1.5, frequency 0.2,
    draft candidates penalised too), warm-up + steps times on the logits of
    one projection (each call penalises the rows again: the same work)."""
    k, R = 8, 9
    pol = vb.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95, repeat=1.1, presence=1.5,
                    frequency=0.2, window=64)
    rng = np.random.default_rng(100)
    a = torch.from_numpy(synth.activations(R, H, 100)).to(dev)
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    ws = vb.workspace(R, H, V, device=dev)
    vb.verify_project(wd, a, lg, ws)
    d = torch.from_numpy(rng.integers(0, V, k).astype(np.int32)).to(dev)
    q = torch.from_numpy(rng.integers(0, V, (k, 8)).astype(np.int32)).to(dev)
    ql = torch.from_numpy(rng.standard_normal((k, 8)).astype(np.float32)).to(dev)
    h = torch.from_numpy(synth.zipf_history(4096, V, seed=100)).to(dev)
    for _ in range(args.warmup):
        vb.verify_penalize(lg, d, h, pol, ws, q_ids=q, q_logits=ql)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vb.verify_penalize(lg, d, h, pol, ws, q_ids=q, q_logits=ql)
    torch.cuda.synchronize(dev)
    print(json.dumps({"mode": "penalize", "rows": R, "steps": args.steps,
                      "us_per_call": 1e6 * (time.perf_counter() - t0) / max(1, args.steps)}))


def run_batched_only(torch, vb, synth, dev, args):
    """The batched-serving call (64 requests x 4 rows, hidden 5120, batch
    tensor-core path): warm-up, then steps timed with events."""
    bs = batched_serving(torch, vb, synth, dev)
    stream = torch.cuda.current_stream(dev)

    def call(i):
        vb.verify_window_batched(bs["wd5"], bs["A"], bs["reqs"], bs["lg"], bs["ws"],
                                 pen_logits=bs["pen"], path=vb.VR_PATH_TC_BATCH, stream=stream)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = 1000.0 * e0.elapsed_time(e1) / max(1, args.steps)
    print(json.dumps({"mode": "batched", "steps": args.steps, "us_per_call": us,
                      "request_windows_per_s": bs["nreq"] / us * 1e6}))


def run_batched_projection_only(torch, vb, synth, dev, args):
    """The batched-serving projection (256 rows, hidden 5120, tensor-core batch
    path), warm-up + steps times."""
    H5, R = 5120, 256
    wd5 = torch.from_numpy(synth.weights(V, H5).view(np.int16)).to(dev)
    a = torch.from_numpy(synth.activations(R, H5, 500)).to(dev)
    lg = torch.empty((R, V), dtype=torch.float32, device=dev)
    ws = vb.workspace(R, H5, V, device=dev)
    for _ in range(args.warmup):
        vb.verify_project(wd5, a, lg, ws, path=vb.VR_PATH_TC_BATCH)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vb.verify_project(wd5, a, lg, ws, path=vb.VR_PATH_TC_BATCH)
    torch.cuda.synchronize(dev)
    print(json.dumps({"mode": "project_batched", "steps": args.steps,
                      "us_per_call": 1e6 * (time.perf_counter() - t0) / max(1, args.steps)}))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    from speculative_decoding_verify_row_gb300 import binding as vb, replicas, synth
    from speculative_decoding_verify_row_gb300 import build as vbuild

    rank, world, local = replicas.init("nccl" if args.gpus > 1 else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    vbuild.build()
    vb.lib()

    if args.mode == "topk":
        run_topk_only(torch, vb, dev, args)
        return
    if args.mode == "project_batched":
        run_batched_projection_only(torch, vb, synth, dev, args)
        return
    if args.mode == "batched":
        run_batched_only(torch, vb, synth, dev, args)
        return
    W = synth.weights(V, H)
    wd = torch.from_numpy(W.view(np.int16)).to(dev)
    if args.mode == "project":
        run_projection_only(torch, vb, synth, wd, dev, args)
        return
    if args.mode == "penalize":
        run_penalize_only(torch, vb, synth, wd, dev, args)
        return
    win = make_windows(torch, vb, synth, wd, dev)
    pol = vb.Policy(**POLICY)
    logits = torch.empty((ROWS, V), dtype=torch.float32, device=dev)
    out = torch.empty(ROWS, dtype=torch.int32, device=dev)
    acc = torch.empty(1, dtype=torch.int32, device=dev)
    ne = torch.empty(1, dtype=torch.int32, device=dev)
    ws = vb.workspace(ROWS, H, V, device=dev)
    stream = torch.cuda.current_stream(dev)

    # each distinct window's call, marshalled once (vb.prepare_window): a
    # timed window costs one C call on the host
    calls = [vb.prepare_window(wd, win["act"][s], win["drafts"][s], pol, s, 4096, logits, out, acc,
                               ne, ws, q_ids=win["q_ids"][s], q_logits=win["q_log"][s],
                               stream=stream) for s in range(N_WINDOWS)]

    def window(i):
        calls[i % N_WINDOWS]()

    def timed_region():
        """W warm-up windows, then exactly K timed windows bracketed by a
        barrier and a device synchronisation on both sides, CUDA events on
        the launching stream.  The clock sampler starts before the warm-up,
        so the GPU does not sit idle (and its clocks do not fall back)
        between the warm-up and the timed region."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clocks:
            for i in range(args.warmup):
                window(i)
            replicas.barrier()
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for i in range(args.steps):
                window(i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            replicas.barrier()
        elapsed_s = e0.elapsed_time(e1) / 1000.0
        job_s, job_windows = replicas.job_time_and_units(elapsed_s, args.steps,
                                                         device=dev if args.gpus > 1 else None)
        if vb.device_status(ws) != 0:
            raise RuntimeError("device status set during the warm-up or the timed region")
        return job_windows / job_s, job_s, clocks

    if args.mode == "window":
        value, job_s, clocks = timed_region()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "windows/s", "mode": "window",
                              "steps": args.steps, "warmup": args.warmup}), flush=True)
        replicas.shutdown()
        return

    # The breakdowns below run before the timed region.  Right after start-up
    # a GPU's first windows run up to 6 % slower for some milliseconds (its
    # power and clock state rising under load), which a timed region of a
    # few windows would otherwise catch; after them the GPU is in the state
    # the timed region is meant to measure.
    # ---- stage breakdown: the same windows through the stage entry points,
    # events between stages on the launching stream ----
    # sample sizes of the breakdowns below are fixed, whatever --steps is
    n_stage = STAGE_SAMPLES
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_stage)]
    pool_ids = torch.empty((ROWS, 64), dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)
    for i in range(n_stage):
        s = i % N_WINDOWS
        evs[i][0].record(stream)
        vb.verify_project(wd, win["act"][s], logits, ws, stream=stream)
        evs[i][1].record(stream)
        vb.verify_sample_accept(logits, win["drafts"][s], pol, s, 4096, out, acc, ne, ws,
                                q_ids=win["q_ids"][s], q_logits=win["q_log"][s], stream=stream)
        evs[i][2].record(stream)
    torch.cuda.synchronize(dev)
    proj_ms = [e[0].elapsed_time(e[1]) for e in evs]
    samp_ms = [e[1].elapsed_time(e[2]) for e in evs]
    proj_avg_s = statistics.fmean(proj_ms) / 1000.0
    proj_sorted = sorted(proj_ms)
    proj_pct = lambda q: 1000.0 * proj_sorted[min(len(proj_sorted) - 1, int(q * len(proj_sorted)))]
    # per-window latency of the fused call: events around every window, so
    # no window overlaps the next (the timed region above lets them overlap
    # their launch and prologue)
    n_lat = LATENCY_SAMPLES
    lat_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_lat)]
    torch.cuda.synchronize(dev)
    for i in range(n_lat):
        lat_ev[i][0].record(stream)
        window(i)
        lat_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    lat_us = sorted(1000.0 * e[0].elapsed_time(e[1]) for e in lat_ev)
    pct = lambda q: lat_us[min(len(lat_us) - 1, int(q * len(lat_us)))]
    window_latency = {"p10": pct(0.10), "p50": pct(0.50), "p90": pct(0.90), "windows": n_lat,
                      "timing": "CUDA events around each fused window"}
    # the pool select alone, on the same logits
    pool_vals = torch.empty((ROWS, 64), dtype=torch.float32, device=dev)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(200):
        vb.verify_select(logits, pool_ids, pool_vals, ws, stream=stream)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    select_us = 1000.0 * s0.elapsed_time(s1) / 200

    # ---- window cost against rows (projection stage, both paths) ----
    sweep = {}
    for path, name in ((vb.VR_PATH_TC, "tc"), (vb.VR_PATH_FFMA, "ffma")):
        sweep[name] = {}
        for R in (1, 2, 4, 8, 9, 16, 24, 25, 32):
            a = torch.from_numpy(synth.activations(R, H, 9000 + R)).to(dev)
            lg = torch.empty((R, V), dtype=torch.float32, device=dev)
            wsr = vb.workspace(R, H, V, device=dev)
            for _ in range(3):
                vb.verify_project(wd, a, lg, wsr, path=path, stream=stream)
            n_it = 30
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(n_it):
                vb.verify_project(wd, a, lg, wsr, path=path, stream=stream)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            sweep[name][str(R)] = round(1000.0 * t0.elapsed_time(t1) / n_it, 2)

    extra = None if args.no_extra else extra_workloads(torch, vb, synth, wd, dev, stream,
                                                       EXTRA_SAMPLES)
    cost_model = None if args.no_extra else window_cost_model(torch, vb, synth, wd, dev, stream)

    # ---- timed region: K fused windows ----
    value, job_s, clocks = timed_region()

    # ---- e2e: host inputs -> window -> host outputs, through the C ABI ----
    # A serving loop over independent windows: each step moves its inputs
    # from pinned host memory to the GPU, runs the window and returns
    # [accept, n, ids] into pinned host memory (vr_verify_window_host_async);
    # the host reads step i - 1's result (after its event) while step i runs.
    # The synchronous call (one wait per window, as a single sequence's
    # decode loop needs) is timed too.
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    h_act = [pin(win["act_np"][s]) for s in range(N_WINDOWS)]
    h_dr = [pin(win["drafts_np"][s]) for s in range(N_WINDOWS)]
    h_qi = [pin(win["q_ids_np"][s]) for s in range(N_WINDOWS)]
    h_ql = [pin(win["q_log_np"][s]) for s in range(N_WINDOWS)]
    h_out = pin(np.zeros(ROWS, np.int32))
    h_res = [pin(np.zeros(ROWS + 2, np.int32)) for _ in range(2)]
    events = [torch.cuda.Event() for _ in range(2)]
    n_e2e = E2E_SAMPLES

    def e2e_async(n, first):
        emitted = 0
        for i in range(n + 1):
            if i < n:
                s = (first + i) % N_WINDOWS
                b = i % 2
                vb.verify_window_host_async(wd, h_act[s], h_dr[s], pol, s, 4096, logits, h_res[b],
                                            ws, q_ids_h=h_qi[s], q_logits_h=h_ql[s], stream=stream)
                events[b].record(stream)
            if i > 0:
                b = (i - 1) % 2
                events[b].synchronize()
                n_em = int(h_res[b][1])
                if n_em < 1:
                    raise RuntimeError("a window emitted nothing")
                emitted += n_em
        return emitted

    e2e_async(10, 0)
    replicas.barrier()
    t0 = time.perf_counter()
    e2e_async(n_e2e, 0)
    e2e_s = time.perf_counter() - t0
    replicas.barrier()
    e2e_job_s, e2e_units = replicas.job_time_and_units(e2e_s, n_e2e,
                                                       device=dev if args.gpus > 1 else None)
    host_calls = [vb.prepare_window_host(wd, h_act[s], h_dr[s], pol, s, 4096, logits, h_out, ws,
                                         q_ids_h=h_qi[s], q_logits_h=h_ql[s], stream=stream)
                  for s in range(N_WINDOWS)]
    for i in range(10):
        host_calls[i]()
    n_sync = E2E_SYNC_SAMPLES
    t0 = time.perf_counter()
    for i in range(n_sync):
        if host_calls[i % N_WINDOWS]()[1] < 1:
            raise RuntimeError("a window emitted nothing")
    sync_s = time.perf_counter() - t0
    h2d = ROWS * H * 4 + K_DRAFTS * 4 + K_DRAFTS * 8 * 4 * 2
    d2h = (ROWS + 2) * 4

    peak, peak_kind = measured_peaks()
    achieved = WEIGHT_BYTES / proj_avg_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * job_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16xf32->f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "hidden": H, "vocab": V,
                   "distinct_windows": N_WINDOWS, "l2": "inputs larger than L2 (1.24 GB weights)",
                   "projection_path": "tc", "parallelism": f"replicas x{world}"},
        "hbm_gbs": WEIGHT_BYTES * value / world / 1e9,
        "hbm_frac_of_8tbs": WEIGHT_BYTES * value / world / 8e12,
        "roofline": {"bound": "hbm", "kernel": "projection (project_tc_kernel, planes built in the kernel)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_record("project_tc_kernel"),
                     "algorithmic_bytes_per_launch": WEIGHT_BYTES,
                     "launches_timed": n_stage,
                     "launch_us": {"mean": 1e6 * proj_avg_s, "p10": proj_pct(0.10),
                                   "p50": proj_pct(0.50), "p90": proj_pct(0.90)}},
        "stages_us": {"projection": 1000.0 * statistics.fmean(proj_ms),
                      "pool_policy_accept": 1000.0 * statistics.fmean(samp_ms),
                      "pool_select_only": select_us,
                      "window": 1e6 * job_s / args.steps},
        "stages_pct_of_window": {
            "projection": 100.0 * statistics.fmean(proj_ms) / (1000.0 * job_s / args.steps),
            "pool_policy_accept": 100.0 * statistics.fmean(samp_ms) / (1000.0 * job_s / args.steps),
            "pool_select_only": 100.0 * select_us / (1e6 * job_s / args.steps)},
        "window_latency_us": window_latency,
        "rows_sweep_us": sweep,
        "window_cost_model": cost_model,
        "other_workloads": extra,
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_units / e2e_job_s, "unit": "windows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "api": "vr_verify_window_host_async, next window "
                "enqueued before the previous result is read; the pinned inputs are read over "
                "the host link by the staging kernel and [accept, n, ids] written back into "
                "pinned memory by the acceptance kernel (no copy-engine transfers)"},
        "e2e_sync": {"value": n_sync / sync_s, "unit": "windows/s",
                     "api": "vr_verify_window_host (prepared call), one wait per window"},
        # per timed window: project_tc (planes built in the kernel for <= 16
        # rows) and sample_rows; no penalties in this workload, so no penalty
        # or q-copy launches
        "gpu_launches": 2 * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times = cpu_oracle_windows(W, win, 3)
        line["cpu_baseline"] = {"value": 3 / sum(times), "unit": "windows/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": "3 full oracle windows of the workload (fp64 projection "
                                          "+ pool/policy/acceptance)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    replicas.shutdown()


if __name__ == "__main__":
    main()
