"""GPU penalty prepass and acceptance, bit for bit against the oracle given
the same logits ("Speculative decoding on RDNA" §02-§04, point-mass drafts
§06; token trees and naive sampling verify from the other two pages)."""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verify_row_gb300 import binding as vb
from gpu_common import require_gpu, dev, same_bits_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def bpol(p):
    return vb.Policy(**p.__dict__)


def random_tree(rng, n, chain):
    if chain:
        return None, ov.chain_parents(n)
    parent = [int(rng.integers(-1, j)) if j else -1 for j in range(n)]
    return np.array(parent, np.int32), parent


PEN_POLICIES = [
    ov.Policy(temperature=0.7, window=64, repeat=1.1, presence=1.5, frequency=0.2),
    ov.Policy(temperature=0.7, window=1, presence=1.5),
    ov.Policy(temperature=0.0, window=512, repeat=0.8, frequency=-0.3),
    ov.Policy(temperature=0.7, window=5, repeat=1.3),
    ov.Policy(temperature=0.7, window=0, presence=9.0),          # disabled by W = 0
    ov.Policy(temperature=0.7, window=30),                       # all neutral
]


@pytest.mark.parametrize("pi", range(len(PEN_POLICIES)))
@pytest.mark.parametrize("chain", [True, False])
def test_penalize_bit_exact(pi, chain):
    pol = PEN_POLICIES[pi]
    rng = np.random.default_rng(pi * 2 + chain)
    V, n = 3000, 12
    pt, parent = random_tree(rng, n, chain)
    tokens = rng.integers(0, 200, n).astype(np.int32)
    hist = rng.integers(-5, 200, 700).astype(np.int32)        # a few ids outside [0, V)
    hist[hist > 150] = V + 3
    logits = (rng.standard_normal((n + 1, V)) * 3).astype(np.float32)
    logits[:, 0] = np.nan
    logits[:, 1] = -0.0
    logits[:, 2] = np.inf
    q_ids = rng.integers(0, 200, (n, 8)).astype(np.int32)
    q_log = rng.standard_normal((n, 8)).astype(np.float32)
    L, Q = dev(logits), dev(q_log)
    ws = vb.workspace(n + 1, 8, V)
    vb.verify_penalize(L, dev(tokens), dev(hist), bpol(pol), ws, parent=None if pt is None else dev(pt),
                       q_ids=dev(q_ids), q_logits=Q)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    H = ov.row_histories(hist, tokens, parent, pol.window)
    for r in range(n + 1):
        assert same_bits_f32(L[r].cpu().numpy(), ov.penalize_row(logits[r], H[r], pol)), r
    for j in range(n):
        ref = ov.penalize_candidates(q_ids[j], q_log[j], H[ov.row_of(parent[j])], pol)
        assert same_bits_f32(Q[j].cpu().numpy(), ref), j


ACC_POLICIES = [
    ov.Policy(temperature=0.0),
    ov.Policy(temperature=0.7),
    ov.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95),
    ov.Policy(temperature=1.5, top_k=0),
    ov.Policy(temperature=0.3, top_k=3, top_p=0.8),
]


def gpu_accept(pen, tokens, pt, q_ids, q_log, pol, seed, position):
    R, V = pen.shape
    out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ne = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = vb.workspace(R, 8, V)
    vb.verify_sample_accept(dev(pen), dev(tokens) if len(tokens) else None, bpol(pol), seed,
                            position, out, acc, ne, ws, parent=None if pt is None else dev(pt),
                            q_ids=None if q_ids is None else dev(q_ids),
                            q_logits=None if q_log is None else dev(q_log))
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(acc.item()), int(ne.item()), vb.device_status(ws)


@pytest.mark.parametrize("pi", range(len(ACC_POLICIES)))
@pytest.mark.parametrize("shape", ["chain_q", "chain_noq", "tree"])
def test_accept_bit_exact(pi, shape):
    pol = ACC_POLICIES[pi]
    rng = np.random.default_rng(31 * pi + len(shape))
    V = 1000
    for trial in range(40):
        n = int(rng.integers(0, 10))
        pt, parent = random_tree(rng, n, shape != "tree")
        pen = (rng.standard_normal((n + 1, V)) * 2).astype(np.float32)
        top = np.argsort(-pen, axis=1)[:, :16]
        # drafts that often agree with the target so that long prefixes occur
        tokens = np.array([top[ov.row_of(parent[j]), int(rng.integers(0, 3))] for j in range(n)],
                          np.int32)
        q_ids = q_log = None
        if shape == "chain_q" and n:
            q_ids = np.stack([rng.permutation(top[j])[:8] for j in range(n)]).astype(np.int32)
            q_ids[:, 0] = tokens
            q_log = (np.take_along_axis(pen[:n], q_ids, 1) + rng.standard_normal((n, 8))).astype(np.float32)
        seed, position = int(rng.integers(0, 2**63)), int(rng.integers(0, 10**6))
        ids, acc, ne, st = gpu_accept(pen, tokens, pt, q_ids, q_log, pol, seed, position)
        ref = ov.verify_window(pen, tokens, parent, q_ids, q_log, (), pol, seed, position)
        assert st == 0
        assert (acc, ne) == (ref.accept, ref.n_emitted), (trial, acc, ne, ref.accept)
        assert list(ids[:ne]) == ref.emitted


def test_invalid_device_data_sets_the_status_word():
    V = 50
    pen = np.zeros((3, V), np.float32)
    _, acc, ne, st = gpu_accept(pen, np.int32([1, 99]), None, None, None, ov.Policy(), 0, 0)
    assert ne == 0 and st & vb.VR_DEV_BAD_TOKEN
    _, acc, ne, st = gpu_accept(pen, np.int32([1, 2]), np.int32([-1, 1]), None, None, ov.Policy(), 0, 0)
    assert ne == 0 and st & vb.VR_DEV_BAD_PARENT
    q = np.zeros((2, 8), np.int32)
    q[1, 3] = -4
    _, acc, ne, st = gpu_accept(pen, np.int32([1, 2]), None, q, np.zeros((2, 8), np.float32),
                                ov.Policy(temperature=1.0), 0, 0)
    assert ne == 0 and st & vb.VR_DEV_BAD_QID
    # a good window afterwards is unaffected
    _, acc, ne, st = gpu_accept(pen, np.int32([0, 0]), None, None, None, ov.Policy(), 0, 0)
    assert ne == 3 and st == 0


def test_point_mass_drafts_match_one_finite_candidate():
    """Sampled chains without candidates take q = delta(draft); the same
    window given 8 candidates of which only the draft is finite must emit the
    same tokens, and both must match the oracle."""
    rng = np.random.default_rng(77)
    V = 2000
    pol = ov.Policy(temperature=0.8, top_k=0, min_p=0.02, top_p=0.95)
    accepted = rejected = 0
    for trial in range(60):
        n = int(rng.integers(1, 9))
        pen = (rng.standard_normal((n + 1, V)) * 4).astype(np.float32)
        top = np.argsort(-pen, axis=1)[:, :2]
        tokens = np.array([top[j, 0 if rng.random() < 0.7 else 1] for j in range(n)], np.int32)
        q_ids = rng.integers(0, V, (n, 8)).astype(np.int32)
        q_ids[:, 0] = tokens
        q_log = np.full((n, 8), -np.inf, np.float32)
        q_log[:, 0] = rng.standard_normal(n).astype(np.float32)
        seed, position = int(rng.integers(0, 2**63)), int(rng.integers(0, 10**6))
        a = gpu_accept(pen, tokens, None, None, None, pol, seed, position)
        b = gpu_accept(pen, tokens, None, q_ids, q_log, pol, seed, position)
        ref = ov.verify_window(pen, tokens, None, None, None, (), pol, seed, position)
        assert a[3] == 0 and b[3] == 0
        assert (a[1], a[2]) == (ref.accept, ref.n_emitted) == (b[1], b[2])
        assert list(a[0][:a[2]]) == ref.emitted == list(b[0][:b[2]])
        accepted += ref.accept
        rejected += ref.accept < n
    assert accepted > 20 and rejected > 20


def special_rows(R, V, rng):
    """Rows with degenerate values: all NaN, all -inf but one 0, +inf
    entries, all -inf, a +0/-0 tie on top of negative values, and plain
    Gaussian rows; NaN with the sign bit set is mixed in."""
    rows = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    neg_nan = np.frombuffer(np.uint32(0xFFC00123).tobytes(), np.float32)[0]
    for r in range(R):
        kind = r % 6
        if kind == 0:
            rows[r] = np.nan
            rows[r, ::3] = neg_nan
        elif kind == 1:
            rows[r] = -np.inf
            rows[r, 17 % V] = 0.0
        elif kind == 2:
            rows[r, 5 % V] = np.inf
            rows[r, 9 % V] = np.inf
        elif kind == 3:
            rows[r] = -np.inf
        elif kind == 4:
            rows[r] = -np.abs(rows[r]) - 1.0
            rows[r, 3 % V] = 0.0
            rows[r, 30 % V] = -0.0
    return rows


@pytest.mark.parametrize("pi", range(len(ACC_POLICIES)))
@pytest.mark.parametrize("shape", ["chain_q", "chain_noq", "tree"])
def test_accept_on_special_values(pi, shape):
    """Pool, policy and acceptance on rows of NaN, -inf and +inf, on a +0/-0
    tie and on draft candidates whose logits are -inf: the GPU's decisions
    equal the oracle's bit for bit."""
    pol = ACC_POLICIES[pi]
    rng = np.random.default_rng(77 * pi + len(shape))
    V = 300
    for trial in range(12):
        n = 5 + int(rng.integers(0, 6))
        pt, parent = random_tree(rng, n, shape != "tree")
        pen = special_rows(n + 1, V, rng)
        order = [ov.target_pool(pen[r])[0][:16] for r in range(n + 1)]
        tokens = np.array([order[ov.row_of(parent[j])][int(rng.integers(0, 4))] for j in range(n)],
                          np.int32)
        q_ids = q_log = None
        if shape == "chain_q":
            q_ids = np.stack([rng.permutation(order[j])[:8] for j in range(n)]).astype(np.int32)
            q_ids[:, 0] = tokens
            q_log = rng.standard_normal((n, 8)).astype(np.float32)
            q_log[rng.random((n, 8)) < 0.3] = -np.inf
            q_log[0] = -np.inf
        seed, position = int(rng.integers(0, 2**63)), int(rng.integers(0, 10**6))
        ids, acc, ne, st = gpu_accept(pen, tokens, pt, q_ids, q_log, pol, seed, position)
        ref = ov.verify_window(pen, tokens, parent, q_ids, q_log, (), pol, seed, position)
        assert st == 0
        assert (acc, ne) == (ref.accept, ref.n_emitted), (trial, acc, ne, ref.accept)
        assert list(ids[:ne]) == ref.emitted
        assert ne >= 1
