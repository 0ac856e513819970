"""GPU pool select and sampler policy, bit for bit against the oracle
("Speculative decoding on RDNA" §03: the pool, its tie-breaking and the
summation order are fixed)."""
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


def adversarial_rows(R, V, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, V)).astype(np.float32)
    kind = seed % 4
    if kind == 1:                       # heavy ties from a small value set
        x = rng.choice(np.float32([2.5, 1.0, 0.0, -0.0, -1.0]), size=(R, V)).astype(np.float32)
    elif kind == 2:                     # specials sprinkled in
        specials = np.float32([np.inf, -np.inf, np.nan, 0.0, -0.0, 3.0e38, -3.0e38, 1e-45])
        mask = rng.random((R, V)) < 0.2
        x[mask] = rng.choice(specials, size=mask.sum())
        neg_nan = rng.random((R, V)) < 0.01
        x[neg_nan] = np.frombuffer(np.uint32(0xFFC00123).tobytes(), np.float32)[0]
    elif kind == 3:                     # all equal: pure id order
        x[:] = np.float32(0.5)
    return x


def gpu_pool(x):
    R, V = x.shape
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    ws = vb.workspace(R, 8, V)
    vb.verify_select(dev(x), ids, vals, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), vals.cpu().numpy()


@pytest.mark.parametrize("V", [1, 7, 63, 64, 65, 2047, 2048, 2049, 5000, 151936, 400000])
@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_pool_matches_oracle(V, kind):
    R = 3 if V > 100000 else 5
    x = adversarial_rows(R, V, 100 * V + kind)
    ids, vals = gpu_pool(x)
    n = min(64, V)
    for r in range(R):
        ref_ids, ref_vals = ov.target_pool(x[r])
        assert np.array_equal(ids[r, :n], ref_ids), (r, ids[r, :n], ref_ids)
        assert np.array_equal(vals[r, :n].view(np.uint32), ref_vals.view(np.uint32))
        assert np.all(ids[r, n:] == -1)


@pytest.mark.parametrize("V", [1_500_007, 4_194_305])
@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_pool_past_the_one_pass_segment(V, kind):
    """Vocabularies above 64 segments of 16384: each segment is longer than
    one register load and is selected sub-block by sub-block with its running
    list carried (pools and the batched top-K against the oracle)."""
    x = adversarial_rows(2, V, V + kind)
    ids, vals = gpu_pool(x)
    tk_ids, tk_vals = gpu_topk(x, 16)
    for r in range(2):
        ref_ids, ref_vals = ov.target_pool(x[r])
        assert np.array_equal(ids[r], ref_ids), r
        assert np.array_equal(vals[r].view(np.uint32), ref_vals.view(np.uint32)), r
        assert np.array_equal(tk_ids[r], ref_ids[:16]), r
        assert np.array_equal(tk_vals[r].view(np.uint32), ref_vals[:16].view(np.uint32)), r


def test_pool_of_the_tree_rows():
    x = adversarial_rows(25, 151936, 8)
    ids, _ = gpu_pool(x)
    for r in range(25):
        assert np.array_equal(ids[r], ov.target_pool(x[r])[0])


POLICIES = [
    ov.Policy(temperature=0.0),
    ov.Policy(temperature=0.7),
    ov.Policy(temperature=0.7, top_k=0, min_p=0.05, top_p=0.95),
    ov.Policy(temperature=1.0, top_k=5),
    ov.Policy(temperature=3.0, top_k=0),
    ov.Policy(temperature=0.05, top_k=0, top_p=0.5),
    ov.Policy(temperature=1.3, top_k=100, min_p=0.3),
    ov.Policy(temperature=0.8, top_k=1),
    ov.Policy(temperature=1e-30, top_k=0),
    ov.Policy(temperature=2.0, top_k=0, top_p=0.0),
    ov.Policy(temperature=0.9, top_k=0, min_p=2.0),
]


def pools_for_policy(seed):
    rng = np.random.default_rng(seed)
    v = -np.sort(-(rng.standard_normal((12, 64)) * rng.uniform(0.1, 8, (12, 1)))).astype(np.float32)
    v[3, 40:] = -np.inf
    v[4, 10:] = np.nan
    v[5, :] = v[5, 0]
    v[6, 20:] = v[6, 19]
    v[7, 1:] = -np.float32(3e38)
    return v


@pytest.mark.parametrize("pi", range(len(POLICIES)))
@pytest.mark.parametrize("pool_len", [64, 8, 3, 1])
def test_policy_bit_exact(pi, pool_len):
    pol = POLICIES[pi]
    v = pools_for_policy(pi * 10 + pool_len)
    R = v.shape[0]
    m = torch.empty(R, dtype=torch.int32, device="cuda")
    e = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    S = torch.empty(R, dtype=torch.float32, device="cuda")
    vb.verify_policy(dev(v), pool_len, vb.Policy(**pol.__dict__), m, e, S)
    torch.cuda.synchronize()
    m, e, S = m.cpu().numpy(), e.cpu().numpy(), S.cpu().numpy()
    for r in range(R):
        rm, re, rS = ov.policy_weights(v[r, :pool_len], pol)
        assert m[r] == rm
        assert np.array_equal(e[r, :rm].view(np.uint32), np.array(re, np.float32).view(np.uint32))
        assert np.all(e[r, rm:] == 0.0)
        assert np.float32(S[r]).view(np.uint32) == np.float32(rS).view(np.uint32)


def gpu_topk(x, k):
    R, V = x.shape
    ids = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.empty((R, k), dtype=torch.float32, device="cuda")
    ws = vb.workspace(R, 8, V)
    vb.topk(dev(x), k, ids, vals, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), vals.cpu().numpy()


@pytest.mark.parametrize("seed", range(12))
def test_topk_byte_identity_15x248320(seed):
    """The draft tuner's batched top-K ("feat(dflash) ...": 15 rows x 248320,
    K = 16, ties, NaN and -inf): ids and value bytes identical to the
    oracle."""
    x = adversarial_rows(15, 248320, seed)
    if seed % 4 == 0:                   # a tie block straddling the 16th place
        x[:, 1000:1040] = x.max()
    ids, vals = gpu_topk(x, 16)
    for r in range(15):
        ref_ids, ref_vals = ov.top_k_entries(x[r], 16)
        assert np.array_equal(ids[r], ref_ids), r
        assert np.array_equal(vals[r].view(np.uint32), ref_vals.view(np.uint32)), r


@pytest.mark.parametrize("k", [1, 7, 16, 33, 64])
@pytest.mark.parametrize("V", [5, 64, 4097, 248320])
def test_topk_widths(k, V):
    x = adversarial_rows(4, V, 7 * k + V)
    ids, vals = gpu_topk(x, k)
    n = min(k, V)
    for r in range(4):
        ref_ids, ref_vals = ov.top_k_entries(x[r], k)
        assert np.array_equal(ids[r, :n], ref_ids)
        assert np.array_equal(vals[r, :n].view(np.uint32), ref_vals.view(np.uint32))
        assert np.all(ids[r, n:] == -1)
    if k == 64:
        pid, pval = gpu_pool(x)
        assert np.array_equal(pid, ids) and np.array_equal(pval.view(np.uint32), vals.view(np.uint32))


def _small_k_edge_rows(V, seed):
    """Rows for the top-k of at most 16 entries (per-segment threshold from
    warp sorts, lists merged by ranks): all NaN but five finite values (the
    rest of the top 16 are NaNs, lowest ids first); one 16384-id segment all
    NaN and another all -inf among normal draws; all equal; the top 16
    entries all in the last, partial segment; a tie block across a segment
    boundary straddling the 16th place."""
    rng = np.random.default_rng(seed)
    rows = rng.standard_normal((6, V)).astype(np.float32)
    rows[0] = np.nan
    rows[0, rng.choice(V, 5, replace=False)] = rng.standard_normal(5).astype(np.float32)
    if V > 2 * 16384:
        rows[1, 16384:2 * 16384] = np.nan
        rows[1, 2 * 16384:min(V, 3 * 16384)] = -np.inf
    rows[2] = np.float32(0.25)
    rows[3, V - 20:] = np.float32(9.0) + np.arange(20, dtype=np.float32) / 8
    b = min(16384, V // 2)
    rows[4, b - 12:b + 12] = rows[4].max() + 1
    rows[5] = rng.choice(np.float32([1.0, 0.5, -0.0, 0.0]), V).astype(np.float32)
    return rows


@pytest.mark.parametrize("k", [1, 2, 7, 16])
@pytest.mark.parametrize("V", [300, 20000, 248320, 262144])
def test_small_k_topk_edges(k, V):
    x = _small_k_edge_rows(V, seed=V + k)
    ids, vals = gpu_topk(x, k)
    for r in range(x.shape[0]):
        ref_ids, ref_vals = ov.top_k_entries(x[r], k)
        assert np.array_equal(ids[r], ref_ids), (r, k, V)
        assert np.array_equal(vals[r].view(np.uint32), ref_vals.view(np.uint32)), (r, k, V)


def test_pools_and_projection_on_a_second_device():
    """Kernel attributes (shared-memory limits) and SM counts belong to a
    device: the select and the tensor-core projection run on cuda:1 after
    cuda:0 and both match the oracle.  Skipped with one GPU."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two CUDA devices")
    from speculative_decoding_verify_row_gb300 import synth
    from gpu_common import assert_logits_close
    V, H, R = 151936, 64, 4
    x = adversarial_rows(R, V, 4242)
    rng = np.random.default_rng(4243)
    W = synth.f32_to_bf16_bits(rng.standard_normal((5000, H)).astype(np.float32) * np.float32(0.1))
    A = rng.standard_normal((R, H)).astype(np.float32)
    ref = ov.project(W, A)
    for d in (0, 1):
        with torch.cuda.device(d):
            dv = torch.device("cuda", d)
            ids = torch.empty((R, 64), dtype=torch.int32, device=dv)
            vals = torch.empty((R, 64), dtype=torch.float32, device=dv)
            vb.verify_select(torch.from_numpy(x).to(dv), ids, vals, vb.workspace(R, 8, V, device=dv))
            logits = torch.empty((R, 5000), dtype=torch.float32, device=dv)
            wd = torch.from_numpy(W.view(np.int16)).to(dv)
            vb.verify_project(wd, torch.from_numpy(A).to(dv), logits, vb.workspace(R, H, 5000, device=dv),
                              path=vb.VR_PATH_TC)
            torch.cuda.synchronize(dv)
        ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
        for r in range(R):
            ref_ids, ref_vals = ov.target_pool(x[r])
            assert np.array_equal(ids[r], ref_ids), (d, r)
            assert same_bits_f32(vals[r], ref_vals), (d, r)
        assert_logits_close(logits.cpu().numpy(), ref)
