"""The workspace-free select (vr_verify_select_noalloc), called through the C
ABI.  It serves callers that cannot give the library device memory (a plugin
whose host application owns every device allocation, a process that must not
grow its device footprint once it is serving).  Checked here:
  * on two calls in a row whose inputs differ, its pools equal those of
    vr_verify_select with a workspace, and every row equals the oracle's
    pool (ids and value bits), with ties, NaN, +-inf, signed zeros, a full
    vocabulary and vocabularies narrower than the pool;
  * calls after the first leave the device's free memory unchanged;
  * rows beyond the documented limit are rejected.
Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import verify as ov

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_verify_row_gb300 import build as vbuild, binding
    vbuild.build()
    return binding.lib()


def _rows(seed, R, V):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    x[:, rng.integers(0, V, max(1, V // 40))] = np.float32(3.5)       # ties
    special = np.float32([np.nan, -np.inf, np.inf, 0.0, -0.0, 3.5, 3.5])[:V]
    x[0, :len(special)] = special
    if R > 1:
        x[1, :] = np.float32(0.0)                                       # a row of equal values
        x[1, rng.integers(0, V, max(1, V // 10))] = -np.float32(0.0)
    if R > 2:
        x[2, rng.random(V) < 0.3] = np.nan                              # NaN with either sign
        x[2, rng.random(V) < 0.1] = -np.float32(np.nan)
    return x


def _select_with_workspace(logits):
    from speculative_decoding_verify_row_gb300 import binding as vb
    R, V = logits.shape
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.verify_select(logits, ids, vals, vb.workspace(R, 8, V))
    return ids, vals


def _call_noalloc(lib, logits, ids, vals):
    R, V = logits.shape
    return lib.vr_verify_select_noalloc(ctypes.c_void_p(logits.data_ptr()), R, V,
                                        ctypes.c_void_p(ids.data_ptr()),
                                        ctypes.c_void_p(vals.data_ptr()), None)


def _select_noalloc(lib, logits):
    R = logits.shape[0]
    ids = torch.full((R, 64), -9, dtype=torch.int32, device="cuda")
    vals = torch.zeros((R, 64), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, logits, ids, vals) == 0
    return ids, vals


def _assert_oracle_pools(x, ids, vals):
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    for r in range(x.shape[0]):
        want_ids, want_vals = ov.target_pool(x[r])
        n = len(want_ids)
        assert np.array_equal(ids[r, :n], want_ids), r
        got, want = vals[r, :n], np.asarray(want_vals, np.float32)
        assert np.array_equal(np.isnan(got), np.isnan(want)), r
        ok = ~np.isnan(want)
        assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32)), r
        assert np.all(ids[r, n:] == -1) and np.all(np.isnan(vals[r, n:])), r


@pytest.mark.parametrize("R,V", [(25, 151936), (4, 5000), (3, 40), (2, 1)])
def test_matches_the_workspace_select_and_the_oracle_on_two_calls_in_a_row(lib, R, V):
    for call in range(2):
        x = _rows(100 * V + call, R, V)
        logits = torch.from_numpy(x).cuda()
        got_ids, got_vals = _select_noalloc(lib, logits)
        torch.cuda.synchronize()
        ref_ids, ref_vals = _select_with_workspace(logits)
        torch.cuda.synchronize()
        assert torch.equal(got_ids, ref_ids)
        assert torch.equal(got_vals.view(torch.int32), ref_vals.view(torch.int32))
        _assert_oracle_pools(x, got_ids, got_vals)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_in_sequence_match_the_oracle(lib, seed):
    """Random row counts (up to the limit) and vocabularies (1 to 300000,
    across the one-pass and sub-block segment sizes), one call after another
    on the library's fixed array: every pool equals the oracle's."""
    from speculative_decoding_verify_row_gb300 import binding as vb
    rng = np.random.default_rng(9_000 + seed)
    for _ in range(3):
        R = int(rng.integers(1, vb.VR_NOALLOC_SELECT_MAX_ROWS + 1))
        V = int(rng.choice([1, 7, 63, 64, 65, 1000, 16384, 16385, 100_003, 300_000]))
        if R * V > 4_000_000:
            R = max(1, 4_000_000 // V)
        x = _rows(int(rng.integers(0, 2**31)), R, V)
        got_ids, got_vals = _select_noalloc(lib, torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        _assert_oracle_pools(x, got_ids, got_vals)


def test_later_calls_leave_free_device_memory_unchanged(lib):
    # inputs and outputs first, then one call (the first call on a device
    # loads the library's fixed array), then two more calls of different
    # sizes between two readings of the device's free memory
    a = torch.from_numpy(_rows(7, 32, 151936)).cuda()
    b = torch.from_numpy(_rows(8, 5, 777)).cuda()
    ids = torch.empty((32, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((32, 64), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, a, ids, vals) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _call_noalloc(lib, b, ids, vals) == 0
    assert _call_noalloc(lib, a, ids, vals) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    _assert_oracle_pools(a.cpu().numpy(), ids, vals)


def test_rejects_rows_beyond_the_limit(lib):
    from speculative_decoding_verify_row_gb300 import binding as vb
    logits = torch.zeros((vb.VR_NOALLOC_SELECT_MAX_ROWS + 1, 100), dtype=torch.float32, device="cuda")
    ids = torch.empty((logits.shape[0], 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((logits.shape[0], 64), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, logits, ids, vals) == vb.VR_ERR_UNSUPPORTED
