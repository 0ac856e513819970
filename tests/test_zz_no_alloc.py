"""The workspace-free select (vr_verify_select_noalloc), called through the C
ABI: same pools as vr_verify_select, on two calls in a row whose inputs
differ, and the documented row limit.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

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
    x[:, rng.integers(0, V, 50)] = np.float32(3.5)                 # ties
    x[0, :7] = np.float32([np.nan, -np.inf, np.inf, 0.0, -0.0, 3.5, 3.5])
    return torch.from_numpy(x).cuda()


def _select_with_workspace(lib, logits):
    from speculative_decoding_verify_row_gb300 import binding as vb
    R, V = logits.shape
    ids = torch.empty((R, 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, 64), dtype=torch.float32, device="cuda")
    vb.verify_select(logits, ids, vals, vb.workspace(R, 8, V))
    return ids, vals


def _select_noalloc(lib, logits):
    R, V = logits.shape
    ids = torch.full((R, 64), -9, dtype=torch.int32, device="cuda")
    vals = torch.zeros((R, 64), dtype=torch.float32, device="cuda")
    st = lib.vr_verify_select_noalloc(ctypes.c_void_p(logits.data_ptr()), R, V,
                                      ctypes.c_void_p(ids.data_ptr()),
                                      ctypes.c_void_p(vals.data_ptr()), None)
    assert st == 0
    return ids, vals


def test_matches_the_workspace_select_on_two_calls_in_a_row(lib):
    for seed, (R, V) in enumerate([(25, 151936), (4, 5000)]):
        logits = _rows(seed, R, V)
        got_ids, got_vals = _select_noalloc(lib, logits)
        torch.cuda.synchronize()
        ref_ids, ref_vals = _select_with_workspace(lib, logits)
        torch.cuda.synchronize()
        assert torch.equal(got_ids, ref_ids)
        assert torch.equal(got_vals.view(torch.int32), ref_vals.view(torch.int32))


def test_rejects_rows_beyond_the_limit(lib):
    from speculative_decoding_verify_row_gb300 import binding as vb
    logits = torch.zeros((vb.VR_NOALLOC_SELECT_MAX_ROWS + 1, 100), dtype=torch.float32, device="cuda")
    ids = torch.empty((logits.shape[0], 64), dtype=torch.int32, device="cuda")
    vals = torch.empty((logits.shape[0], 64), dtype=torch.float32, device="cuda")
    st = lib.vr_verify_select_noalloc(ctypes.c_void_p(logits.data_ptr()), logits.shape[0], 100,
                                      ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(vals.data_ptr()),
                                      None)
    assert st == vb.VR_ERR_UNSUPPORTED
