"""Helpers for the GPU parity tests (imported by test_gpu_*.py only)."""
import numpy as np
import pytest
import torch

from speculative_decoding_verify_row_gb300 import binding as vb
from speculative_decoding_verify_row_gb300 import build as vbuild

LOGIT_TOL = 1e-3      # |gpu - ref| <= 1e-3 * max(1, |ref|), ref = the fp64 oracle


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    vbuild.build()
    vb.lib()


def dev_weight(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def project(wd, act, path, rows_first=None):
    act_d = act if isinstance(act, torch.Tensor) else dev(act)
    R, H = act_d.shape
    V = wd.shape[0]
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    ws = vb.workspace(R, H, V)
    vb.verify_project(wd, act_d, logits, ws, path=path)
    torch.cuda.synchronize()
    assert vb.device_status(ws) == 0
    return logits


def assert_logits_close(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = LOGIT_TOL * np.maximum(1.0, np.abs(ref))
    worst = np.max(err / bound) if err.size else 0.0
    assert worst <= 1.0, f"max |d| = {err.max():.3e}, worst ratio to bound {worst:.3f}"
    return err.max()


def same_bits_f32(a, b):
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a.view(np.uint32)[~na], b.view(np.uint32)[~nb])
