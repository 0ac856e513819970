"""Thin Python binding of libverifyrow (argument marshalling only).

Every function here checks tensor devices, dtypes and shapes, passes raw
pointers and sizes to the C ABI declared in include/verifyrow.h, and turns a
negative status into VerifyRowError.  All computation happens in the CUDA
kernels behind the C ABI; there is no fallback: if the shared library is
missing or fails to load, every call raises.

Device tensors are torch CUDA tensors; the stream is the current torch
stream of the tensors' device unless one is given.
"""
import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libverifyrow.so")

VR_OK = 0
VR_ERR_ARG = -1
VR_ERR_CUDA = -2
VR_ERR_UNSUPPORTED = -3
VR_ERR_DEVICE = -4
VR_ERR_WORKSPACE = -5
VR_DEV_BAD_TOKEN = 1
VR_DEV_BAD_PARENT = 2
VR_DEV_BAD_QID = 4
VR_DEV_TIMEOUT = 8
VR_PATH_AUTO = 0
VR_PATH_FFMA = 1
VR_PATH_TC = 2
VR_PATH_TC_BATCH = 3
VR_POOL = 64
VR_QCAND = 8
VR_MAX_WINDOW_ROWS = 64
VR_MAX_ROWS = 1024
VR_MAX_PENALTY_WINDOW = 512
VR_MAX_REQUESTS = 256
VR_NOALLOC_SELECT_MAX_ROWS = 32


class VerifyRowError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().vr_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} ({status})")


class vr_policy(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32),
                ("min_p", ctypes.c_float), ("top_p", ctypes.c_float),
                ("repeat", ctypes.c_float), ("presence", ctypes.c_float),
                ("frequency", ctypes.c_float), ("window", ctypes.c_int32)]


class vr_request(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("tokens", ctypes.c_void_p),
                ("parent", ctypes.c_void_p), ("q_ids", ctypes.c_void_p),
                ("q_logits", ctypes.c_void_p), ("hist", ctypes.c_void_p),
                ("hist_len", ctypes.c_int32), ("policy", vr_policy),
                ("seed", ctypes.c_uint64), ("position", ctypes.c_uint64),
                ("out_ids", ctypes.c_void_p), ("out_accept", ctypes.c_void_p),
                ("out_n_emitted", ctypes.c_void_p)]


@dataclass
class Policy:
    """Sampler and penalty settings of one request (mirrors vr_policy)."""
    temperature: float = 0.0
    top_k: int = -1
    min_p: float = 0.0
    top_p: float = 1.0
    repeat: float = 1.0
    presence: float = 0.0
    frequency: float = 0.0
    window: int = 0

    def c(self):
        return vr_policy(self.temperature, self.top_k, self.min_p, self.top_p, self.repeat,
                         self.presence, self.frequency, self.window)


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64

_SIGNATURES = {
    "vr_abi_version": ([], _I),
    "vr_status_string": ([_I], ctypes.c_char_p),
    "vr_workspace_bytes": ([_I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "vr_workspace_init": ([_P, _SZ, _P], _I),
    "vr_verify_project": ([_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "vr_verify_penalize": ([_P, _I, _I, _P, _P, _I, _P, _I, ctypes.POINTER(vr_policy), _P, _P,
                            _P, _SZ, _P], _I),
    "vr_verify_select": ([_P, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "vr_verify_select_noalloc": ([_P, _I, _I, _P, _P, _P], _I),
    "vr_topk": ([_P, _I, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "vr_ngram_propose": ([_P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "vr_cost_fit": ([_P, _P, _I, _P, _P], _I),
    "vr_choose_depth": ([_P, _I, ctypes.c_double, ctypes.c_double, _P, _P], _I),
    "vr_takeover": ([_P, _I, _P, _I, ctypes.c_double, ctypes.c_double, _P], _I),
    "vr_ar_floor": ([ctypes.c_double, _P, _P, _I, _P], _I),
    "vr_verify_policy": ([_P, _I, _I, ctypes.POINTER(vr_policy), _P, _P, _P, _P], _I),
    "vr_verify_sample_accept": ([_P, _I, _I, _P, _P, _I, _P, _P, ctypes.POINTER(vr_policy),
                                 _U64, _U64, _P, _P, _P, _P, _SZ, _P], _I),
    "vr_verify_window": ([_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _I,
                          ctypes.POINTER(vr_policy), _U64, _U64, _P, _P, _P, _P, _P, _P, _SZ,
                          _P], _I),
    "vr_verify_window_batched": ([_P, _P, _I, _I, _I, ctypes.POINTER(vr_request), _I, _P, _P,
                                  _P, _SZ, _P], _I),
    "vr_verify_window_host": ([_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _I,
                               ctypes.POINTER(vr_policy), _U64, _U64, _P, _P, _P, _P, _P, _P,
                               _SZ, _P], _I),
    "vr_verify_window_host_async": ([_P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _I,
                                     ctypes.POINTER(vr_policy), _U64, _U64, _P, _P, _P, _P,
                                     _SZ, _P], _I),
    "vr_window_pools": ([_P, _SZ, _I, _I, _I, _P, _P, _P], _I),
    "vr_device_status": ([_P, ctypes.POINTER(ctypes.c_int32), _P], _I),
}


def lib():
    """Load libverifyrow.so (built by __graft_entry__.build() or build.py)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libverifyrow.so is not built ({LIB_PATH}); run the build step")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = handle
    return _LIB


def _check(status, where):
    if status != VR_OK:
        raise VerifyRowError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype, name, shape=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _stream(stream, device=None):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


_WEIGHT_DTYPES = (torch.bfloat16, torch.int16, torch.uint16)


def workspace_bytes(rows, hidden, vocab):
    out = _SZ(0)
    _check(lib().vr_workspace_bytes(rows, hidden, vocab, ctypes.byref(out)), "vr_workspace_bytes")
    return out.value


def workspace(rows, hidden, vocab, device="cuda", stream=None):
    """Allocate (through torch) and initialise a workspace for these sizes."""
    n = workspace_bytes(rows, hidden, vocab)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    _check(lib().vr_workspace_init(_ptr(ws), n, _stream(stream, ws.device)), "vr_workspace_init")
    return ws


def device_status(ws, stream=None):
    out = ctypes.c_int32(0)
    _check(lib().vr_device_status(_ptr(ws), ctypes.byref(out), _stream(stream, ws.device)),
           "vr_device_status")
    return out.value


def verify_project(weight, act, logits, ws, path=VR_PATH_AUTO, stream=None):
    V, H = weight.shape
    R = act.shape[0]
    _dev(weight, _WEIGHT_DTYPES, "weight")
    _dev(act, torch.float32, "act", (R, H))
    _dev(logits, torch.float32, "logits", (R, V))
    _check(lib().vr_verify_project(_ptr(weight), _ptr(act), R, H, V, path, _ptr(logits), _ptr(ws),
                                   ws.numel(), _stream(stream, act.device)), "vr_verify_project")
    return logits


def _opt_i32(t, name, shape=None):
    _dev(t, torch.int32, name, shape)
    return _ptr(t)


def verify_penalize(logits, tokens, hist, policy, ws, parent=None, q_ids=None, q_logits=None,
                    stream=None):
    R, V = logits.shape
    n = R - 1
    _dev(logits, torch.float32, "logits")
    _dev(q_logits, torch.float32, "q_logits", (n, VR_QCAND))
    pol = policy.c()
    _check(lib().vr_verify_penalize(_ptr(logits), R, V, _opt_i32(tokens, "tokens", (n,)),
                                    _opt_i32(parent, "parent", (n,)), n,
                                    _opt_i32(hist, "hist"), 0 if hist is None else hist.numel(),
                                    ctypes.byref(pol), _opt_i32(q_ids, "q_ids", (n, VR_QCAND)),
                                    _ptr(q_logits), _ptr(ws), ws.numel(),
                                    _stream(stream, logits.device)), "vr_verify_penalize")
    return logits


def verify_select(logits, pool_ids, pool_vals, ws, stream=None):
    R, V = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(pool_ids, torch.int32, "pool_ids", (R, VR_POOL))
    _dev(pool_vals, torch.float32, "pool_vals", (R, VR_POOL))
    _check(lib().vr_verify_select(_ptr(logits), R, V, _ptr(pool_ids), _ptr(pool_vals), _ptr(ws),
                                  ws.numel(), _stream(stream, logits.device)), "vr_verify_select")
    return pool_ids, pool_vals


def topk(x, k, ids, vals, ws, stream=None):
    """vr_topk: the first k entries of each row of x in pool order."""
    R, V = x.shape
    _dev(x, torch.float32, "x")
    _dev(ids, torch.int32, "ids", (R, k))
    _dev(vals, torch.float32, "vals", (R, k))
    _check(lib().vr_topk(_ptr(x), R, V, k, _ptr(ids), _ptr(vals), _ptr(ws), ws.numel(),
                         _stream(stream, x.device)), "vr_topk")
    return ids, vals


def verify_select_noalloc(logits, pool_ids, pool_vals, stream=None):
    """vr_verify_select without a workspace: for callers that cannot give
    the library device memory; its scratch is a fixed array inside the
    library, shared by all calls on a device (serialise them)."""
    R, V = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(pool_ids, torch.int32, "pool_ids", (R, VR_POOL))
    _dev(pool_vals, torch.float32, "pool_vals", (R, VR_POOL))
    _check(lib().vr_verify_select_noalloc(_ptr(logits), R, V, _ptr(pool_ids), _ptr(pool_vals),
                                          _stream(stream, logits.device)),
           "vr_verify_select_noalloc")
    return pool_ids, pool_vals


def verify_policy(pool_vals, pool_len, policy, out_m, out_e, out_S, stream=None):
    R = pool_vals.shape[0]
    _dev(pool_vals, torch.float32, "pool_vals", (R, VR_POOL))
    _dev(out_m, torch.int32, "out_m", (R,))
    _dev(out_e, torch.float32, "out_e", (R, VR_POOL))
    _dev(out_S, torch.float32, "out_S", (R,))
    pol = policy.c()
    _check(lib().vr_verify_policy(_ptr(pool_vals), R, pool_len, ctypes.byref(pol), _ptr(out_m),
                                  _ptr(out_e), _ptr(out_S), _stream(stream, pool_vals.device)),
           "vr_verify_policy")


def verify_sample_accept(pen_logits, tokens, policy, seed, position, out_ids, out_accept,
                         out_n, ws, parent=None, q_ids=None, q_logits=None, stream=None):
    R, V = pen_logits.shape
    n = R - 1
    _dev(pen_logits, torch.float32, "pen_logits")
    _dev(q_logits, torch.float32, "q_logits", (n, VR_QCAND))
    _dev(out_ids, torch.int32, "out_ids", (R,))
    _dev(out_accept, torch.int32, "out_accept", (1,))
    _dev(out_n, torch.int32, "out_n", (1,))
    pol = policy.c()
    _check(lib().vr_verify_sample_accept(_ptr(pen_logits), R, V, _opt_i32(tokens, "tokens", (n,)),
                                         _opt_i32(parent, "parent", (n,)), n,
                                         _opt_i32(q_ids, "q_ids", (n, VR_QCAND)), _ptr(q_logits),
                                         ctypes.byref(pol), seed, position, _ptr(out_ids),
                                         _ptr(out_accept), _ptr(out_n), _ptr(ws), ws.numel(),
                                         _stream(stream, pen_logits.device)),
           "vr_verify_sample_accept")


def _window_args(weight, act, tokens, policy, seed, position, logits, out_ids, out_accept,
                 out_n, ws, parent, q_ids, q_logits, hist, pen_logits, path, stream):
    V, H = weight.shape
    R = act.shape[0]
    n = R - 1
    _dev(weight, _WEIGHT_DTYPES, "weight")
    _dev(act, torch.float32, "act", (R, H))
    _dev(logits, torch.float32, "logits", (R, V))
    _dev(pen_logits, torch.float32, "pen_logits", (R, V))
    _dev(q_logits, torch.float32, "q_logits", (n, VR_QCAND))
    _dev(out_ids, torch.int32, "out_ids", (R,))
    _dev(out_accept, torch.int32, "out_accept", (1,))
    _dev(out_n, torch.int32, "out_n", (1,))
    pol = policy.c()
    return pol, (_ptr(weight), _ptr(act), R, H, V, path, _opt_i32(tokens, "tokens", (n,)),
                 _opt_i32(parent, "parent", (n,)), n, _opt_i32(q_ids, "q_ids", (n, VR_QCAND)),
                 _ptr(q_logits), _opt_i32(hist, "hist"), 0 if hist is None else hist.numel(),
                 ctypes.byref(pol), seed, position, _ptr(logits), _ptr(pen_logits),
                 _ptr(out_ids), _ptr(out_accept), _ptr(out_n), _ptr(ws), ws.numel(),
                 _stream(stream, act.device))


def verify_window(weight, act, tokens, policy, seed, position, logits, out_ids, out_accept,
                  out_n, ws, parent=None, q_ids=None, q_logits=None, hist=None, pen_logits=None,
                  path=VR_PATH_AUTO, stream=None):
    _, args = _window_args(weight, act, tokens, policy, seed, position, logits, out_ids,
                           out_accept, out_n, ws, parent, q_ids, q_logits, hist, pen_logits, path,
                           stream)
    _check(lib().vr_verify_window(*args), "vr_verify_window")


def prepare_window(weight, act, tokens, policy, seed, position, logits, out_ids, out_accept,
                   out_n, ws, parent=None, q_ids=None, q_logits=None, hist=None, pen_logits=None,
                   path=VR_PATH_AUTO, stream=None):
    """verify_window with its arguments checked and marshalled once: returns
    a callable that enqueues that same window (same buffers, seed, position
    and stream) each time it is called, at the cost of one C call.  For a
    loop that reuses its buffers; the tensors must outlive the callable."""
    pol, args = _window_args(weight, act, tokens, policy, seed, position, logits, out_ids,
                             out_accept, out_n, ws, parent, q_ids, q_logits, hist, pen_logits,
                             path, stream)
    fn = lib().vr_verify_window

    def call(_keep=(pol, weight, act, tokens, logits, out_ids, out_accept, out_n, ws, parent,
                    q_ids, q_logits, hist, pen_logits)):
        st = fn(*args)
        if st != VR_OK:
            raise VerifyRowError(st, "vr_verify_window")
    return call


def make_request(n_nodes, tokens, policy, seed, position, out_ids, out_accept, out_n,
                 parent=None, q_ids=None, q_logits=None, hist=None):
    """A vr_request descriptor over device tensors (the tensors must outlive the call)."""
    for t, name, dt in ((tokens, "tokens", torch.int32), (parent, "parent", torch.int32),
                        (q_ids, "q_ids", torch.int32), (q_logits, "q_logits", torch.float32),
                        (hist, "hist", torch.int32), (out_ids, "out_ids", torch.int32),
                        (out_accept, "out_accept", torch.int32), (out_n, "out_n", torch.int32)):
        _dev(t, dt, name)
    return vr_request(n_nodes, _ptr(tokens), _ptr(parent), _ptr(q_ids), _ptr(q_logits),
                      _ptr(hist), 0 if hist is None else hist.numel(), policy.c(), seed, position,
                      _ptr(out_ids), _ptr(out_accept), _ptr(out_n))


def verify_window_batched(weight, act, requests, logits, ws, pen_logits=None, path=VR_PATH_AUTO,
                          stream=None):
    V, H = weight.shape
    R = act.shape[0]
    _dev(weight, _WEIGHT_DTYPES, "weight")
    _dev(act, torch.float32, "act", (R, H))
    _dev(logits, torch.float32, "logits", (R, V))
    _dev(pen_logits, torch.float32, "pen_logits", (R, V))
    arr = (vr_request * len(requests))(*requests)
    _check(lib().vr_verify_window_batched(_ptr(weight), _ptr(act), H, V, path, arr, len(requests),
                                          _ptr(logits), _ptr(pen_logits), _ptr(ws), ws.numel(),
                                          _stream(stream, act.device)),
           "vr_verify_window_batched")


def _host_ptr(a, dtype, name):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if a.is_cuda or a.dtype != dtype or not a.is_contiguous():
            raise TypeError(f"{name} must be a contiguous host tensor of {dtype}")
        return ctypes.c_void_p(a.data_ptr())
    raise TypeError(f"{name} must be a host torch tensor")


_TLS = threading.local()


def _pinned_head():
    """A per-thread pinned int32 pair for accept / n_emitted, so the kernel
    writes them directly instead of a copy back to pageable memory."""
    head = getattr(_TLS, "head", None)
    if head is None:
        t = torch.zeros(2, dtype=torch.int32).pin_memory()
        head = _TLS.head = (t, t.numpy())
    return head


def _window_host_args(weight, act_h, tokens_h, policy, seed, position, logits, out_ids_h, ws,
                      parent_h, q_ids_h, q_logits_h, hist_h, pen_logits, path, stream, head):
    V, H = weight.shape
    R = act_h.shape[0]
    n = R - 1
    _dev(weight, _WEIGHT_DTYPES, "weight")
    _dev(logits, torch.float32, "logits", (R, V))
    _dev(pen_logits, torch.float32, "pen_logits", (R, V))
    pol = policy.c()
    return pol, (_ptr(weight), _host_ptr(act_h, torch.float32, "act_h"), R, H, V, path,
                 _host_ptr(tokens_h, torch.int32, "tokens_h"),
                 _host_ptr(parent_h, torch.int32, "parent_h"), n,
                 _host_ptr(q_ids_h, torch.int32, "q_ids_h"),
                 _host_ptr(q_logits_h, torch.float32, "q_logits_h"),
                 _host_ptr(hist_h, torch.int32, "hist_h"), 0 if hist_h is None else hist_h.numel(),
                 ctypes.byref(pol), seed, position, _ptr(logits), _ptr(pen_logits),
                 _host_ptr(out_ids_h, torch.int32, "out_ids_h"), ctypes.c_void_p(head.data_ptr()),
                 ctypes.c_void_p(head.data_ptr() + 4), _ptr(ws), ws.numel(),
                 _stream(stream, logits.device))


def verify_window_host(weight, act_h, tokens_h, policy, seed, position, logits, out_ids_h,
                       ws, parent_h=None, q_ids_h=None, q_logits_h=None, hist_h=None,
                       pen_logits=None, path=VR_PATH_AUTO, stream=None):
    """The window with host inputs and outputs (pinned host tensors are read
    and written by the kernels directly, pageable ones copied).  Returns
    (accept, n_emitted); synchronises."""
    head, head_np = _pinned_head()
    _, args = _window_host_args(weight, act_h, tokens_h, policy, seed, position, logits,
                                out_ids_h, ws, parent_h, q_ids_h, q_logits_h, hist_h, pen_logits,
                                path, stream, head)
    _check(lib().vr_verify_window_host(*args), "vr_verify_window_host")
    return int(head_np[0]), int(head_np[1])


def prepare_window_host(weight, act_h, tokens_h, policy, seed, position, logits, out_ids_h,
                        ws, parent_h=None, q_ids_h=None, q_logits_h=None, hist_h=None,
                        pen_logits=None, path=VR_PATH_AUTO, stream=None):
    """verify_window_host with its arguments checked and marshalled once:
    returns a callable that runs that window (reading the host inputs as
    they are at the time of the call) and returns (accept, n_emitted), one C
    call and one wait each time.  The accept/n_emitted pair lives in a
    pinned pair owned by the callable; the tensors must outlive it."""
    head = torch.zeros(2, dtype=torch.int32).pin_memory()
    head_np = head.numpy()
    pol, args = _window_host_args(weight, act_h, tokens_h, policy, seed, position, logits,
                                  out_ids_h, ws, parent_h, q_ids_h, q_logits_h, hist_h,
                                  pen_logits, path, stream, head)
    fn = lib().vr_verify_window_host

    def call(_keep=(pol, head, weight, act_h, tokens_h, logits, out_ids_h, ws, parent_h, q_ids_h,
                    q_logits_h, hist_h, pen_logits)):
        st = fn(*args)
        if st != VR_OK:
            raise VerifyRowError(st, "vr_verify_window_host")
        return int(head_np[0]), int(head_np[1])
    return call


def verify_window_host_async(weight, act_h, tokens_h, policy, seed, position, logits, out_h,
                             ws, parent_h=None, q_ids_h=None, q_logits_h=None, hist_h=None,
                             pen_logits=None, path=VR_PATH_AUTO, stream=None):
    """vr_verify_window_host_async: enqueues the window and one copy of
    [accept, n_emitted, ids...] into out_h (pinned int32 [rows + 2]); returns
    at once.  out_h is valid after the stream (or a later event) completes;
    pinned inputs must stay unchanged until then."""
    V, H = weight.shape
    R = act_h.shape[0]
    n = R - 1
    _dev(weight, _WEIGHT_DTYPES, "weight")
    _dev(logits, torch.float32, "logits", (R, V))
    _dev(pen_logits, torch.float32, "pen_logits", (R, V))
    if out_h.numel() < R + 2:
        raise ValueError("out_h needs rows + 2 int32")
    pol = policy.c()
    _check(lib().vr_verify_window_host_async(
        _ptr(weight), _host_ptr(act_h, torch.float32, "act_h"), R, H, V, path,
        _host_ptr(tokens_h, torch.int32, "tokens_h"), _host_ptr(parent_h, torch.int32, "parent_h"),
        n, _host_ptr(q_ids_h, torch.int32, "q_ids_h"),
        _host_ptr(q_logits_h, torch.float32, "q_logits_h"), _host_ptr(hist_h, torch.int32, "hist_h"),
        0 if hist_h is None else hist_h.numel(), ctypes.byref(pol), seed, position, _ptr(logits),
        _ptr(pen_logits), _host_ptr(out_h, torch.int32, "out_h"), _ptr(ws), ws.numel(),
        _stream(stream, logits.device)), "vr_verify_window_host_async")


def window_pools(ws, rows, hidden, vocab, ids, vals, stream=None):
    """vr_window_pools: the last window's pools (ids int32 [rows][64], vals
    float32 [rows][64], device tensors) from the workspace it ran with."""
    _dev(ids, torch.int32, "ids", (rows, 64))
    _dev(vals, torch.float32, "vals", (rows, 64))
    _check(lib().vr_window_pools(_ptr(ws), ws.numel(), rows, hidden, vocab, _ptr(ids), _ptr(vals),
                                 _stream(stream, ids.device)), "vr_window_pools")


# ---------------------------------------------------------------------------
# host-side draft proposal and window pricing (CPU only, numpy in and out)

def _np(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def ngram_propose(context, match=5, propose=3, branches=1, max_nodes=VR_MAX_WINDOW_ROWS - 1):
    """vr_ngram_propose: (tokens int32 [n], parent int32 [n]) of the
    prompt-lookup proposal for the context (prompt || emitted)."""
    ctx, pctx = _np(context, np.int32)
    toks = np.zeros(max(1, max_nodes), np.int32)
    par = np.zeros(max(1, max_nodes), np.int32)
    n = ctypes.c_int32(0)
    _check(lib().vr_ngram_propose(pctx if ctx.size else None, ctx.size, match, propose, branches,
                                  max_nodes, toks.ctypes.data_as(ctypes.c_void_p),
                                  par.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n)),
           "vr_ngram_propose")
    return toks[:n.value].copy(), par[:n.value].copy()


def cost_fit(rows, ms):
    """vr_cost_fit: (a, b) of ms = a + b (rows - 1)."""
    r, pr = _np(rows, np.int32)
    m, pm = _np(ms, np.float64)
    if r.size != m.size:
        raise ValueError("rows and ms differ in length")
    a, b = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().vr_cost_fit(pr, pm, r.size, ctypes.byref(a), ctypes.byref(b)), "vr_cost_fit")
    return a.value, b.value


def choose_depth(alpha, a, b, kmax=None):
    """vr_choose_depth: (k, tokens per unit cost)."""
    al, pal = _np(alpha, np.float64)
    kmax = al.size if kmax is None else kmax
    if kmax > al.size:
        raise ValueError("alpha needs kmax entries")
    k = ctypes.c_int32(0)
    rate = ctypes.c_double(0)
    _check(lib().vr_choose_depth(pal, kmax, a, b, ctypes.byref(k), ctypes.byref(rate)),
           "vr_choose_depth")
    return k.value, rate.value


def takeover(alpha_native, alpha_ngram, a, b):
    """vr_takeover: True if the n-gram window prices at least as well."""
    an, pan = _np(alpha_native, np.float64)
    ag, pag = _np(alpha_ngram, np.float64)
    out = ctypes.c_int32(0)
    _check(lib().vr_takeover(pan, an.size, pag, ag.size, a, b, ctypes.byref(out)), "vr_takeover")
    return bool(out.value)


def ar_floor(ar_ms, window_ms, emitted):
    """vr_ar_floor: True to keep speculating, False to retire."""
    w, pw = _np(window_ms, np.float64)
    e, pe = _np(emitted, np.int32)
    if w.size != e.size:
        raise ValueError("window_ms and emitted differ in length")
    out = ctypes.c_int32(0)
    _check(lib().vr_ar_floor(ar_ms, pw, pe, w.size, ctypes.byref(out)), "vr_ar_floor")
    return bool(out.value)
