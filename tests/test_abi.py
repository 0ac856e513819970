"""The C ABI without a GPU: the library builds and loads, exports every
function include/verifyrow.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verify_row_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verifyrow.h")


@pytest.fixture(scope="module")
def lib():
    path = vbuild.build()
    from speculative_decoding_verify_row_gb300 import binding
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vr_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
    # nothing but the C ABI is exported
    nm = os.popen(f"nm -D --defined-only {vbuild.LIB}").read()
    exported = set(re.findall(r" T (vr_\w+)", nm))
    assert exported == set(names)


def test_version_and_status_strings(lib):
    assert lib.vr_abi_version() == 1
    assert lib.vr_status_string(0) == b"ok"
    assert lib.vr_status_string(-1) == b"invalid argument"


def test_workspace_size_is_host_only(lib):
    out = ctypes.c_size_t(0)
    assert lib.vr_workspace_bytes(4, 4096, 151936, ctypes.byref(out)) == 0
    assert out.value > 4 * 64 * 8
    assert lib.vr_workspace_bytes(0, 4096, 151936, ctypes.byref(out)) == -1
    assert lib.vr_workspace_bytes(4, 4100, 151936, ctypes.byref(out)) == -3   # hidden % 8
    assert lib.vr_workspace_bytes(4, 4096, 151936, None) == -1


def test_bad_arguments_are_rejected_on_the_host(lib):
    from speculative_decoding_verify_row_gb300.binding import vr_policy
    p = ctypes.c_void_p(256)            # never dereferenced: validation fails first
    assert lib.vr_verify_project(p, p, 0, 4096, 100, 0, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_project(None, p, 4, 4096, 100, 0, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_project(p, p, 4, 4096, 100, 7, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_project(p, p, 4, 4096, 100, 0, p, None, 1 << 30, None) == -5
    assert lib.vr_verify_project(p, p, 4, 4096, 100, 0, p, p, 16, None) == -5
    good = vr_policy(0.7, -1, 0.0, 1.0, 1.0, 0.0, 0.0, 0)
    for bad in (vr_policy(float("nan"), -1, 0, 1, 1, 0, 0, 0), vr_policy(-1, -1, 0, 1, 1, 0, 0, 0),
                vr_policy(0.7, -1, 0, 1, 0.0, 0, 0, 0), vr_policy(0.7, -1, 0, 1, 1, 0, 0, 513),
                vr_policy(0.7, -1, 0, float("inf"), 1, 0, 0, 0)):
        assert lib.vr_verify_window(p, p, 4, 4096, 100, 0, p, None, 3, None, None, None, 0,
                                    ctypes.byref(bad), 0, 0, p, None, p, p, p, p, 1 << 30,
                                    None) == -1
    # rows must be nodes + 1; q ids and logits come together
    assert lib.vr_verify_window(p, p, 4, 4096, 100, 0, p, None, 2, None, None, None, 0,
                                ctypes.byref(good), 0, 0, p, None, p, p, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_window(p, p, 4, 4096, 100, 0, p, None, 3, p, None, None, 0,
                                ctypes.byref(good), 0, 0, p, None, p, p, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_window(p, p, 65, 4096, 100, 0, p, None, 64, None, None, None, 0,
                                ctypes.byref(good), 0, 0, p, None, p, p, p, p, 1 << 30, None) == -1
    assert lib.vr_verify_policy(p, 4, 65, ctypes.byref(good), p, p, p, None) == -1
    # top-K width in [1, 64]
    for k in (0, 65, -3):
        assert lib.vr_topk(p, 15, 248320, k, p, p, p, 1 << 30, None) == -1
    assert lib.vr_topk(p, 15, 248320, 16, None, p, p, 1 << 30, None) == -1
    assert lib.vr_topk(p, 15, 248320, 16, p, p, p, 64, None) == -5


def test_host_window_and_pool_arguments_are_rejected_on_the_host(lib):
    from speculative_decoding_verify_row_gb300.binding import vr_policy
    p = ctypes.c_void_p(256)            # never dereferenced: validation fails first
    good = vr_policy(0.7, -1, 0.0, 1.0, 1.0, 0.0, 0.0, 0)
    bad = vr_policy(-1.0, -1, 0.0, 1.0, 1.0, 0.0, 0.0, 0)

    def host_async(rows, nodes, pol, out_h, ws_bytes):
        return lib.vr_verify_window_host_async(p, p, rows, 4096, 100, 0, p, None, nodes, None, None,
                                               None, 0, ctypes.byref(pol), 0, 0, p, None, out_h, p,
                                               ws_bytes, None)
    assert host_async(4, 3, good, None, 1 << 30) == -1          # no result buffer
    assert host_async(4, 3, bad, p, 1 << 30) == -1              # negative temperature
    assert host_async(4, 2, good, p, 1 << 30) == -1             # rows != nodes + 1
    assert host_async(4, 3, good, p, 16) == -5                  # workspace too small
    # pools of the last window: outputs, shape and workspace are checked
    assert lib.vr_window_pools(p, 1 << 30, 4, 4096, 100, None, p, None) == -1
    assert lib.vr_window_pools(p, 1 << 30, 0, 4096, 100, p, p, None) == -1
    assert lib.vr_window_pools(p, 16, 4, 4096, 100, p, p, None) == -5
    assert lib.vr_window_pools(None, 1 << 30, 4, 4096, 100, p, p, None) == -5
