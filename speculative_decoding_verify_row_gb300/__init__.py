"""verifyrow for GB300: the data-parallel hot path of the speculative-decoding
verify step (projection, penalty prepass, pool and sampler policy,
acceptance) as hand-written sm_103a CUDA kernels behind a C ABI
(include/verifyrow.h, libverifyrow.so), with a thin ctypes binding."""
from .binding import (  # noqa: F401
    LIB_PATH, Policy, VerifyRowError, device_status, lib, make_request, topk, verify_penalize,
    verify_policy, verify_project, verify_sample_accept, verify_select, verify_window,
    verify_window_batched, verify_window_host, verify_window_host_async, window_pools, workspace,
    workspace_bytes,
    VR_PATH_AUTO, VR_PATH_FFMA, VR_PATH_TC, VR_PATH_TC_BATCH, VR_POOL, VR_QCAND, VR_OK, VR_ERR_ARG,
    VR_ERR_CUDA, VR_ERR_UNSUPPORTED, VR_ERR_DEVICE, VR_ERR_WORKSPACE, VR_DEV_BAD_TOKEN,
    VR_DEV_BAD_PARENT, VR_DEV_BAD_QID, VR_DEV_TIMEOUT)
