"""Multi-process replica bookkeeping on CPU (gloo, world size 2): the job's
time is the slowest rank's and its work the sum of the ranks' work."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    from speculative_decoding_verify_row_gb300 import replicas
    r, w, local = replicas.init("gloo")
    replicas.barrier()
    t, u = replicas.job_time_and_units(0.5 + rank, 100 * (rank + 1))
    q.put((r, w, t, u))
    replicas.shutdown()


def test_two_gloo_ranks_reduce_time_and_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:2] for r in res] == [(0, 2), (1, 2)]
    for _, _, t, u in res:
        assert t == 1.5 and u == 300.0


def test_single_process_is_identity():
    from speculative_decoding_verify_row_gb300 import replicas
    assert replicas.job_time_and_units(2.0, 7) == (2.0, 7.0)
