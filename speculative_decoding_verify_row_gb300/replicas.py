"""Replica bookkeeping for multi-process runs (one process per GPU).

The verify step has no exchange between requests, so N GPUs run N
independent replicas of the same workload: no collective touches the data
path.  The only cross-process steps are a barrier around the timed region
and the reduction of its timing: the job's time is the slowest rank's, and
its work is the sum of the ranks' work.
"""
import os

import torch
import torch.distributed as dist


def env_world():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend):
    rank, world, local = env_world()
    if world > 1 and not dist.is_initialized():
        if backend == "nccl":
            # each rank's own GPU before NCCL binds its communicator
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def barrier():
    if dist.is_initialized():
        dist.barrier()


def job_time_and_units(elapsed_s, units, device=None):
    """(max elapsed over ranks, sum of units over ranks)."""
    if not dist.is_initialized():
        return float(elapsed_s), float(units)
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def shutdown():
    if dist.is_initialized():
        dist.destroy_process_group()
