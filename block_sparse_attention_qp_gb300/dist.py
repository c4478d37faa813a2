"""Process-group helpers for running independent MSA problems on several GPUs.

The method's work partitions into independent problems (batches / sequences), so N ranks each
process their own batch with no collective on the data path ("weak" scaling).  The only
communication is for measurement: a barrier around the timed region and a max over ranks of the
elapsed time.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_world():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), int(
        os.environ.get("LOCAL_RANK", "0"))


def init(backend: str):
    """Initialise the default process group from torchrun's environment (no-op for 1 rank)."""
    world, rank, local = env_world()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank, local


def barrier():
    if dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device="cpu") -> float:
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Every rank draws its own batch."""
    return base + 7919 * rank


def whole_job_rate(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Units of all ranks divided by the slowest rank's time."""
    return units_per_rank * world / seconds_max


def shutdown():
    if dist.is_initialized():
        dist.destroy_process_group()
