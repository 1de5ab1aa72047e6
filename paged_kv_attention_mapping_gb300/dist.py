"""Multi-process helpers for running one replica of the tick per GPU.

Attention over paged KV has no cross-sequence exchange: every (row, KV head)
unit is independent, so N GPUs run N replicas (weak scaling) and the only
collectives are a barrier around the timed region and the max of the
per-rank step times. No collective touches the data path.
"""
from __future__ import annotations

import os
from typing import Sequence


def rank_world():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init(backend: str = "nccl"):
    import torch.distributed as dist
    rank, local, world = rank_world()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return rank, local, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(values: Sequence[float], device=None) -> list:
    """Element-wise max of `values` over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_tokens_per_s(tokens_per_rank: int, ms_per_step_by_rank: float, world: int) -> float:
    """Whole-job throughput: all ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step_by_rank / 1000.0)
