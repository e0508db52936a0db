"""Host logic of multi-GPU runs: one process per GPU, each holding its own sequences.

The decode shards by independent sequences (no exchange on the data path), so a
run on N GPUs is N replicas: rank r draws its own sequences (seed + r), and the
only communication is the timing reduction at the end (max of the per-rank
times, sum of the per-rank attended tokens).
"""
from __future__ import annotations

import os

import torch


def rank_env():
    """(rank, local_rank, world_size) from the torchrun environment (1 process if unset)."""
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def shard_seed(seed: int, rank: int) -> int:
    """Seed of the sequences held by `rank`: every rank serves different sequences."""
    return seed + rank


def reduce_timing(ms: float, tokens: float, device=None):
    """Whole-job (max time over ranks, total tokens over ranks); identity for one process."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(ms), float(tokens)
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())
