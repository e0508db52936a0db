"""Host logic of multi-GPU runs: one process per GPU, each holding its own sequences.

The decode shards by independent sequences (no exchange on the data path), so a
run on N GPUs is N replicas: rank r draws its own sequences (seed + r), and the
only communication is the timing reduction at the end (max of the per-rank
times, sum of the per-rank attended tokens).

A context too long for one GPU shards by position instead: rank r holds one slice
of every sequence's context (a cache created with pos_offset at the slice's first
position), decodes it with witcert_decode_partial, and the ranks' per-cell records
are gathered (one all_gather, about 0.5 KB per sequence, query head and rank) and
merged with witcert_merge_partials.
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


def gather_partials(part):
    """Context-parallel exchange: every rank's shard records [B, Hq, R] -> [B, Hq, world, R] in
    rank order on every rank (one all_gather); a single process returns its own as one shard."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return part.unsqueeze(2).contiguous()
    import torch.distributed as dist
    bufs = [torch.empty_like(part) for _ in range(dist.get_world_size())]
    dist.all_gather(bufs, part.contiguous())
    return torch.stack(bufs, dim=2).contiguous()
