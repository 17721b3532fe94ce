"""L-sharded selection across ranks: the host-side exchange protocol.

One sequence's latent cache can be split into contiguous shards of token
positions, one per rank (a 128K-token cache over eight GPUs, the setting of
the explainer page's storage paragraph).  Every rank scores its own shard
(eq. (8) of the summary page, restricted to its positions) and keeps, per
layer, the top-k of that shard with the shard's global positions.  The ranks
then all-gather these k (score, position) pairs and every rank takes the
top-k of the gathered candidates, ties to the lower position.

Exactness: a position outside its shard's top-k has k positions of its own
shard ahead of it in (score desc, position asc) order, so it is not in the
row's top-k either; the row's top-k therefore lies inside the union of the
shards' top-k lists, and a merge with the same order returns exactly the
one-pass set, ties across shards included.

This module holds only the bookkeeping of that protocol -- shard ranges,
local-to-global positions and the gather in rank order -- so it runs the same
on CPU (gloo) and GPU (NCCL) process groups.  The selections themselves are
the caller's (on the GPU, li_topk on the shard and on the gathered lists).
Shards must hold at least k positions each so that no shard list is padded.
"""
from __future__ import annotations

import torch


def shard_range(L: int, world: int, rank: int) -> tuple[int, int]:
    """Positions [start, stop) of rank's shard: contiguous, in rank order, the
    first L % world shards one position longer."""
    if not (0 <= rank < world) or L < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(L, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def check_shards(L: int, world: int, k: int) -> None:
    """Every shard must hold at least k positions (no padded shard lists)."""
    if L // world < k:
        raise ValueError(f"shards of {L // world} positions cannot each give k = {k} candidates")


def to_global(local_idx: torch.Tensor, start: int) -> torch.Tensor:
    """Shard-local selected indices -> global token positions."""
    if (local_idx < 0).any():
        raise ValueError("a shard list is padded: shards need at least k positions")
    return local_idx + start


def gather_candidates(vals: torch.Tensor, pos: torch.Tensor, group=None):
    """All-gather every rank's [..., k] candidate scores and global positions.

    Returns ([..., world * k] scores, [..., world * k] positions), rank r's
    list at [..., r * k:(r + 1) * k].  Shards are in rank order, so every
    candidate of rank r lies before every candidate of rank r + 1."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    vs = [torch.empty_like(vals) for _ in range(world)]
    ps = [torch.empty_like(pos) for _ in range(world)]
    dist.all_gather(vs, vals.contiguous(), group=group)
    dist.all_gather(ps, pos.contiguous(), group=group)
    return torch.cat(vs, dim=-1), torch.cat(ps, dim=-1)
