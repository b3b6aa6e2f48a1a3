"""Multi-rank deterministic token mapping (UniEP page, section 2.2,
Algorithm 1: local stable sort, AllGather of the per-expert counts, prefix
sums over lower ranks).

With G ranks and experts partitioned over owners, token-slot (t, j) of rank
r routed to expert e gets the global address
    (owner(e), seg_start[e] + sum_{r' < r} counts[r'][e] + local_rank(t, j))
where seg_start[e] is the start of expert e's segment in its owner's
receive buffer (experts of one owner stored in index order, each segment
holding rank 0's slots, then rank 1's, ...) and local_rank is the slot's
stable rank among rank r's slots to e (what the single-rank permutation
builder computes).  No atomics decide an address, so the mapping does not
depend on execution order, and with G = 1 it is the single-GPU mapping.

The counts exchange is the only collective (all_gather over the default
process group: NCCL between GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch


def owner_of(E: int, G: int):
    """Experts are split into G contiguous blocks of ceil(E/G)."""
    per = -(-E // G)
    return [min(e // per, G - 1) for e in range(E)]


def rank_bases(all_counts: torch.Tensor, rank: int, owners):
    """all_counts [G, E] (CUDA tensor, the all-gathered counts) -> ([E] base
    address inside the owner's receive buffer of rank `rank`'s first slot
    for every expert, [G] rows each owner receives), both int32 on the same
    device, computed by the library (moe_rank_bases)."""
    from . import moe
    if not all_counts.is_cuda:
        raise ValueError("all_counts must be a CUDA tensor: the library computes the bases on the device")
    G, E = all_counts.shape
    dev = all_counts.device
    counts = all_counts.to(torch.int32).contiguous()
    owner = torch.tensor(list(owners), dtype=torch.int32, device=dev)
    base = torch.empty(E, dtype=torch.int32, device=dev)
    rows = torch.empty(G, dtype=torch.int32, device=dev)
    moe.moe_rank_bases(counts, owner, rank, base, rows)
    return base, rows


def all_gather_counts(local_counts: torch.Tensor) -> torch.Tensor:
    """[E] counts of this rank -> [G, E] counts of every rank (int64)."""
    import torch.distributed as dist
    x = local_counts.to(torch.int64)
    if not (dist.is_available() and dist.is_initialized()):
        return x[None]
    bufs = [torch.empty_like(x) for _ in range(dist.get_world_size())]
    dist.all_gather(bufs, x)
    return torch.stack(bufs)
