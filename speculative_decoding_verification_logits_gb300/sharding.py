"""Row sharding of a verify batch across devices.

Rows of a verify round are independent and the verify step's uniforms are
keyed by the global row number (``row_base + b``), so a batch split into
contiguous row ranges gives exactly the tokens of the unsplit batch.  The
only cross-shard quantity is the packed-token layout: a shard's offsets are
shifted by the token total of the shards before it (an exclusive scan of one
integer per rank).
"""
from __future__ import annotations

import torch


def shard_rows(B: int, world: int, rank: int) -> tuple[int, int]:
    """(row_base, rows) of `rank`'s contiguous share of B rows."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def global_offsets(local_offsets: torch.Tensor, group=None) -> tuple[torch.Tensor, int]:
    """Shift this shard's packed-token offsets ([rows+1], exclusive scan of
    tau) by the token totals of lower ranks.  Returns (shifted offsets,
    global token total).  One all_gather of one int64 per rank."""
    import torch.distributed as dist
    total = local_offsets[-1:].to(torch.int64)
    world = dist.get_world_size(group)
    parts = [torch.zeros_like(total) for _ in range(world)]
    dist.all_gather(parts, total, group=group)
    rank = dist.get_rank(group)
    before = int(sum(int(p.item()) for p in parts[:rank]))
    grand = int(sum(int(p.item()) for p in parts))
    return local_offsets.to(torch.int64) + before, grand
