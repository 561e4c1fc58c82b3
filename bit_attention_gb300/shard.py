"""Head partition of one attention problem over ranks (one GPU per rank).

Attention treats every (batch, head) pair on its own: no step of the path
exchanges data between heads.  So one problem of B*H heads splits over G
ranks with no collective on the data path: rank r takes a contiguous range
of the flattened heads b*H + h, about B*H/G of them, and runs the whole path
(quantize + attention) on that range.  A contiguous range of heads of a
contiguous [B, H, N, D] tensor is itself a contiguous [1, c, N, D] tensor, so
each rank calls the library with B = 1 and H = c.  Gathering O onto every
rank is optional, for callers who want the whole output in one place.
"""
from __future__ import annotations


def shard_heads(B: int, H: int, rank: int, world: int) -> tuple[int, int]:
    """(first head, head count) of `rank`'s share of the B*H flattened heads.

    The first (B*H) % world ranks take one head more than the others; ranks
    past the last head get an empty range (count 0)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if B < 0 or H < 0:
        raise ValueError(f"B={B}, H={H}")
    total = B * H
    base, extra = divmod(total, world)
    count = base + (1 if rank < extra else 0)
    first = rank * base + min(rank, extra)
    return first, count


def head_view(x, first: int, count: int):
    """The [1, count, N, D] view of heads first..first+count-1 of a contiguous
    [B, H, N, D] tensor (no copy)."""
    B, H, N, D = x.shape
    if not x.is_contiguous():
        raise ValueError("head_view needs a contiguous [B, H, N, D] tensor")
    return x.reshape(B * H, N, D)[first:first + count].unsqueeze(0)


def gather_heads(local, B: int, H: int, group=None):
    """All-gather every rank's [1, c_r, N, D] share into the full [B, H, N, D]
    tensor on every rank, heads in order.  Shares may differ in size by one
    head; they are padded to the largest for the collective and trimmed."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    _, c, N, D = local.shape
    cmax = shard_heads(B, H, 0, world)[1]
    pad = torch.zeros((cmax, N, D), dtype=local.dtype, device=local.device)
    pad[:c] = local[0]
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    out = [parts[r][:shard_heads(B, H, r, world)[1]] for r in range(world)]
    return torch.cat(out, 0).reshape(B, H, N, D)
