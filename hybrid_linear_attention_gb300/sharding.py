"""Partitioning of KDA work across ranks (one process per GPU).

KDA heads are independent -- each has its own q, k, v, g, beta, state and output ("KDA state,
by contrast, splits by head": "Ling-3.1-flash: What 63 Linear-Attention Layers Do to the KV
Budget", section "The memory math") -- and so are sequences.  A rank therefore owns a
contiguous range of heads, or a subset of the packed batch's sequences, and runs the library on
its share with no collective on the data path.  These helpers only compute the shares.
"""
from __future__ import annotations


def head_shard(H: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous head range [h0, h1) of `rank`; sizes differ by at most one."""
    if not (0 <= rank < world) or H < 0:
        raise ValueError("bad head shard request")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def sequence_shard(lengths, world: int, rank: int) -> list[int]:
    """Indices of the sequences `rank` owns: longest-first greedy assignment to the rank with
    the fewest tokens so far (ties to the lower rank), so token counts stay balanced."""
    if not (0 <= rank < world):
        raise ValueError("bad sequence shard request")
    load = [0] * world
    owner = [0] * len(lengths)
    for i in sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i)):
        r = min(range(world), key=lambda r: (load[r], r))
        owner[i] = r
        load[r] += int(lengths[i])
    return [i for i in range(len(lengths)) if owner[i] == rank]
