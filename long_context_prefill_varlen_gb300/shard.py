"""Request sharding of the drop step across GPUs (host-side bookkeeping only).

Every stage of the step (score, select, compact, scatter-back, seqused) is local to a request, so a
batch runs on several GPUs by giving each rank whole requests; no data crosses GPUs.  This module
holds the two host-side pieces that need a rule: which rank takes which request (token-balanced,
deterministic), and, for callers that want one global packed view of the compacted stream, the
global query_start_loc rebuilt from the per-rank kept lengths (an all-gather of R int32 values: it is
metadata, not part of the data path).  The tensor-parallel score sync of the paper (Eq. 15) is a
different split (by heads) and is not used here.
"""
from __future__ import annotations

import torch


def assign_requests(lengths, world_size):
    """Rank of each request: longest first onto the least-loaded rank (ties: lower rank), a fixed rule."""
    load = [0] * world_size
    owner = [0] * len(lengths)
    for r in sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i)):
        k = min(range(world_size), key=lambda j: (load[j], j))
        owner[r] = k
        load[k] += int(lengths[r])
    return owner


def local_requests(lengths, world_size, rank):
    """This rank's requests (in global order) and its packed cu_seqlens."""
    owner = assign_requests(lengths, world_size)
    mine = [r for r in range(len(lengths)) if owner[r] == rank]
    cu = [0]
    for r in mine:
        cu.append(cu[-1] + int(lengths[r]))
    return mine, cu


def global_query_start_loc(lengths, local_kept_lens, world_size, rank, group=None):
    """Global query_start_loc of the compacted stream, requests in their original order.

    local_kept_lens: kept tokens of this rank's requests (the new_seq_lens of its up_compact), in the
    order of local_requests().  One all_gather of R int32 values per call.
    """
    import torch.distributed as dist
    R = len(lengths)
    mine, _ = local_requests(lengths, world_size, rank)
    full = torch.zeros(R, dtype=torch.int64)
    for r, k in zip(mine, local_kept_lens):
        full[r] = int(k)
    parts = [torch.zeros(R, dtype=torch.int64) for _ in range(world_size)]
    dist.all_gather(parts, full, group=group)
    kept = torch.stack(parts).sum(dim=0)          # every request is owned by exactly one rank
    return torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(kept, 0)])
