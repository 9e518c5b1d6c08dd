"""Splitting grouped attention across ranks (one process per GPU).

Two ways the work shards, both exact:

* by group: groups are independent problems (each has its own prefix and responses), so a rank
  that owns whole groups needs no communication at all.  ``assign_groups`` balances them by their
  visible-pair count (longest-processing-time first).
* by response within a group: every rank holds the group's prefix and a subset of its responses
  and runs grouped attention on [P; R_subset].  Prefix outputs are the same on every rank (prefix
  rows never see responses).  In the backward, the upstream gradient of the prefix rows is routed
  to rank 0 only, so each rank's prefix dQ / dK / dV is a partial sum over its own responses (plus
  the prefix queries on rank 0); the shared prefix's gradient is the sum of the partials (the same
  statement as for the G baseline copies, Pith review of Prefix Grouper, Appendix A.1 objection).
  ``reduce_prefix_grads`` sums the partials in rank order, so the result does not depend on
  arrival order.

Only host-side bookkeeping and the exchange live here; the attention itself is the library's.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import torch

from . import flops


def assign_groups(prefix_lens: Sequence[int], group_sizes: Sequence[int],
                  suffix_lens: Sequence[int], world: int) -> List[List[int]]:
    """Groups of each rank, balanced by visible pairs (heaviest group to the least-loaded rank)."""
    per_group = flops.split_groups(group_sizes, suffix_lens)
    cost = [flops.group_pairs(lp, rs) for lp, rs in zip(prefix_lens, per_group)]
    order = sorted(range(len(cost)), key=lambda b: (-cost[b], b))
    load = [0] * world
    out: List[List[int]] = [[] for _ in range(world)]
    for b in order:
        r = min(range(world), key=lambda i: (load[i], i))
        out[r].append(b)
        load[r] += cost[b]
    return [sorted(x) for x in out]


def split_responses(num_responses: int, world: int, rank: int) -> List[int]:
    """Contiguous block of response indices for `rank` (sizes differ by at most one)."""
    base, extra = divmod(num_responses, world)
    start = rank * base + min(rank, extra)
    return list(range(start, start + base + (1 if rank < extra else 0)))


def shard_rows(prefix_len: int, suffix_lens: Sequence[int], responses: Sequence[int]) -> torch.Tensor:
    """Packed row indices (within one group) of the prefix followed by the given responses."""
    starts, s = [], prefix_len
    for r in suffix_lens:
        starts.append(s)
        s += r
    rows = list(range(prefix_len))
    for i in responses:
        rows += list(range(starts[i], starts[i] + suffix_lens[i]))
    return torch.tensor(rows, dtype=torch.int64)


def reduce_prefix_grads(partials: Sequence[torch.Tensor]) -> torch.Tensor:
    """Sum per-rank prefix gradients in rank order (deterministic)."""
    out = partials[0].clone()
    for p in partials[1:]:
        out += p
    return out


def allgather_prefix_grads(local: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange step: gather every rank's prefix partial, then sum them in rank order."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    bufs = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(bufs, local.contiguous(), group=group)
    return reduce_prefix_grads(bufs)


def route_prefix_do(do_shard: torch.Tensor, prefix_len: int, rank: int) -> torch.Tensor:
    """Upstream gradient of a rank's shard: the prefix rows' dO goes to rank 0 only."""
    if rank == 0:
        return do_shard
    out = do_shard.clone()
    out[:prefix_len] = 0
    return out


def shard_summary(prefix_len: int, suffix_lens: Sequence[int], world: int) -> Tuple[int, ...]:
    """Visible pairs per rank when the responses of one group are split across `world` ranks."""
    return tuple(flops.group_pairs(prefix_len, [suffix_lens[i] for i in
                                                split_responses(len(suffix_lens), world, r)])
                 for r in range(world))
