"""Sort across ranks by one exchange of top-digit buckets.

The pages' strategy for data that does not fit one device ("Parallel
Patterns: Sorting on the GPU", 10.5, strategy 3) splits the keys into
buckets that fit, sorts each bucket, and concatenates the buckets.  Here the
buckets are the 256 values of the top 8-bit digit and each rank owns a
contiguous range of them:

1. every rank counts the top digit of its shard (``gsort_digit_histograms``
   on bits [24, 32) of the key);
2. the ranks all-gather their 256 counts, so every rank knows the size of
   every bucket and how many keys of each bucket every rank holds;
3. ``plan`` gives rank r the buckets whose keys start at or after
   r * total / world in the global order, and up to the next rank's start:
   whole buckets, contiguous, in digit order (a bucket larger than total /
   world makes its owner hold more than the average; nothing is split);
4. every rank groups its keys by bucket with a stable sort on the top digit
   (``gsort_radix_pairs``, bits [24, 32)), so the keys for each destination
   rank are contiguous;
5. one ``all_to_all_single`` moves keys (and values) to their owners; a rank
   receives first what rank 0 sends, then rank 1, ...;
6. every rank sorts what it received with a full stable LSD sort
   (``gsort_radix_pairs``, all bits), in its own device memory.

The result: rank r holds a contiguous piece of the sorted sequence, and the
concatenation of the ranks' pieces (rank 0 first) is the stable sort of the
concatenation of their inputs: within one rank the received keys of equal
value are in (source rank, source position) order, which the stable local
passes keep.  Remote keys always land in local device memory (the
collective's receive buffer) before any kernel reads them.

Only 32-bit unsigned keys with optional 32-bit values are handled (the
problem's configurations); float and signed keys map onto this order with the
library's order map first.  The local steps are gsort calls on the rank's own
GPU; ``LocalOps`` lets a test supply host stand-ins for them so that the plan
and the exchange can run on CPU ranks (gloo) without a GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np
import torch

TOP_BITS = (24, 32)   # the digit that defines the buckets
BUCKETS = 256


@dataclass
class Plan:
    """Who owns which buckets, and who sends how many keys to whom.

    owner_start[r] .. owner_start[r + 1] - 1 are the buckets of rank r
    (owner_start has world + 1 entries, 0 first, 256 last); send[s, d] is
    the number of keys rank s sends to rank d; recv_total[d] = send[:, d].sum().
    """
    owner_start: np.ndarray
    send: np.ndarray
    recv_total: np.ndarray


def plan(hists: np.ndarray) -> Plan:
    """The bucket ranges and the send counts from every rank's top-digit counts.

    hists: integer array [world, 256], row s = the counts of rank s's keys
    per top digit.  Rank r's buckets start at the first bucket whose exclusive
    prefix over all keys reaches r * total / world (rank 0 starts at bucket 0,
    the last rank ends at bucket 255); a rank may own no bucket.
    """
    h = np.asarray(hists, dtype=np.int64)
    if h.ndim != 2 or h.shape[1] != BUCKETS or h.shape[0] < 1:
        raise ValueError("hists must be [world, 256]")
    if (h < 0).any():
        raise ValueError("counts must be non-negative")
    world = h.shape[0]
    total_per_bucket = h.sum(axis=0)
    excl = np.concatenate([[0], np.cumsum(total_per_bucket)[:-1]])   # keys before bucket b
    total = int(total_per_bucket.sum())
    owner_start = np.empty(world + 1, dtype=np.int64)
    owner_start[0] = 0
    owner_start[world] = BUCKETS
    for r in range(1, world):
        target = -(-r * total // world)   # ceil(r * total / world)
        # the first bucket whose keys start at or after the target
        b = int(np.searchsorted(excl, target, side="left"))
        owner_start[r] = max(min(b, BUCKETS), owner_start[r - 1])
    send = np.zeros((world, world), dtype=np.int64)
    for d in range(world):
        lo, hi = owner_start[d], owner_start[d + 1]
        send[:, d] = h[:, lo:hi].sum(axis=1)
    return Plan(owner_start=owner_start, send=send, recv_total=send.sum(axis=0))


@dataclass
class LocalOps:
    """The per-rank steps on local data (gsort calls by default).

    top_hist(keys) -> int64 tensor [256] of top-digit counts;
    group(keys, values) -> (keys, values) stably sorted by the top digit;
    sort(keys, values) -> (keys, values) stably sorted by every bit.
    """
    top_hist: Callable
    group: Callable
    sort: Callable


def gsort_ops() -> LocalOps:
    """The local steps as gsort calls on the tensors' CUDA device."""
    from . import gsort

    def top_hist(keys: torch.Tensor) -> torch.Tensor:
        h = gsort.digit_histograms(keys, TOP_BITS[0], TOP_BITS[1])
        return h.reshape(-1)[:BUCKETS].to(torch.int64)

    def group(keys, values):
        return gsort.sort_pairs(keys, values, TOP_BITS[0], TOP_BITS[1])

    def sort(keys, values):
        return gsort.sort_pairs(keys, values, 0, 32)

    return LocalOps(top_hist=top_hist, group=group, sort=sort)


def sort_across_ranks(keys: torch.Tensor, values: Optional[torch.Tensor] = None, *,
                      group=None, ops: Optional[LocalOps] = None):
    """Stable sort of the concatenation (rank order) of every rank's keys.

    keys: 1-D uint32-as-int32 tensor of this rank's shard (any length, 0
    included); values: None or a 1-D 32-bit tensor of the same length.
    Returns (keys, values or None, plan): this rank's piece of the sorted
    sequence.  Collective: every rank of `group` must call it.
    """
    import torch.distributed as dist

    ops = ops or gsort_ops()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if keys.dim() != 1 or (values is not None and values.shape != keys.shape):
        raise ValueError("keys must be 1-D and values, if given, of the same shape")

    # 1-2: top-digit counts of every rank
    h_local = ops.top_hist(keys).to(torch.int64).reshape(1, BUCKETS)
    h_all = [torch.empty_like(h_local) for _ in range(world)]
    dist.all_gather(h_all, h_local, group=group)
    p = plan(torch.cat(h_all).cpu().numpy())

    # 4: keys grouped by bucket, hence by destination rank
    if keys.numel() > 0:
        gk, gv = ops.group(keys, values)
    else:
        gk, gv = keys, values

    # 5: one exchange (the receive buffers are this rank's own memory)
    send = [int(x) for x in p.send[rank]]
    recv = [int(x) for x in p.send[:, rank]]
    rk = torch.empty(sum(recv), dtype=keys.dtype, device=keys.device)
    dist.all_to_all_single(rk, gk.contiguous(), recv, send, group=group)
    rv = None
    if values is not None:
        rv = torch.empty(sum(recv), dtype=values.dtype, device=values.device)
        dist.all_to_all_single(rv, gv.contiguous(), recv, send, group=group)

    # 6: local stable sort of everything received
    if rk.numel() > 0:
        rk, rv = ops.sort(rk, rv)
    return rk, rv, p
