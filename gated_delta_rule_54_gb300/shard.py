"""Sharding of independent sequences across ranks (one process per GPU).

Every (sequence, value head) chain of the chunked gated delta rule is
independent in the forward and in the STE backward, so a batch splits across
ranks with no exchange: each rank runs the library on its own sequences.
This module holds only the host-side bookkeeping (no compute).
"""
from __future__ import annotations

import numpy as np


def shard_range(n_units: int, world: int, rank: int):
    """Contiguous, balanced [start, stop) of n_units for this rank."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_packed(cu_seqlens, world: int, rank: int):
    """Split packed sequences into `world` contiguous groups of near-equal
    token counts.  Returns (seq_start, seq_stop, tok_start, tok_stop, local_cu):
    this rank's sequences, their token range in the packed tensors and the
    rank-local cu_seqlens (starting at 0)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu.size - 1
    total = int(cu[-1])
    # sequence boundaries closest to the ideal token split points
    cuts = [0]
    for r in range(1, world):
        target = total * r / world
        i = int(np.searchsorted(cu, target))
        i = min(max(i, cuts[-1]), n)
        if i > 0 and abs(cu[i - 1] - target) <= abs(cu[min(i, n)] - target):
            i = max(i - 1, cuts[-1])
        cuts.append(i)
    cuts.append(n)
    s0, s1 = cuts[rank], cuts[rank + 1]
    t0, t1 = int(cu[s0]), int(cu[s1])
    local = (cu[s0:s1 + 1] - t0).astype(np.int32)
    return s0, s1, t0, t1, local
