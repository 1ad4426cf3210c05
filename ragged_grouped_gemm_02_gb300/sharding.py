"""Expert-parallel sharding of one grouped GEMM across ranks (host logic).

Experts are independent GEMMs ("Grouped GEMM for Imbalanced Experts on
Blackwell: A WIP Worklog", section 2: a tile never crosses an expert
boundary), so a layer's experts split into contiguous ranges, one per GPU,
with no exchange inside the GEMM -- the Pearl article's example runs 32 of
GLM 5.3's 256 experts on each of eight GPUs ("Why MoE needs a grouped GEMM").
Each rank then calls the same grouped GEMM on its own rows, its own slice of
W and offsets rebased to its first row.  The token dispatch around the GEMM
(all-gather / reduce-scatter of activations) is not part of this path.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class ExpertShard:
    rank: int
    expert_begin: int      # first expert of this rank
    expert_end: int        # one past the last
    row_begin: int         # first row of X / Y owned by this rank
    row_end: int
    local_offsets: np.ndarray  # int32 [expert_end - expert_begin + 1], rebased to row_begin


def expert_ranges(E: int, world: int):
    """Contiguous, as-equal-as-possible expert ranges: the first E % world
    ranks get one extra expert."""
    if E < 1 or world < 1:
        raise ValueError("need E >= 1 and world >= 1")
    base, extra = divmod(E, world)
    out, start = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((start, start + n))
        start += n
    return out


def expert_shard(offsets, world: int, rank: int) -> ExpertShard:
    off = np.asarray(offsets, dtype=np.int64)
    E = off.size - 1
    e0, e1 = expert_ranges(E, world)[rank]
    r0, r1 = int(off[e0]), int(off[e1])
    local = (off[e0:e1 + 1] - r0).astype(np.int32)
    return ExpertShard(rank, e0, e1, r0, r1, local)
