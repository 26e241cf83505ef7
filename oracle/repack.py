"""Owner-segment repacking (oracle; test infrastructure only).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":

* §4.1 — every parameter has one contiguous local segment on its owner; each FSDP block's
  local shard on rank r holds the block's parameters owned by r (O_{B,r} elements);
* §4.2 — owner-segment collectives move only the nonempty segments;
* §4.4 — reshard load rebuilds every parameter on its canonical [0, numel) axis from the saved
  segments, then repacks it into the target owner assignment and world size.

Layouts, as plain definitions (the pages fix the segments, not how buffers are concatenated;
the reading here is the plainest one):

* canonical buffer: the parameters back to back in declaration order, parameter i at
  sum_{j<i} numel_j;
* owner shard of rank r: the rank's block-local shards back to back in block order (first
  appearance), parameter i at sum_{B' before B} O_{B',r} + local_offset_i.

Packing copies each parameter from its canonical place to its owner's shard, unpacking the
reverse, resharding is unpack under one plan followed by pack under another.  Elements are
copied bit for bit, so the functions work on any numpy dtype.
"""

from __future__ import annotations

from typing import List, Sequence

import numpy as np

from .plan import Param, Segment, block_order


def canonical_offsets(params: Sequence[Param]) -> List[int]:
    out, o = [], 0
    for p in params:
        out.append(o)
        o += p.numel
    return out


def shard_offsets(params: Sequence[Param], segs: Sequence[Segment], world_size: int):
    """(offset of each parameter in its owner's shard, numel of every rank's shard)."""
    blocks = block_order(params)
    o = {(b, r): 0 for b in blocks for r in range(world_size)}
    for p, s in zip(params, segs):
        o[(p.block, s.owner)] += s.numel
    base = {}
    size = [0] * world_size
    for b in blocks:
        for r in range(world_size):
            base[(b, r)] = size[r]
            size[r] += o[(b, r)]
    offs = [base[(p.block, s.owner)] + s.local_offset for p, s in zip(params, segs)]
    return offs, size


def pack(params: Sequence[Param], segs: Sequence[Segment], world_size: int,
         canonical: np.ndarray) -> List[np.ndarray]:
    """Canonical buffer -> every rank's owner shard."""
    coff = canonical_offsets(params)
    soff, size = shard_offsets(params, segs, world_size)
    shards = [np.zeros(n, dtype=canonical.dtype) for n in size]
    for i, (p, s) in enumerate(zip(params, segs)):
        shards[s.owner][soff[i]:soff[i] + p.numel] = canonical[coff[i]:coff[i] + p.numel]
    return shards


def unpack(params: Sequence[Param], segs: Sequence[Segment], world_size: int,
           shards: Sequence[np.ndarray]) -> np.ndarray:
    """Every rank's owner shard -> canonical buffer."""
    coff = canonical_offsets(params)
    soff, _ = shard_offsets(params, segs, world_size)
    total = sum(p.numel for p in params)
    canon = np.zeros(total, dtype=shards[0].dtype if len(shards) else np.uint16)
    for i, (p, s) in enumerate(zip(params, segs)):
        canon[coff[i]:coff[i] + p.numel] = shards[s.owner][soff[i]:soff[i] + p.numel]
    return canon


def reshard(params: Sequence[Param], segs_from: Sequence[Segment], world_from: int,
            shards: Sequence[np.ndarray], segs_to: Sequence[Segment],
            world_to: int) -> List[np.ndarray]:
    """Owner shards under one plan -> owner shards under another (§4.4 reshard load)."""
    return pack(params, segs_to, world_to, unpack(params, segs_from, world_from, shards))
