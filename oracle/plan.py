"""Owner planning: roles, greedy owner assignment, segment layout (oracle).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":

* §3 — each data-parallel-sharded 2D weight is whole on one owner rank and empty elsewhere;
  the non-2D tensors of one FSDP unit are packed into one tail role, whole on a tail owner.
* §4.1 — planning sees every FSDP block; each block becomes roles (one per 2D matrix, one
  packed non-2D tail); the greedy load is owner-resident numel; RoleGreedy is the
  memory-conservative default and ScopeGreedy pools the roles of all blocks for global
  balance; each block layout must give every parameter one contiguous local segment.
* §4.2 — the bandwidth model gamma_B = max_r O_{B,r} / (P_B / W).

The owner-assignment algorithm itself is not printed on the pages (its listing was lost),
so this follows the plainest reading of the prose:

* blocks are visited in model order (first appearance in declaration order);
* RoleGreedy: within a block, roles go largest first, ties by first declaration index;
  each role goes to the rank with the least cumulative load over all blocks so far, ties
  to the lowest rank id;
* ScopeGreedy: the same rule over all roles pooled, ordered by (numel descending, block
  order, first declaration index);
* layout: in each (block, rank) the owned roles are laid out by first declaration index,
  each role's parameters in declaration order, unpadded — so the tail is one whole
  segment.  The hot path also needs each rank's flat *matrix* buffer (Muon) and flat
  *tail* buffer (AdamW): those take the owned matrices, respectively tail vectors, in
  (block order, declaration order), unpadded.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Sequence, Tuple

ROLE_GREEDY = 0
SCOPE_GREEDY = 1


@dataclass(frozen=True)
class Param:
    rows: int
    cols: int
    block: int
    is_matrix: bool

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Role:
    rid: int
    block: int
    members: Tuple[int, ...]  # parameter indices, declaration order
    numel: int

    @property
    def first(self) -> int:
        return self.members[0]


@dataclass(frozen=True)
class Segment:
    owner: int
    role: int
    local_offset: int  # offset in the owner's block-local shard (mixed matrices + tail)
    rank_offset: int  # offset in the owner's flat matrix buffer, or flat tail buffer
    numel: int


def block_order(params: Sequence[Param]) -> List[int]:
    seen, order = set(), []
    for p in params:
        if p.block not in seen:
            seen.add(p.block)
            order.append(p.block)
    return order


def roles_of(params: Sequence[Param]) -> List[Role]:
    """One role per 2D matrix and one packed tail role per block (§3, §4.1).

    Role ids count blocks in model order and, inside a block, roles by first declaration index.
    """
    roles: List[Role] = []
    for b in block_order(params):
        idx = [i for i, p in enumerate(params) if p.block == b]
        mats = [(i,) for i in idx if params[i].is_matrix]
        tail = tuple(i for i in idx if not params[i].is_matrix)
        groups = mats + ([tail] if tail else [])
        groups.sort(key=lambda g: g[0])
        for g in groups:
            roles.append(Role(len(roles), b, g, sum(params[i].numel for i in g)))
    return roles


def _least_loaded(loads: List[int]) -> int:
    return min(range(len(loads)), key=lambda r: (loads[r], r))


def assign_role_greedy(params: Sequence[Param], world_size: int) -> Dict[int, int]:
    roles = roles_of(params)
    loads = [0] * world_size
    owner: Dict[int, int] = {}
    for b in block_order(params):
        rb = [r for r in roles if r.block == b]
        rb.sort(key=lambda r: (-r.numel, r.first))
        for r in rb:
            o = _least_loaded(loads)
            owner[r.rid] = o
            loads[o] += r.numel
    return owner


def assign_scope_greedy(params: Sequence[Param], world_size: int) -> Dict[int, int]:
    roles = roles_of(params)
    pos = {b: k for k, b in enumerate(block_order(params))}
    loads = [0] * world_size
    owner: Dict[int, int] = {}
    for r in sorted(roles, key=lambda r: (-r.numel, pos[r.block], r.first)):
        o = _least_loaded(loads)
        owner[r.rid] = o
        loads[o] += r.numel
    return owner


def layout(params: Sequence[Param], owner: Dict[int, int], world_size: int) -> List[Segment]:
    """Segment table: where each parameter lives on its owner (§4.1 contiguity rule)."""
    roles = roles_of(params)
    seg: List[Segment] = [None] * len(params)  # type: ignore[list-item]
    mat_off = [0] * world_size
    tail_off = [0] * world_size
    for b in block_order(params):
        local = [0] * world_size
        for r in (r for r in roles if r.block == b):  # already by first declaration index
            o = owner[r.rid]
            for i in r.members:
                p = params[i]
                if p.is_matrix:
                    ro = mat_off[o]
                    mat_off[o] += p.numel
                else:
                    ro = tail_off[o]
                    tail_off[o] += p.numel
                seg[i] = Segment(o, r.rid, local[o], ro, p.numel)
                local[o] += p.numel
    return seg


def plan(params: Sequence[Param], world_size: int, policy: int = ROLE_GREEDY) -> List[Segment]:
    if world_size <= 0:
        raise ValueError("world_size must be positive")
    if policy == ROLE_GREEDY:
        owner = assign_role_greedy(params, world_size)
    elif policy == SCOPE_GREEDY:
        owner = assign_scope_greedy(params, world_size)
    else:
        raise ValueError("unknown policy")
    return layout(params, owner, world_size)


def block_rank_numel(params: Sequence[Param], segs: Sequence[Segment],
                     world_size: int) -> Dict[Tuple[int, int], int]:
    """O_{B,r} in elements: numel of block B resident on rank r (§4.2)."""
    out = {(b, r): 0 for b in block_order(params) for r in range(world_size)}
    for p, s in zip(params, segs):
        out[(p.block, s.owner)] += s.numel
    return out


def rank_loads(segs: Sequence[Segment], world_size: int) -> List[int]:
    loads = [0] * world_size
    for s in segs:
        loads[s.owner] += s.numel
    return loads


def gamma(params: Sequence[Param], segs: Sequence[Segment], world_size: int) -> Dict[int, float]:
    """gamma_B = max_r O_{B,r} / (P_B / W) per block (§4.2); 0 for an empty block."""
    o = block_rank_numel(params, segs, world_size)
    out = {}
    for b in block_order(params):
        pb = sum(p.numel for p in params if p.block == b)
        mx = max(o[(b, r)] for r in range(world_size))
        out[b] = (mx / (pb / world_size)) if pb else 0.0
    return out


def owned(params: Sequence[Param], segs: Sequence[Segment], rank: int):
    """The rank's owned matrices and tail vectors, each sorted by offset in its flat buffer."""
    mats = sorted((s.rank_offset, i) for i, s in enumerate(segs)
                  if s.owner == rank and params[i].is_matrix)
    tails = sorted((s.rank_offset, i) for i, s in enumerate(segs)
                   if s.owner == rank and not params[i].is_matrix)
    return [i for _, i in mats], [i for _, i in tails]
