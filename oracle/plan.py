"""Owner planning: roles, greedy owner assignment, segment layout (oracle).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":

* §3 — each data-parallel-sharded 2D weight is whole on one owner rank and empty elsewhere;
  the non-2D tensors of one FSDP unit are packed into one tail role, whole on a tail owner.
* §4.1 — planning sees every FSDP block; each block becomes roles (one per 2D matrix, one
  packed non-2D tail); the greedy load is the numel resident on the owner; RoleGreedy is the
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


# ---------------------------------------------------------------------------------------------
# Resource scorer and the cost-aware policy (§4.1, §4.2).
#
# The pages name the scorer's outputs (per-rank parameter, gradient, optimizer-state,
# communication and workspace estimates) and the CostAware rule (take the ScopeGreedy plan
# when its better balance does not cost more workspace than a cap) but print no formulas.
# Readings, each the plainest one the §4.2 bandwidth model supports:
#
# * parameter / gradient bytes of rank r: its owned numel times the element size;
# * optimizer-state bytes: one momentum buffer per owned matrix element (Muon), two moments
#   per owned tail element (AdamW), at the state element size;
# * communication bytes of rank r for one owner-segment collective over every block
#   (materialise, or gradient reduce: the two move the same bytes in opposite directions):
#   sum over blocks of (W - 1) O_{B,r} sent (its segment to every other rank) plus
#   P_B - O_{B,r} received (everyone else's segments), times the element size;
# * workspace bytes of rank r: the receive buffers of the gradient reduce into its owner
#   segments, (W - 1) O_{B,r} gradient elements, for the block where that is largest;
# * optimizer compute of rank r: nominal Newton–Schulz FLOPs of its owned matrices,
#   steps * (4 m^2 n + 2 m^3) with m = min(rows, cols), n = max(rows, cols);
# * CostAware: plan with RoleGreedy and with ScopeGreedy; take the scope plan if its largest
#   per-rank workspace is at most the cap, else keep the role plan.  A cap <= 0 means the
#   role plan's own largest workspace (the scope plan may not need more).
# ---------------------------------------------------------------------------------------------

COST_AWARE = 2


@dataclass(frozen=True)
class RankResources:
    param_bytes: int
    grad_bytes: int
    state_bytes: int
    comm_bytes: int
    workspace_bytes: int
    optimizer_flops: float


def score_plan(params: Sequence[Param], segs: Sequence[Segment], world_size: int,
               param_bytes: int = 2, grad_bytes: int = 2, state_bytes: int = 4,
               ns_steps: int = 5) -> List[RankResources]:
    """Per-rank resource estimates of a completed plan (§4.1 resource scorer)."""
    W = world_size
    o = block_rank_numel(params, segs, W)
    blocks = block_order(params)
    pb = {b: sum(p.numel for p in params if p.block == b) for b in blocks}
    out = []
    for r in range(W):
        own = [i for i, s in enumerate(segs) if s.owner == r]
        numel = sum(params[i].numel for i in own)
        mat = sum(params[i].numel for i in own if params[i].is_matrix)
        tail = numel - mat
        comm = sum((W - 1) * o[(b, r)] + (pb[b] - o[(b, r)]) for b in blocks) * param_bytes
        ws = max([(W - 1) * o[(b, r)] for b in blocks] + [0]) * grad_bytes
        flops = 0.0
        for i in own:
            p = params[i]
            if p.is_matrix and p.numel > 0:
                m, n = min(p.rows, p.cols), max(p.rows, p.cols)
                flops += ns_steps * (4.0 * m * m * n + 2.0 * m ** 3)
        out.append(RankResources(numel * param_bytes, numel * grad_bytes,
                                 (mat + 2 * tail) * state_bytes, comm, ws, flops))
    return out


def imbalance(values: Sequence[float]) -> float:
    """max / mean over ranks (1 = flat); 0 when every value is 0."""
    tot = float(sum(values))
    return (max(values) / (tot / len(values))) if tot > 0 else 0.0


def plan_cost_aware(params: Sequence[Param], world_size: int, workspace_cap_bytes: int = 0,
                    param_bytes: int = 2, grad_bytes: int = 2, state_bytes: int = 4,
                    ns_steps: int = 5) -> Tuple[List[Segment], int]:
    """CostAware (§4.1): the ScopeGreedy plan if its largest workspace is within the cap,
    else the RoleGreedy plan.  Returns (segments, the policy taken)."""
    role = plan(params, world_size, ROLE_GREEDY)
    scope = plan(params, world_size, SCOPE_GREEDY)
    kw = dict(param_bytes=param_bytes, grad_bytes=grad_bytes, state_bytes=state_bytes,
              ns_steps=ns_steps)
    ws_role = max(x.workspace_bytes for x in score_plan(params, role, world_size, **kw))
    ws_scope = max(x.workspace_bytes for x in score_plan(params, scope, world_size, **kw))
    cap = workspace_cap_bytes if workspace_cap_bytes > 0 else ws_role
    return (scope, SCOPE_GREEDY) if ws_scope <= cap else (role, ROLE_GREEDY)
