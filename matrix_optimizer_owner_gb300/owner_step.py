"""The owner-local optimizer step as a sequence of C-ABI calls over flat device buffers.

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §3 / §4.4:
after the gradient reduction the owner holds each owned 2D gradient whole and runs Muon on it,
and runs AdamW on its packed tail; there is no communication in the step.  This module only
allocates buffers (torch, on the current device), plans ownership through the library's
planner and issues the calls; every arithmetic step runs in the library's kernels.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import torch

from . import mfsdp

# Matrices up to this many elements run Newton–Schulz with split (hi + lo) bf16 operands: for
# them a bf16 Newton–Schulz error (~1e-2) is not small against the weights once the update is a
# sizeable fraction of ||W||, and the split path costs little at these sizes.
DEFAULT_SPLIT_MAX_NUMEL = 65536


@dataclass
class OwnedLayout:
    matrices: List[int]                    # parameter indices, flat-buffer order
    matrix_offsets: List[int]
    tails: List[int]
    tail_offsets: List[int]
    n_matrix: int                          # elements of the flat matrix buffer
    n_tail: int


def owned_layout(params: Sequence[Tuple[int, int, int, bool]], world_size: int, rank: int,
                 policy: int = mfsdp.POLICY_ROLE_GREEDY) -> OwnedLayout:
    """Plan ownership with the library's planner and list what ``rank`` owns."""
    segs, _, _ = mfsdp.mfsdp_plan_owner_set(params, world_size, policy)
    mats = sorted((s["rank_offset"], i) for i, s in enumerate(segs)
                  if s["owner"] == rank and params[i][3])
    tails = sorted((s["rank_offset"], i) for i, s in enumerate(segs)
                   if s["owner"] == rank and not params[i][3])
    nm = sum(segs[i]["numel"] for _, i in mats)
    nt = sum(segs[i]["numel"] for _, i in tails)
    return OwnedLayout([i for _, i in mats], [o for o, _ in mats], [i for _, i in tails],
                       [o for o, _ in tails], nm, nt)


class OwnerStep:
    """Buffers and handle of one owner's step.

    shapes[i] = (rows, cols) of owned matrix i at element offset offsets[i] of the flat
    buffers; n_tail elements of packed tail.
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], offsets: Sequence[int], n_tail: int,
                 split_max_numel: int = DEFAULT_SPLIT_MAX_NUMEL, device=None,
                 n_flat: Optional[int] = None):
        self.device = torch.device(device if device is not None else "cuda")
        dev = self.device
        self.shapes = list(shapes)
        self.offsets = list(offsets)
        n = max([o + r * c for (r, c), o in zip(self.shapes, self.offsets)] + [0])
        self.n = n if n_flat is None else n_flat
        self.oset = mfsdp.OwnerSet([(r, c, o) for (r, c), o in zip(self.shapes, self.offsets)],
                                   split_max_numel)
        split = self.oset.split_count() > 0
        bf = torch.bfloat16
        self.weights = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.momentum = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.ns_input = torch.zeros(self.n, dtype=bf, device=dev)
        self.ortho = torch.zeros(self.n, dtype=bf, device=dev)
        self.ns_input_lo = torch.zeros(self.n, dtype=bf, device=dev) if split else None
        self.ortho_lo = torch.zeros(self.n, dtype=bf, device=dev) if split else None
        self.norm = torch.zeros(max(len(self.shapes), 1), dtype=torch.float32, device=dev)
        self.workspace = torch.empty(self.oset.workspace_bytes(), dtype=torch.uint8, device=dev)
        self.oset.bind(self.workspace, self.ns_input, self.ns_input_lo, self.ortho, self.ortho_lo)
        self.n_tail = n_tail
        self.tail_p = torch.zeros(n_tail, dtype=torch.float32, device=dev)
        self.tail_m = torch.zeros(n_tail, dtype=torch.float32, device=dev)
        self.tail_v = torch.zeros(n_tail, dtype=torch.float32, device=dev)
        self.t = 0

    # -- the four calls of one step -------------------------------------------------------
    def reduce_momentum(self, contribs, hyper, reduced_grad=None, stream=None):
        mfsdp.mfsdp_owner_reduce_momentum(self.oset, contribs, hyper.grad_scale, hyper.momentum,
                                          hyper.nesterov, self.momentum, self.ns_input,
                                          self.ns_input_lo, reduced_grad, self.norm, stream)

    def newton_schulz(self, hyper, stream=None):
        mfsdp.mfsdp_newton_schulz(self.oset, self.ns_input, self.ns_input_lo, self.norm,
                                  hyper.ns_steps, hyper.ns_a, hyper.ns_b, hyper.ns_c,
                                  hyper.ns_eps, self.ortho, self.ortho_lo, stream)

    def apply_update(self, hyper, stream=None):
        mode = mfsdp.LR_ORIGINAL if hyper.lr_adjust == "original" else mfsdp.LR_MATCH_RMS_ADAMW
        mfsdp.mfsdp_apply_update(self.oset, self.weights, self.ortho, self.ortho_lo, hyper.lr,
                                 hyper.weight_decay, mode, stream)

    def adamw_tail(self, tail_contribs, hyper, step, stream=None):
        if self.n_tail == 0:
            return
        b1, b2 = hyper.adam_betas
        mfsdp.mfsdp_adamw_tail(tail_contribs, hyper.grad_scale, self.tail_p, self.tail_m,
                               self.tail_v, step, hyper.adam_lr, b1, b2, hyper.adam_eps,
                               hyper.adam_wd, stream)

    def step(self, contribs, tail_contribs, hyper, reduced_grad=None, stream=None):
        """One whole owner step: deposit + momentum + norm, Newton–Schulz, update, AdamW tail."""
        self.t += 1
        self.reduce_momentum(contribs, hyper, reduced_grad, stream)
        self.newton_schulz(hyper, stream)
        self.apply_update(hyper, stream)
        self.adamw_tail(tail_contribs, hyper, self.t, stream)

    def capture(self, contribs, hyper, reduced_grad=None):
        """Capture deposit + momentum + norm, Newton–Schulz and the update of this owner step
        (18 launches for a bf16 owned set) in one CUDA graph on a side stream, reading the
        given contribution buffers; returns the graph.  The AdamW tail stays outside (its
        bias correction changes every step): ``graph_step`` replays the graph and launches
        it."""
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(self.device)
        with torch.cuda.graph(g):
            stream = torch.cuda.current_stream(self.device)
            self.reduce_momentum(contribs, hyper, reduced_grad, stream)
            self.newton_schulz(hyper, stream)
            self.apply_update(hyper, stream)
        return g

    def graph_step(self, graph, tail_contribs, hyper, stream=None):
        """One owner step through a graph from ``capture`` plus the AdamW tail."""
        self.t += 1
        graph.replay()
        self.adamw_tail(tail_contribs, hyper, self.t, stream)

    def close(self):
        self.oset.close()


class OwnerSecondOrderStep:
    """The same owner placement with Shampoo or SOAP in place of Muon (§5.7: the optimizer is
    swapped while placement and the gradient deposit stay).  One step: the W-way deposit (the
    deposit kernel, whose fp32 reduced-gradient output is the gradient the optimizer reads;
    its momentum and Newton-Schulz outputs go unused), the Shampoo or SOAP step of every owned
    matrix, AdamW on the tail.

    optimizer "shampoo": ``root_iters`` coupled-Newton steps per inverse fourth root,
    ``precision`` mfsdp.SHAMPOO_FP32 or SHAMPOO_SPLIT_BF16, statistics from ``shampoo_eps`` I.
    optimizer "soap": Adam moments with ``soap_betas`` and ``soap_eps``, statistics EMA with
    ``beta_stats``, eigenbases refreshed every ``refresh_every`` steps (1: every step).
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], offsets: Sequence[int], n_tail: int,
                 optimizer: str = "shampoo", device=None, root_iters: int = 30,
                 precision: int = mfsdp.SHAMPOO_SPLIT_BF16, shampoo_eps: float = 1e-6,
                 soap_betas=(0.9, 0.95), beta_stats: float = 0.95, soap_eps: float = 1e-8,
                 refresh_every: int = 1, max_sweeps: int = 20):
        if optimizer not in ("shampoo", "soap"):
            raise ValueError("optimizer must be 'shampoo' or 'soap'")
        self.optimizer = optimizer
        self.base = OwnerStep(shapes, offsets, n_tail, split_max_numel=0, device=device)
        dev = self.base.device
        self.grad = torch.zeros(self.base.n, dtype=torch.float32, device=dev)
        mats = [(r, c, o) for (r, c), o in zip(self.base.shapes, self.base.offsets)]
        self.root_iters, self.precision = root_iters, precision
        self.soap_betas, self.beta_stats, self.soap_eps = soap_betas, beta_stats, soap_eps
        self.refresh_every, self.max_sweeps = max(1, refresh_every), max_sweeps
        if optimizer == "shampoo":
            self.opt = mfsdp.ShampooSet(mats)
            self.ws = torch.empty(max(self.opt.workspace_bytes, 1), dtype=torch.uint8, device=dev)
            self.l = torch.empty(max(self.opt.l_numel, 1), dtype=torch.float32, device=dev)
            self.r = torch.empty(max(self.opt.r_numel, 1), dtype=torch.float32, device=dev)
            self.opt.init_state(shampoo_eps, self.l, self.r, self.ws)
        else:
            self.opt = mfsdp.SoapSet(mats)
            self.ws = torch.empty(max(self.opt.workspace_bytes, 1), dtype=torch.uint8, device=dev)
            self.state = {k: torch.empty(max(n, 1), dtype=torch.float32, device=dev)
                          for k, n in self.opt.state_sizes(self.base.n).items()}
            self.opt.init_state(self.state, self.ws)
        self.t = 0

    @property
    def weights(self):
        return self.base.weights

    @property
    def tail_p(self):
        return self.base.tail_p

    def step(self, contribs, tail_contribs, hyper, stream=None):
        """One owner step: deposit, Shampoo or SOAP on the owned matrices, AdamW on the tail.
        Uses hyper.grad_scale, lr, weight_decay and the AdamW tail settings."""
        self.t += 1
        b = self.base
        b.reduce_momentum(contribs, hyper, self.grad, stream)
        if self.optimizer == "shampoo":
            self.opt.step(self.grad, self.l, self.r, b.weights, hyper.lr, hyper.weight_decay,
                          self.root_iters, self.ws, stream=stream, precision=self.precision)
        else:
            b1, b2 = self.soap_betas
            self.opt.step(self.grad, b.weights, self.state, self.t, lr=hyper.lr, beta1=b1,
                          beta2=b2, beta_stats=self.beta_stats, eps=self.soap_eps,
                          weight_decay=hyper.weight_decay, max_sweeps=self.max_sweeps,
                          workspace=self.ws, stream=stream,
                          refresh=(self.t - 1) % self.refresh_every == 0)
        b.adamw_tail(tail_contribs, hyper, self.t, stream)

    def close(self):
        self.opt.close()
        self.base.close()
