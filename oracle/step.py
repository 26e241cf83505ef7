"""Several owner-local optimizer steps over an owned set, float64 (oracle).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §3 and
§4.4: the owner runs Muon on each owned 2D matrix and AdamW on each owned tail; ranks with
empty shards do no work.  Owned matrices are independent of one another, so a step over the
set is the per-matrix step applied to each matrix.  Momentum, AdamW moments start at zero;
the AdamW step counter starts at 1 and is shared by the whole tail.
"""

from __future__ import annotations

from typing import Callable, Dict, List, Sequence

import numpy as np

from . import adamw, muon


def muon_matrix_step(W, B, contribs: Sequence[np.ndarray], *, momentum: float, nesterov: bool,
                     grad_scale: float, ns_steps: int, a: float, b: float, c: float,
                     eps: float, lr: float, weight_decay: float, lr_adjust: str) -> Dict:
    """One Muon step of one owned matrix; returns every intermediate."""
    G = muon.reduce_contributions(contribs, grad_scale)
    B = muon.momentum_update(B, G, momentum)
    U = muon.nesterov_input(G, B, momentum, nesterov)
    nu = muon.frobenius_norm(U)
    O = muon.newton_schulz(U, ns_steps, a, b, c, eps)
    W = muon.apply_update(W, O, lr, weight_decay, lr_adjust)
    return {"G": G, "B": B, "U": U, "nu": nu, "O": O, "W": W}


def muon_trajectory(W0: np.ndarray, contribs_at: Callable[[int], Sequence[np.ndarray]],
                    steps: int, hyper) -> List[Dict]:
    """``steps`` Muon steps of one matrix from W0, zero momentum; contribs_at(t) for t = 0.."""
    W = muon.f64(W0)
    B = np.zeros_like(W)
    out = []
    for t in range(steps):
        r = muon_matrix_step(
            W, B, contribs_at(t), momentum=hyper.momentum, nesterov=hyper.nesterov,
            grad_scale=hyper.grad_scale, ns_steps=hyper.ns_steps, a=hyper.ns_a, b=hyper.ns_b,
            c=hyper.ns_c, eps=hyper.ns_eps, lr=hyper.lr, weight_decay=hyper.weight_decay,
            lr_adjust=hyper.lr_adjust)
        W, B = r["W"], r["B"]
        out.append(r)
    return out


def adamw_trajectory(p0: np.ndarray, contribs_at: Callable[[int], Sequence[np.ndarray]],
                     steps: int, hyper) -> List[Dict]:
    """``steps`` AdamW steps of the packed tail from p0 (t = 1..steps)."""
    p = muon.f64(p0)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    b1, b2 = hyper.adam_betas
    out = []
    for t in range(steps):
        p, m, v = adamw.adamw_tail_step(p, m, v, contribs_at(t), t + 1, hyper.adam_lr, b1, b2,
                                        hyper.adam_eps, hyper.adam_wd, hyper.grad_scale)
        out.append({"p": p, "m": m, "v": v})
    return out
