"""AdamW step for the packed non-2D tail, float64 (oracle).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §3: the
non-2D tensors of an FSDP unit are packed into one tail role on a tail owner and stay on the
AdamW path; §4.4: tail-owner shards are routed to AdamW; §5.1: AdamW with lr 1e-3, weight
decay 1e-2, no schedule.  The tail gradient is deposited like a matrix gradient: the sum
of the W rank contributions (times ``grad_scale``).

Per element, step counter t >= 1 (decoupled weight decay, bias-corrected moments):
    p <- p * (1 - lr*wd)
    m <- b1*m + (1-b1)*g
    v <- b2*v + (1-b2)*g^2
    p <- p - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
"""

from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np

from .muon import f64, reduce_contributions


def adamw_step(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, t: int, lr: float,
               beta1: float, beta2: float, eps: float, weight_decay: float
               ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    if t < 1:
        raise ValueError("AdamW step counter starts at 1")
    p, m, v, g = f64(p), f64(m), f64(v), f64(g)
    p = p * (1.0 - lr * weight_decay)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


def adamw_tail_step(p, m, v, contribs: Sequence[np.ndarray], t: int, lr: float, beta1: float,
                    beta2: float, eps: float, weight_decay: float, grad_scale: float = 1.0):
    """Deposit the tail gradient (sum of contributions), then one AdamW step."""
    g = reduce_contributions(contribs, grad_scale)
    return adamw_step(p, m, v, g, t, lr, beta1, beta2, eps, weight_decay)
