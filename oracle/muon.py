"""Owner-local Muon step for one 2D matrix, float64 (oracle).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":

* §3 / §4.2 — gradient reduction deposits the full 2D gradient on the matrix owner: every
  rank contributes its local full gradient and the reduced result lands in the owner
  segment.  Here the W contributions are summed (scaled by ``grad_scale``; 1/W would give
  the data-parallel average of §5.3).
* §2 — Muon orthogonalises the momentum-buffered gradient by Newton–Schulz steps built from
  products such as X X^T, which couple all rows: the whole matrix is the input.
* §5.1 / §5.3 — the semantics are those of full-matrix Muon (torch.optim.Muon): momentum
  buffer, Nesterov input, decoupled weight decay, a shape-dependent learning-rate scale.

Specification of the step where the pages print no formula:
* momentum (EMA form): B <- mu*B + (1-mu)*G; Nesterov input U = (1-mu)*G + mu*B
  (the updated B); without Nesterov U = B;
* Newton–Schulz, quintic: X = U / (||U||_F + eps); if rows > cols work on X^T; repeat
  ``steps`` times A = X X^T, B = b*A + c*A A, X = a*X + B X; transpose back.
  (a, b, c) = (3.4445, -4.7750, 2.0315), 5 steps, eps = 1e-7 added to the norm;
* update: W <- W * (1 - lr*wd), then W <- W - lr * s(rows, cols) * O with
  s = sqrt(max(1, rows/cols)) ("original") or 0.2*sqrt(max(rows, cols)) ("match_rms_adamw").
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315


def f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def reduce_contributions(contribs: Sequence[np.ndarray], grad_scale: float = 1.0) -> np.ndarray:
    """G = grad_scale * sum_w g_w, in float64."""
    G = np.zeros_like(f64(contribs[0]))
    for g in contribs:
        G = G + f64(g)
    return grad_scale * G


def momentum_update(B: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """B <- mu*B + (1-mu)*G."""
    return mu * f64(B) + (1.0 - mu) * f64(G)


def nesterov_input(G: np.ndarray, B_new: np.ndarray, mu: float, nesterov: bool = True) -> np.ndarray:
    """U = (1-mu)*G + mu*B_new with Nesterov, else U = B_new."""
    if not nesterov:
        return f64(B_new)
    return (1.0 - mu) * f64(G) + mu * f64(B_new)


def frobenius_norm(U: np.ndarray) -> float:
    """nu = ||U||_F = sqrt(sum of squares)."""
    return float(np.sqrt(np.sum(f64(U) ** 2)))


def newton_schulz(U: np.ndarray, steps: int = 5, a: float = NS_A, b: float = NS_B,
                  c: float = NS_C, eps: float = 1e-7) -> np.ndarray:
    """Quintic Newton–Schulz orthogonalisation of one matrix."""
    X = f64(U) / (frobenius_norm(U) + eps)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if transposed else X


def update_scale(rows: int, cols: int, mode: str = "original") -> float:
    if mode == "original":
        return float(np.sqrt(max(1.0, rows / cols)))
    if mode == "match_rms_adamw":
        return 0.2 * float(np.sqrt(max(rows, cols)))
    raise ValueError(mode)


def apply_update(W: np.ndarray, O: np.ndarray, lr: float, weight_decay: float,
                 mode: str = "original") -> np.ndarray:
    """Decoupled weight decay, then the scaled orthogonalised step."""
    W = f64(W)
    rows, cols = W.shape
    W = W * (1.0 - lr * weight_decay)
    return W - lr * update_scale(rows, cols, mode) * f64(O)
