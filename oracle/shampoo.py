"""Owner Shampoo step (oracle, fp64; test infrastructure only).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §5.7:
with each 2D matrix whole on its owner, the owner can run Shampoo — full left / right
preconditioners with an inverse fourth root — instead of Muon, on the same placement.  The
pages name the optimizer and its inverse fourth root, nothing more; this follows the plainest
reading, the original Shampoo update for a matrix parameter:

    L_t = L_{t-1} + G_t G_t^T          (rows x rows),  L_0 = eps I
    R_t = R_{t-1} + G_t^T G_t          (cols x cols),  R_0 = eps I
    P_t = L_t^{-1/4} G_t R_t^{-1/4}
    W_{t+1} = W_t (1 - lr wd) - lr P_t  (decoupled weight decay, as the Muon step)

with G_t the owner's deposited gradient (grad_scale times the sum of the W contributions).
The inverse fourth root is the plain definition: eigendecomposition A = Q diag(lambda) Q^T,
A^{-1/4} = Q diag(lambda^{-1/4}) Q^T.
"""

from __future__ import annotations

from typing import Dict, Sequence

import numpy as np


def inverse_root(a: np.ndarray, p: int = 4) -> np.ndarray:
    """A^{-1/p} of a symmetric positive-definite matrix, by eigendecomposition."""
    a = 0.5 * (np.asarray(a, dtype=np.float64) + np.asarray(a, dtype=np.float64).T)
    lam, q = np.linalg.eigh(a)
    if lam.min() <= 0:
        raise ValueError("matrix is not positive definite")
    return (q * lam ** (-1.0 / p)) @ q.T


def statistics_update(l: np.ndarray, r: np.ndarray, g: np.ndarray):
    """(L + G G^T, R + G^T G)."""
    g = np.asarray(g, dtype=np.float64)
    return l + g @ g.T, r + g.T @ g


def preconditioned(l: np.ndarray, r: np.ndarray, g: np.ndarray) -> np.ndarray:
    """L^{-1/4} G R^{-1/4}."""
    return inverse_root(l) @ np.asarray(g, dtype=np.float64) @ inverse_root(r)


def shampoo_matrix_step(w: np.ndarray, l: np.ndarray, r: np.ndarray,
                        contributions: Sequence[np.ndarray], *, grad_scale: float, lr: float,
                        weight_decay: float) -> Dict[str, np.ndarray]:
    """One owner Shampoo step of one matrix; returns the new W, L, R and the update P."""
    g = sum(np.asarray(c, dtype=np.float64) for c in contributions) * grad_scale
    l, r = statistics_update(l, r, g)
    p = preconditioned(l, r, g)
    w = np.asarray(w, dtype=np.float64) * (1.0 - lr * weight_decay) - lr * p
    return {"W": w, "L": l, "R": r, "P": p, "G": g}


def coupled_newton_inverse_root(a: np.ndarray, p: int = 4, iters: int = 30) -> np.ndarray:
    """A^{-1/p} by the coupled Newton iteration (Guo and Higham, "A Schur–Newton method for
    the matrix p-th root and its inverse", 2006), in fp64: with c = ||A||_F,
        X_0 = c^{-1/p} I,  M_0 = A / c,
        T_k = ((p + 1) I - M_k) / p,  X_{k+1} = X_k T_k,  M_{k+1} = T_k^p M_k.
    M_k -> I and X_k -> A^{-1/p} for SPD A (eigenvalues of M_0 in (0, 1]).  Not the oracle's
    definition of the root (that is the eigendecomposition): a cross-check of the iteration
    the GPU path runs."""
    a = np.asarray(a, dtype=np.float64)
    n = a.shape[0]
    c = float(np.linalg.norm(a))
    x = np.eye(n) * c ** (-1.0 / p)
    m = a / c
    eye = np.eye(n)
    for _ in range(iters):
        t = ((p + 1) * eye - m) / p
        x = x @ t
        m = np.linalg.matrix_power(t, p) @ m
    return x
