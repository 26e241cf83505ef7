"""Owner SOAP step (oracle, fp64; test infrastructure only).

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §5.7:
with each 2D matrix whole on its owner, the owner can run SOAP — Adam in the Shampoo
eigenbasis — instead of Muon, on the same placement.  The pages give that one-line
description only.  This follows the plainest reading of it, the SOAP update of Vyas et al.
("SOAP: Improving and Stabilizing Shampoo using Adam", 2024) with the eigenbasis taken
exactly at every step:

    L <- beta_s L + (1 - beta_s) G G^T,  R <- beta_s R + (1 - beta_s) G^T G   (L_0 = R_0 = 0)
    Q_L, Q_R = eigenvectors of L, R, columns in descending eigenvalue order
    M <- beta1 M + (1 - beta1) G                       (first moment, parameter coordinates)
    G' = Q_L^T G Q_R,  M' = Q_L^T M Q_R                (into the eigenbasis)
    V <- beta2 V + (1 - beta2) G'^2                    (second moment, eigenbasis coordinates)
    N' = (M' / (1 - beta1^t)) / (sqrt(V / (1 - beta2^t)) + eps)
    N  = Q_L N' Q_R^T                                  (back to parameter coordinates)
    W <- W (1 - lr wd) - lr N

G is the owner's deposited gradient (grad_scale times the sum of the contributions); t >= 1
counts steps.  SOAP itself refreshes the eigenbasis only every f steps (its preconditioning
frequency); ``refresh=False`` keeps the previous basis for a step, as it does in between.
The eigenvectors are only fixed up to sign, and N does not depend on the
signs: flipping column j of Q_L flips row j of G' and M' and so of N', which Q_L flips back.
Within an eigenspace of a repeated eigenvalue the basis is free; where that eigenspace lies
in the null space of every gradient seen (a rank-deficient L or R), G' and M' vanish there
and N does not depend on the choice either.
"""

from __future__ import annotations

from typing import Dict, Sequence

import numpy as np


def eigenbasis(a: np.ndarray):
    """(eigenvalues, eigenvectors) of a symmetric matrix, in descending eigenvalue order."""
    a = np.asarray(a, dtype=np.float64)
    lam, q = np.linalg.eigh(0.5 * (a + a.T))
    order = np.argsort(-lam, kind="stable")
    return lam[order], q[:, order]


def soap_direction(g, m, v, q_l, q_r, *, t: int, beta1: float, beta2: float, eps: float):
    """Adam in the basis (Q_L, Q_R): returns (N, M', V_new) for the moments after step t.
    ``m`` is the updated first moment (parameter coordinates), ``v`` the previous second
    moment (eigenbasis coordinates)."""
    g_rot = q_l.T @ np.asarray(g, dtype=np.float64) @ q_r
    m_rot = q_l.T @ np.asarray(m, dtype=np.float64) @ q_r
    v_new = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g_rot * g_rot
    n_rot = (m_rot / (1.0 - beta1 ** t)) / (np.sqrt(v_new / (1.0 - beta2 ** t)) + eps)
    return q_l @ n_rot @ q_r.T, m_rot, v_new


def soap_matrix_step(w, l, r, m, v, contributions: Sequence[np.ndarray], *, t: int,
                     grad_scale: float, lr: float, weight_decay: float, beta1: float,
                     beta2: float, eps: float, beta_stats: float, refresh: bool = True,
                     basis=None) -> Dict[str, np.ndarray]:
    """One owner SOAP step of one matrix; returns the new W, L, R, M, V, the eigenbases and
    eigenvalues, and the direction N.

    With ``refresh`` false the eigenbases are not recomputed: ``basis`` = (lam_l, Q_L, lam_r,
    Q_R) from the last refreshing step is used as it stands (SOAP's preconditioning
    frequency: the statistics still accumulate every step)."""
    g = sum(np.asarray(c, dtype=np.float64) for c in contributions) * grad_scale
    l = beta_stats * np.asarray(l, dtype=np.float64) + (1.0 - beta_stats) * (g @ g.T)
    r = beta_stats * np.asarray(r, dtype=np.float64) + (1.0 - beta_stats) * (g.T @ g)
    if refresh:
        lam_l, q_l = eigenbasis(l)
        lam_r, q_r = eigenbasis(r)
    else:
        lam_l, q_l, lam_r, q_r = basis
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    n, _, v = soap_direction(g, m, v, q_l, q_r, t=t, beta1=beta1, beta2=beta2, eps=eps)
    w = np.asarray(w, dtype=np.float64) * (1.0 - lr * weight_decay) - lr * n
    return {"W": w, "L": l, "R": r, "M": m, "V": v, "N": n, "G": g, "QL": q_l, "QR": q_r,
            "lamL": lam_l, "lamR": lam_r}
