"""Parity at the full sizes of the Llama-3-8B share, the skewed batch and the Llama-3-70B share,
in the launch configuration ``bench.py`` times (same owned sets, draws, split threshold).

One optimizer step from zero state, then:
  * every owned matrix: its Frobenius norm against the fp64 sum of its contributions
    (after one step from zero momentum U = (1 - mu)(1 + mu) G, so nu = (1 - mu^2) ||G||);
  * every owned matrix: momentum, NS input and updated weights on sampled elements, against
    the oracle's elementwise formulas (the update from the kernel's own NS output);
  * one matrix of every shape whose fp64 Newton–Schulz costs at most 2e13 FLOPs: the whole
    oracle step (NS within 2e-2, weights within 1e-3);
  * larger shapes: a property that holds at any size — with v the top right singular vector of
    the kernel's input U (power iteration in fp64), NS(U) v = phi(s / (nu + eps)) U v / s,
    phi the scalar quintic iterated ns_steps times, s = ||U v|| (within 3e-2);
  * the AdamW tail in full.
"""

import math
import os
import sys

import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import muon as omuon
from oracle import step as ostep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu

FULL_ORACLE_MAX_FLOPS = 2e13
N_SAMPLES = 4096


def _phi(x, hp):
    for _ in range(hp.ns_steps):
        x = hp.ns_a * x + hp.ns_b * x ** 3 + hp.ns_c * x ** 5
    return x


def _h(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _rel(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def _run(cfg):
    import bench
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wb = bench.Workload(cfg, 0, dev)
    r = wb.runner
    hp = wb.wl.hyper
    W0 = r.weights.clone()
    p0 = r.tail_p.clone() if wb.lay.n_tail else None
    r.step(wb.contrib, wb.tail_contrib, hp)
    torch.cuda.synchronize()
    from matrix_optimizer_owner_gb300 import mfsdp
    assert mfsdp.mfsdp_query_status() == 0
    return wb, W0, p0


def _check(cfg):
    wb, W0, p0 = _run(cfg)
    r, hp, lay = wb.runner, wb.wl.hyper, wb.lay
    mu = hp.momentum
    gen = np.random.default_rng(cfg)
    nu_gpu = _h(r.norm)
    seen = set()
    for k, ((rows, cols), off) in enumerate(zip(wb.shapes, lay.matrix_offsets)):
        n = rows * cols
        sl = slice(off, off + n)
        # the norm of every matrix, from the fp64 sum of its contributions
        G2 = 0.0
        for c0 in range(0, n, 1 << 26):
            c1 = min(n, c0 + (1 << 26))
            g = sum(_h(c[off + c0:off + c1]) for c in wb.contrib) * hp.grad_scale
            G2 += float(np.dot(g, g))
        nu_ref = (1 - mu) * (1 + mu) * math.sqrt(G2)
        assert abs(nu_gpu[k] - nu_ref) <= 1e-5 * nu_ref, (k, nu_gpu[k], nu_ref)
        # sampled elements of the streaming outputs
        idx = torch.from_numpy(gen.integers(0, n, size=min(N_SAMPLES, n))).to(r.device) + off
        g = sum(_h(c[idx]) for c in wb.contrib) * hp.grad_scale
        B_ref = (1 - mu) * g
        U_ref = (1 - mu) * g + mu * B_ref
        np.testing.assert_allclose(_h(r.momentum[idx]), B_ref, rtol=1e-5, atol=1e-6 * np.abs(B_ref).max())
        np.testing.assert_allclose(_h(r.ns_input[idx]), U_ref, rtol=2 ** -8, atol=0)
        s_upd = omuon.update_scale(rows, cols, hp.lr_adjust)
        O_s = _h(r.ortho[idx])
        if r.ortho_lo is not None:
            O_s = O_s + _h(r.ortho_lo[idx])
        W_ref = _h(W0[idx]) * (1 - hp.lr * hp.weight_decay) - hp.lr * s_upd * O_s
        np.testing.assert_allclose(_h(r.weights[idx]), W_ref, rtol=1e-5, atol=1e-7)
        if (rows, cols) in seen:
            continue
        seen.add((rows, cols))
        m, nn = min(rows, cols), max(rows, cols)
        U = _h(r.ns_input[sl]).reshape(rows, cols)
        O = _h(r.ortho[sl]).reshape(rows, cols)
        if r.ortho_lo is not None and 0 < n <= 65536:
            U = U + _h(r.ns_input_lo[sl]).reshape(rows, cols)
            O = O + _h(r.ortho_lo[sl]).reshape(rows, cols)
        if hp.ns_steps * (4 * m * m * nn + 2 * m ** 3) <= FULL_ORACLE_MAX_FLOPS:
            cs = [_h(c[sl]).reshape(rows, cols) for c in wb.contrib]
            ref = ostep.muon_matrix_step(_h(W0[sl]).reshape(rows, cols), np.zeros((rows, cols)),
                                         cs, momentum=mu, nesterov=hp.nesterov,
                                         grad_scale=hp.grad_scale, ns_steps=hp.ns_steps,
                                         a=hp.ns_a, b=hp.ns_b, c=hp.ns_c, eps=hp.ns_eps,
                                         lr=hp.lr, weight_decay=hp.weight_decay,
                                         lr_adjust=hp.lr_adjust)
            assert _rel(O, ref["O"]) < 2e-2, ((rows, cols), _rel(O, ref["O"]))
            Wk = _h(r.weights[sl]).reshape(rows, cols)
            assert _rel(Wk, ref["W"]) < 1e-3, ((rows, cols), _rel(Wk, ref["W"]))
        else:
            v = gen.normal(size=cols)
            v /= np.linalg.norm(v)
            for _ in range(40):
                w = U.T @ (U @ v)
                v = w / np.linalg.norm(w)
            Uv = U @ v
            s = float(np.linalg.norm(Uv))
            pred = _phi(s / (float(nu_gpu[k]) + hp.ns_eps), hp) * Uv / s
            got = O @ v
            assert _rel(got, pred) < 3e-2, ((rows, cols), _rel(got, pred))
    if lay.n_tail:
        b1, b2 = hp.adam_betas
        g = sum(_h(c) for c in wb.tail_contrib) * hp.grad_scale
        p, m_, v_ = oadamw.adamw_step(_h(p0), np.zeros_like(g), np.zeros_like(g), g, 1, hp.adam_lr,
                                      b1, b2, hp.adam_eps, hp.adam_wd)
        for got, ref in ((r.tail_p, p), (r.tail_m, m_), (r.tail_v, v_)):
            assert _rel(_h(got), ref) < 1e-5


def test_llama3_8b_share_full_size():
    _check(2)


def test_skewed_batch_full_size():
    _check(3)


def test_llama3_70b_share_full_size():
    _check(4)
