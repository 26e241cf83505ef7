"""Parity at the full sizes of the Llama-3-8B share, the skewed batch and the Llama-3-70B share,
over the step counts the workloads state (3, 3 and 5), in the launch configuration
``bench.py`` times (same owned sets, draws and split threshold).

Every step draws fresh seeded contributions on the device and runs the whole owner step.  The
host then replays the oracle on the same inputs:

  * every owned matrix, every step: the oracle's deposit, momentum and Nesterov input over all
    elements (fp64, the momentum buffer carried from step to step), compared element by element
    with the kernel's momentum (1e-5) and its bf16 Newton–Schulz input (one bf16 rounding of
    the fp32 U, 2^-8 of each element, plus the fp32 rounding of the sums that form U, which
    shows only where U nearly cancels; split-precision matrices hi + lo within 1e-5), and the Frobenius
    norm of the oracle's input against the kernel's (1e-5);
  * every owned matrix, every step, sampled elements: the update of the previous step's
    weights with the kernel's own Newton–Schulz output (a check of the update kernel, 1e-5);
  * "trajectory" matrices (one of each shape where the fp64 recursion is affordable): the
    oracle's Newton–Schulz output and weights at every step, within 2e-2 and 1e-3;
  * the largest shapes (8192x28672, 28672x8192, 8192x8192): the oracle's whole fp64
    Newton–Schulz output at the last step, after the momentum buffer has carried every earlier
    step, within 2e-2.  Its weights then differ from the oracle's by at most
    lr * s * ||O - O_ref|| <= lr * s * 2e-2 * ||O||, under 2e-4 of ||W|| at these shapes;
  * the largest shapes at the earlier steps: a property that holds at any size — with v the
    top right singular vector of the kernel's input U (power iteration in fp64),
    NS(U) v = phi(s / (nu + eps)) U v / s, phi the scalar quintic iterated ns_steps times,
    s = ||U v|| (within 3e-2);
  * the AdamW tail in full at every step.

The host keeps one fp64 momentum buffer per owned element (54 GB for the Llama-3-70B share)
and an fp32 bound on the magnitudes that went into it (27 GB), and runs the oracle's
elementwise functions on chunks of each matrix in a thread pool (numpy releases the
interpreter lock inside its loops).
"""

import concurrent.futures as cf
import math
import os
import sys

import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import muon as omuon

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu

N_SAMPLES = 4096
STREAM_TOL = 1e-5
NS_TOL = 2e-2
W_TOL = 1e-3
N_THREADS = os.cpu_count() or 8


def _phi(x, hp):
    for _ in range(hp.ns_steps):
        x = hp.ns_a * x + hp.ns_b * x ** 3 + hp.ns_c * x ** 5
    return x


def _h(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _rel(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def _draw_step(wb, t):
    """The seeded contributions of step t, drawn on the device into the resident buffers."""
    from workloads import synth
    wl, lay = wb.wl, wb.lay
    for w, buf in enumerate(wb.contrib):
        for pi, off, (rr, cc) in zip(lay.matrices, lay.matrix_offsets, wb.shapes):
            buf[off:off + rr * cc] = synth.contribution(wl, t, pi, w, wb.dev)
    for w, buf in enumerate(wb.tail_contrib):
        for pi, off in zip(lay.tails, lay.tail_offsets):
            n = wl.params[pi].numel
            buf[off:off + n] = synth.contribution(wl, t, pi, w, wb.dev)


class _Replay:
    """The oracle's deposit, momentum and Nesterov input for one matrix over all its elements,
    in chunks on a thread pool, with the element-by-element comparison against the kernel."""

    def __init__(self, pool, hp):
        self.pool = pool
        self.hp = hp

    def step(self, B64, Babs, cs_host, mom_host, uhat_host, ulo_host, U_out=None):
        hp = self.hp
        n = B64.size
        nch = max(1, min(2 * N_THREADS, n // 65536))
        bounds = np.linspace(0, n, nch + 1).astype(np.int64)

        def work(j):
            a, b = int(bounds[j]), int(bounds[j + 1])
            cs = [c[a:b].double().numpy() for c in cs_host]
            G = omuon.reduce_contributions(cs, hp.grad_scale)
            B = omuon.momentum_update(B64[a:b], G, hp.momentum)
            B64[a:b] = B
            # the same recursion over magnitudes, mu Babs + (1 - mu) |G|: a bound on every
            # term that went into B, whose fp32 rounding stays in B where B itself cancels
            babs = hp.momentum * Babs[a:b] + (1.0 - hp.momentum) * np.abs(G)
            Babs[a:b] = babs
            U = omuon.nesterov_input(G, B, hp.momentum, hp.nesterov)
            if U_out is not None:
                U_out[a:b] = U
            nsq = omuon.frobenius_norm(U) ** 2
            dB = mom_host[a:b].double().numpy() - B
            Ug = uhat_host[a:b].double().numpy()
            if ulo_host is not None:
                Ug = Ug + ulo_host[a:b].double().numpy()
                u_bad = 0
                dU = Ug - U
                u_err = (float(np.max(np.abs(dU), initial=0.0)), float(np.sum(dU * dU)))
            else:
                # the kernel sums the W contributions, forms B and U in fp32 (each operation
                # within u = 2^-24 of its operands' magnitudes, and B carries the rounding of
                # every earlier step: in all under 2^-20 (sum |g_w| + Babs) for W <= 8 and
                # these step counts, Babs the magnitude recursion above), then rounds U to bf16
                # (half a unit in the last place: at most 2^-8 |U|).  The fp32 part matters
                # only where U or B nearly cancels.
                floor = 2.0 ** -20 * (sum(np.abs(c) for c in cs) + babs)
                bad = np.abs(Ug - U) > 2.0 ** -8 * np.abs(U) + floor
                u_bad = int(np.count_nonzero(bad))
                u_err = (0.0, 0.0)
                if u_bad:
                    e = int(np.flatnonzero(bad)[0])
                    u_err = (float(U[e]), float(Ug[e]), float(floor[e]), float(B[e]),
                             float(babs[e]), [float(c[e]) for c in cs])
            return (nsq, float(np.sum(dB * dB)), float(np.sum(B * B)),
                    float(np.max(np.abs(dB), initial=0.0)), float(np.max(np.abs(B), initial=0.0)),
                    u_bad, u_err, float(np.max(np.abs(U), initial=0.0)), float(np.sum(U * U)))

        parts = list(self.pool.map(work, range(nch)))
        nu = math.sqrt(sum(p[0] for p in parts))
        rel_B = math.sqrt(sum(p[1] for p in parts) / max(sum(p[2] for p in parts), 1e-300))
        max_B = max(p[3] for p in parts) / max(max(p[4] for p in parts), 1e-300)
        u_bad = sum(p[5] for p in parts)
        maxU = max(p[7] for p in parts)
        if u_bad:
            return nu, rel_B, max_B, u_bad, next(p[6] for p in parts if p[5]), None
        rel_U = math.sqrt(sum(p[6][1] for p in parts) / max(sum(p[8] for p in parts), 1e-300))
        max_U = max(p[6][0] for p in parts) / max(maxU, 1e-300)
        return nu, rel_B, max_B, u_bad, rel_U, max_U


def _plan(cfg, shapes):
    """(trajectory matrices, {matrix: steps with a whole fp64 Newton–Schulz check}) of a
    workload: one matrix of each shape whose 5-iteration recursion costs at most 6e12 nominal
    FLOPs runs the oracle's trajectory; one matrix of each larger shape gets the whole recursion
    at the last step."""
    traj, last_ns, seen = [], [], set()
    for k, (r, c) in enumerate(shapes):
        if (r, c) in seen:
            continue
        seen.add((r, c))
        m, n = min(r, c), max(r, c)
        if 5 * (4 * m * m * n + 2 * m ** 3) <= 6e12:
            traj.append(k)
        else:
            last_ns.append(k)
    return traj, last_ns


def _check(cfg):
    import bench
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wb = bench.Workload(cfg, 0, dev)
    r, lay, wl = wb.runner, wb.lay, wb.wl
    hp = wl.hyper
    steps = wl.steps
    d = 1 - hp.lr * hp.weight_decay
    gen = np.random.default_rng(cfg)
    traj, last_ns = _plan(cfg, wb.shapes)
    sizes = [rr * cc for rr, cc in wb.shapes]
    B64 = [np.zeros(n) for n in sizes]
    Babs = [np.zeros(n, dtype=np.float32) for n in sizes]
    W64 = {k: _h(r.weights[lay.matrix_offsets[k]:lay.matrix_offsets[k] + sizes[k]])
           .reshape(wb.shapes[k]) for k in traj}
    samples = [torch.from_numpy(gen.integers(0, n, size=min(N_SAMPLES, n))).to(dev) + off
               for n, off in zip(sizes, lay.matrix_offsets)]
    W_prev = [_h(r.weights[idx]) for idx in samples]
    tail = None
    if lay.n_tail:
        p0 = _h(r.tail_p)
        tail = (p0, np.zeros_like(p0), np.zeros_like(p0))
    checked_full = set()
    with cf.ThreadPoolExecutor(max_workers=N_THREADS) as pool:
        rep = _Replay(pool, hp)
        for t in range(steps):
            _draw_step(wb, t)
            r.step(wb.contrib, wb.tail_contrib, hp)
            torch.cuda.synchronize()
            assert mfsdp.mfsdp_query_status() == 0
            nu_gpu = _h(r.norm)
            for k, ((rows, cols), off) in enumerate(zip(wb.shapes, lay.matrix_offsets)):
                n = sizes[k]
                sl = slice(off, off + n)
                split = r.ortho_lo is not None and 0 < n <= 65536
                full = k in traj or (k in last_ns and t == steps - 1)
                U_full = np.empty(n) if full else None
                nu, rel_B, max_B, u_bad, u_err, max_U = rep.step(
                    B64[k], Babs[k], [c[sl].cpu() for c in wb.contrib], r.momentum[sl].cpu(),
                    r.ns_input[sl].cpu(), r.ns_input_lo[sl].cpu() if split else None, U_full)
                tag = (cfg, t, k, (rows, cols))
                assert abs(nu_gpu[k] - nu) <= STREAM_TOL * nu, (tag, nu_gpu[k], nu)
                assert rel_B <= STREAM_TOL and max_B <= STREAM_TOL, (tag, rel_B, max_B)
                assert u_bad == 0, (tag, u_bad, u_err)
                if split:
                    assert u_err <= STREAM_TOL and max_U <= STREAM_TOL, (tag, u_err, max_U)
                # the update kernel on sampled elements, from the kernel's own NS output
                idx = samples[k]
                O_s = _h(r.ortho[idx])
                if split:
                    O_s = O_s + _h(r.ortho_lo[idx])
                s_upd = omuon.update_scale(rows, cols, hp.lr_adjust)
                W_ref = W_prev[k] * d - hp.lr * s_upd * O_s
                W_now = _h(r.weights[idx])
                np.testing.assert_allclose(W_now, W_ref, rtol=1e-5, atol=1e-7, err_msg=str(tag))
                W_prev[k] = W_now
                if not full and k not in last_ns:
                    continue
                O = _h(r.ortho[sl]).reshape(rows, cols)
                if split:
                    O = O + _h(r.ortho_lo[sl]).reshape(rows, cols)
                if full:
                    U = U_full.reshape(rows, cols)
                    O_ref = omuon.newton_schulz(U, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c,
                                                hp.ns_eps)
                    assert _rel(O, O_ref) < NS_TOL, (tag, _rel(O, O_ref))
                    checked_full.add(k)
                    if k in W64:
                        W64[k] = omuon.apply_update(W64[k], O_ref, hp.lr, hp.weight_decay,
                                                    hp.lr_adjust)
                        Wk = _h(r.weights[sl]).reshape(rows, cols)
                        assert _rel(Wk, W64[k]) < W_TOL, (tag, _rel(Wk, W64[k]))
                    del U, O_ref
                else:
                    U = _h(r.ns_input[sl]).reshape(rows, cols)
                    v = gen.normal(size=cols)
                    v /= np.linalg.norm(v)
                    for _ in range(40):
                        w = U.T @ (U @ v)
                        v = w / np.linalg.norm(w)
                    Uv = U @ v
                    s = float(np.linalg.norm(Uv))
                    pred = _phi(s / (float(nu_gpu[k]) + hp.ns_eps), hp) * Uv / s
                    got = O @ v
                    assert _rel(got, pred) < 3e-2, (tag, _rel(got, pred))
                del O
            if tail is not None:
                b1, b2 = hp.adam_betas
                g = sum(_h(c) for c in wb.tail_contrib) * hp.grad_scale
                tail = oadamw.adamw_step(tail[0], tail[1], tail[2], g, t + 1, hp.adam_lr, b1,
                                         b2, hp.adam_eps, hp.adam_wd)
                for got, ref in zip((r.tail_p, r.tail_m, r.tail_v), tail):
                    assert _rel(_h(got), ref) < STREAM_TOL, (cfg, t)
    assert checked_full == set(traj) | set(last_ns)
    bench.free_workload(wb)


def test_llama3_8b_share_full_size():
    _check(2)


def test_skewed_batch_full_size():
    _check(3)


def test_llama3_70b_share_full_size():
    _check(4)
