"""The owner step with Shampoo or SOAP in place of Muon, end to end, against the oracle.

The tiny owned set (64^2, 64x256, 256x64, 128^2; W = 4 fp32 contributions; a 768-element
tail), three steps through `OwnerSecondOrderStep`: the deposit kernel's reduced gradient
feeds the optimizer, and the oracle takes the same contributions (fp32 values in fp64) through
the plain sum, then `oracle.shampoo` / `oracle.soap`.  Per step and matrix the update
direction (recovered from the weights) is held to 1e-3 relative Frobenius, as in the
optimizers' own parity tests, and the tail to AdamW's 1e-5.

Shampoo runs its roots in split-bf16 with statistics from 1e-3 I: the gradients here are
~2e-2, so with eps = 1e-6 the statistics' eigenvalue ratio would reach ~1e-6, below what
bf16 pairs (~16 significant bits) resolve (the fp32 precision is the one for such statistics).
SOAP starts from seeded statistics Q diag(linspace(0.3, 0.01, d)) Q^T, so that every
eigenvector is determined (gaps >= 1.1e-3 against the solve's 1e-6 lambda_max stopping
threshold), with eps = 1e-3; its eigenbases refresh on steps 1 and 3.
"""

import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import shampoo as oshampoo
from oracle import soap as osoap
from workloads import get_config

pytestmark = pytest.mark.gpu

SHAMPOO_EPS, SOAP_EPS, STEPS = 1e-3, 1e-3, 3


def _rel(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


@pytest.mark.parametrize("optimizer", ["shampoo", "soap"])
def test_owner_step_with_second_order_optimizer(optimizer):
    from matrix_optimizer_owner_gb300 import mfsdp
    from matrix_optimizer_owner_gb300.owner_step import OwnerSecondOrderStep, owned_layout
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl = get_config(0)
    hyper = wl.hyper
    params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
    lay = owned_layout(params, wl.world_size, 0)
    shapes = [(wl.params[i].rows, wl.params[i].cols) for i in lay.matrices]
    step = OwnerSecondOrderStep(shapes, lay.matrix_offsets, lay.n_tail, optimizer=optimizer,
                                device=dev, shampoo_eps=SHAMPOO_EPS, soap_eps=SOAP_EPS,
                                soap_betas=(0.9, 0.95), beta_stats=0.95, refresh_every=2)
    gen = torch.Generator(device=dev)
    gen.manual_seed(31)
    step.weights.copy_(torch.randn(step.base.n, generator=gen, device=dev) * 0.02)
    step.tail_p.copy_(torch.randn(lay.n_tail, generator=gen, device=dev) * 0.02)
    ref = []
    rng = np.random.default_rng(32)
    lo = ro = 0
    for (r, c), off in zip(shapes, lay.matrix_offsets):
        w0 = step.weights[off:off + r * c].double().cpu().numpy().reshape(r, c)
        st = {"W": w0, "M": np.zeros((r, c)), "V": np.zeros((r, c))}
        if optimizer == "shampoo":
            st.update(L=SHAMPOO_EPS * np.eye(r), R=SHAMPOO_EPS * np.eye(c))
        else:
            spd = []
            for d in (r, c):
                q, _ = np.linalg.qr(rng.standard_normal((d, d)))
                spd.append(((q * np.linspace(0.3, 0.01, d)) @ q.T).astype(np.float32))
            step.state["l"][lo:lo + r * r] = torch.from_numpy(spd[0].ravel()).to(dev)
            step.state["r"][ro:ro + c * c] = torch.from_numpy(spd[1].ravel()).to(dev)
            st.update(L=spd[0].astype(np.float64), R=spd[1].astype(np.float64), basis=None)
        lo, ro = lo + r * r, ro + c * c
        ref.append(st)
    tail = {"p": step.tail_p.double().cpu().numpy(), "m": np.zeros(lay.n_tail),
            "v": np.zeros(lay.n_tail)}
    b1, b2 = hyper.adam_betas
    for t in range(1, STEPS + 1):
        contribs = [torch.randn(step.base.n, generator=gen, device=dev) * wl.grad_std
                    for _ in range(wl.W)]
        tails = [torch.randn(lay.n_tail, generator=gen, device=dev) * wl.grad_std
                 for _ in range(wl.W)]
        w_old = step.weights.double().cpu().numpy()
        step.step(contribs, tails, hyper)
        torch.cuda.synchronize()
        assert mfsdp.mfsdp_query_status() == 0
        w_new = step.weights.double().cpu().numpy()
        host = [x.double().cpu().numpy() for x in contribs]
        for (r, c), off, st in zip(shapes, lay.matrix_offsets, ref):
            gs = [h[off:off + r * c].reshape(r, c) for h in host]
            if optimizer == "shampoo":
                o = oshampoo.shampoo_matrix_step(st["W"], st["L"], st["R"], gs,
                                                 grad_scale=hyper.grad_scale, lr=hyper.lr,
                                                 weight_decay=hyper.weight_decay)
                want = o["P"]
                st.update(L=o["L"], R=o["R"])
            else:
                fresh = (t - 1) % 2 == 0
                o = osoap.soap_matrix_step(st["W"], st["L"], st["R"], st["M"], st["V"], gs, t=t,
                                           grad_scale=hyper.grad_scale, lr=hyper.lr,
                                           weight_decay=hyper.weight_decay, beta1=0.9,
                                           beta2=0.95, eps=SOAP_EPS, beta_stats=0.95,
                                           refresh=fresh, basis=st["basis"])
                want = o["N"]
                st.update(L=o["L"], R=o["R"], M=o["M"], V=o["V"],
                          basis=(o["lamL"], o["QL"], o["lamR"], o["QR"]))
            wo = w_old[off:off + r * c].reshape(r, c)
            got = (wo * (1 - hyper.lr * hyper.weight_decay) -
                   w_new[off:off + r * c].reshape(r, c)) / hyper.lr
            assert _rel(got, want) < 1e-3, (optimizer, (r, c), t, _rel(got, want))
            st["W"] = w_new[off:off + r * c].reshape(r, c)
        tg = sum(x.double().cpu().numpy() for x in tails) * hyper.grad_scale
        tail["p"], tail["m"], tail["v"] = oadamw.adamw_step(
            tail["p"], tail["m"], tail["v"], tg, t, hyper.adam_lr, b1, b2, hyper.adam_eps,
            hyper.adam_wd)
        np.testing.assert_allclose(step.tail_p.double().cpu().numpy(), tail["p"], rtol=1e-5,
                                   atol=1e-7)
    step.close()
