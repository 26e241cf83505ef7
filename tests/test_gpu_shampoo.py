"""Owner Shampoo on the GPU against the oracle.

Three steps on the tiny owned set (64^2, 64x256, 256x64, 128^2) and one step on one matrix of
every GPT-2-small shape, from the same seeded deposited gradients: the statistics L, R within
1e-5 relative (fp32 sums of fp32 products), the preconditioned update P = L^{-1/4} G R^{-1/4}
within 1e-3 relative Frobenius of the oracle's eigendecomposition roots (the GPU takes the
roots by 30 fp32 coupled-Newton steps; an fp32 emulation of that iteration is 3e-5..3e-4 from
the exact roots on these spectra), and the weights within 1e-6 relative.  P is recovered from
the weights, W_new = W_old (1 - lr wd) - lr P, in fp64.

The split-bf16 precision runs the root iteration and P on the tensor cores with values held
as bf16 pairs (about 16 significant bits each); an emulation of the iteration at that
precision is 0.7e-4..1.2e-4 from the exact roots, so P keeps the same 1e-3 bound.
"""

import numpy as np
import pytest
import torch

from oracle import shampoo as oshampoo

pytestmark = pytest.mark.gpu

LR, WD, EPS, ITERS = 0.02, 0.01, 1e-6, 30


def _rel(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def _run(shapes, steps, seed, precision):
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    offs, o = [], 0
    for r, c in shapes:
        offs.append(o)
        o += r * c
    sset = mfsdp.ShampooSet([(r, c, off) for (r, c), off in zip(shapes, offs)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
    l = torch.empty(sset.l_numel, dtype=torch.float32, device=dev)
    r_ = torch.empty(sset.r_numel, dtype=torch.float32, device=dev)
    sset.init_state(EPS, l, r_, ws)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    w = torch.randn(o, generator=g, device=dev) * 0.02
    w_h = [w.double().cpu().numpy()]
    grads = []
    for t in range(steps):
        gr = torch.randn(o, generator=g, device=dev) * 1e-3
        grads.append(gr.double().cpu().numpy())
        sset.step(gr, l, r_, w, LR, WD, ITERS, ws, precision=precision)
        w_h.append(w.double().cpu().numpy())
    torch.cuda.synchronize()
    assert mfsdp.mfsdp_query_status() == 0
    return offs, grads, w_h, l.double().cpu().numpy(), r_.double().cpu().numpy()


def _check(shapes, steps, seed, precision):
    offs, grads, w_h, l_gpu, r_gpu = _run(shapes, steps, seed, precision)
    lo = ro = 0
    for (rows, cols), off in zip(shapes, offs):
        n = rows * cols
        L, R = EPS * np.eye(rows), EPS * np.eye(cols)
        W = w_h[0][off:off + n].reshape(rows, cols)
        for t in range(steps):
            G = grads[t][off:off + n].reshape(rows, cols)
            out = oshampoo.shampoo_matrix_step(W, L, R, [G], grad_scale=1.0, lr=LR,
                                               weight_decay=WD)
            L, R, W = out["L"], out["R"], out["W"]
            w_old = w_h[t][off:off + n].reshape(rows, cols)
            w_new = w_h[t + 1][off:off + n].reshape(rows, cols)
            p_gpu = (w_old * (1 - LR * WD) - w_new) / LR
            ref = oshampoo.preconditioned(L, R, G)
            assert _rel(p_gpu, ref) < 1e-3, ((rows, cols), t, _rel(p_gpu, ref))
            W = w_new  # continue from the GPU's weights (P is compared step by step)
        assert _rel(l_gpu[lo:lo + rows * rows].reshape(rows, rows), L) < 1e-5
        assert _rel(r_gpu[ro:ro + cols * cols].reshape(cols, cols), R) < 1e-5
        lo += rows * rows
        ro += cols * cols


PRECISIONS = pytest.mark.parametrize("precision", [0, 1], ids=["fp32", "split_bf16"])


@PRECISIONS
def test_tiny_set_three_steps(precision):
    _check([(64, 64), (64, 256), (256, 64), (128, 128)], 3, 1, precision)


@PRECISIONS
def test_ragged_shapes(precision):
    _check([(100, 37), (37, 100), (129, 130), (1, 50), (50, 1)], 2, 2, precision)


@PRECISIONS
def test_ragged_sides_over_several_tiles(precision):
    """Sides of 300 and 520: two and three 256-row tiles of the CTA-pair products, each with
    a ragged last tile (and 64-wide k-blocks with a ragged last one); a side of 257, whose
    second tile has one row, so that the second CTA of its pair lies wholly outside it."""
    _check([(300, 520), (520, 300), (257, 130)], 2, 4, precision)


@PRECISIONS
def test_gpt2_small_shapes_one_step(precision):
    _check([(2304, 768), (768, 768), (3072, 768), (768, 3072)], 1, 3, precision)


@PRECISIONS
def test_empty_set_is_a_no_op(precision):
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    sset = mfsdp.ShampooSet([])
    ws = torch.empty(max(sset.workspace_bytes, 1), dtype=torch.uint8, device="cuda")
    x = torch.zeros(4, device="cuda")
    sset.init_state(EPS, x, x, ws)
    sset.step(x, x, x, x, LR, WD, ITERS, ws, precision=precision)
    torch.cuda.synchronize()
    assert torch.count_nonzero(x) == 0


@PRECISIONS
def test_non_finite_gradient_sets_the_status(precision):
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sset = mfsdp.ShampooSet([(64, 96, 0)])
    ws = torch.empty(sset.workspace_bytes, dtype=torch.uint8, device=dev)
    l = torch.empty(sset.l_numel, device=dev)
    r = torch.empty(sset.r_numel, device=dev)
    sset.init_state(EPS, l, r, ws)
    g = torch.randn(64 * 96, device=dev) * 1e-3
    g[17] = float("nan")
    w = torch.zeros(64 * 96, device=dev)
    assert mfsdp.mfsdp_query_status() == 0
    sset.step(g, l, r, w, LR, WD, ITERS, ws, precision=precision)
    assert mfsdp.mfsdp_query_status() == -8   # MFSDP_ENONFINITE, then cleared
    assert mfsdp.mfsdp_query_status() == 0
