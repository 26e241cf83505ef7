"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element.

Tolerances (relative, per tensor ||x - y|| / ||y||, plus max-element checks):
  reduced gradient, momentum, norm, AdamW tail ........ 1e-5  (fp32 arithmetic vs fp64)
  Newton–Schulz output, bf16 operands ................. 2e-2  relative Frobenius
  Newton–Schulz output, split (hi + lo) operands ...... 1e-3
  weights after the steps ............................. 1e-3
The NS-only check re-runs the oracle's Newton–Schulz on the exact bf16 input the kernel saw
(and its norm), isolating the GEMM kernels from the rounding of their input.
"""

import numpy as np
import pytest
import torch

from oracle import muon as omuon
from workloads import get_config
from workloads.configs import Hyper

from harness import DeviceRun, case_from_shapes, case_from_workload, max_rel, oracle_matrix, \
    oracle_tail, rel

pytestmark = pytest.mark.gpu

TOL_STREAM = 1e-5
TOL_NS_BF16 = 2e-2
TOL_NS_SPLIT = 1e-3
TOL_W = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_optimizer_owner_gb300 import _lib
    _lib.load()
    torch.cuda.init()


def _split_flags(run):
    smax = run.split_max_numel
    return [0 < r * c <= smax for r, c in run.case.shapes]


def derived_w_tol(ref, t, hp, shape):
    """Weight tolerance implied by the NS bound: W_t - W_ref,t = -sum_tau lr*s*(O - O_ref)
    (times decay factors <= 1), so |dW| <= TOL_NS_BF16 * sum_tau lr*s*||O_ref,tau||."""
    s = omuon.update_scale(shape[0], shape[1], hp.lr_adjust)
    step = sum(hp.lr * s * np.linalg.norm(ref[u]["O"]) for u in range(t + 1))
    return max(TOL_W, 1.25 * TOL_NS_BF16 * step / np.linalg.norm(ref[t]["W"]))


def check_run(run: DeviceRun, init, steps, ns_tol_bf16=TOL_NS_BF16, check_stream=True, mats=None,
              derive_w_tol=False):
    """derive_w_tol: for matrices forced onto bf16 operands whose update is a large fraction of
    the weight (small matrices), bound the weight error by the NS bound instead of 1e-3."""
    c = run.case
    split = _split_flags(run)
    ks = range(len(c.shapes)) if mats is None else mats
    for k in ks:
        rr, cc = c.shapes[k]
        if rr * cc == 0:
            continue
        ref = oracle_matrix(run, init, k, steps)
        for t in range(steps):
            h, o = run.history[t], ref[t]
            if check_stream:
                assert rel(run.mat(h["G"], k), o["G"]) < TOL_STREAM, ("G", k, t)
                assert max_rel(run.mat(h["G"], k), o["G"]) < TOL_STREAM, ("G", k, t)
                assert rel(run.mat(h["B"], k), o["B"]) < TOL_STREAM, ("B", k, t)
                assert max_rel(run.mat(h["B"], k), o["B"]) < TOL_STREAM, ("B", k, t)
                assert abs(h["nu"][k] - o["nu"]) <= TOL_STREAM * o["nu"], ("nu", k, t)
            # Newton–Schulz on exactly the kernel's input
            U = run.mat(h["Uhat"], k)
            O = run.mat(h["O"], k)
            if split[k]:
                U = U + run.mat(h["Uhat_lo"], k)
                O = O + run.mat(h["O_lo"], k)
            hp = c.hyper
            # (the kernel scales by 1/(nu + eps) with nu the norm of the fp32 U; the oracle
            # normalises the rounded input by its own norm: the two differ by ~1e-6 relative)
            O_ref_same_input = omuon.newton_schulz(U, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c,
                                                   hp.ns_eps)
            tol = TOL_NS_SPLIT if split[k] else ns_tol_bf16
            assert rel(O, O_ref_same_input) < tol, ("NS same input", k, t, rel(O, O_ref_same_input))
            # against the oracle's own fp64 trajectory
            assert rel(O, o["O"]) < tol, ("NS", k, t, rel(O, o["O"]))
            # update kernel alone: oracle update from the kernel's W_before and O
            W_unit = omuon.apply_update(run.mat(h["W_before"], k), O, hp.lr, hp.weight_decay,
                                        hp.lr_adjust)
            assert rel(run.mat(h["W"], k), W_unit) < TOL_STREAM, ("update", k, t)
            tol_w = derived_w_tol(ref, t, hp, c.shapes[k]) if (derive_w_tol and not split[k]) \
                else TOL_W
            assert rel(run.mat(h["W"], k), o["W"]) < tol_w, ("W", k, t, rel(run.mat(h["W"], k), o["W"]))
    if c.n_tail and mats is None:
        ref = oracle_tail(run, init, steps)
        for t in range(steps):
            for key in ("p", "m", "v"):
                assert rel(run.history[t][key], ref[t][key]) < TOL_STREAM, (key, t)
                assert max_rel(run.history[t][key], ref[t][key]) < TOL_STREAM, (key, t)


def test_tiny_workload_three_steps():
    wl = get_config(0)
    case = case_from_workload(wl)
    run = DeviceRun(case)
    assert run.runner.oset.split_count() == 4
    init = run.run(wl.steps)
    check_run(run, init, wl.steps)


def test_gpt2_small_workload_three_steps():
    wl = get_config(1)
    case = case_from_workload(wl)
    run = DeviceRun(case)
    assert run.runner.oset.split_count() == 0
    init = run.run(wl.steps)
    check_run(run, init, wl.steps)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_multi_tile_and_ragged_shapes(dtype):
    # several 128 x 256 tiles in every dimension plus ragged tails; tall and wide; K not a
    # multiple of 64; a matrix with m spanning 3 row tiles.
    shapes = [(384, 640), (640, 384), (300, 700), (700, 300), (200, 136), (136, 200),
              (257, 520), (520, 257), (512, 512)]
    run = DeviceRun(case_from_shapes(shapes, W=3, dtype=dtype, grad_std=1e-3, n_tail=1000, seed=3),
                 split_max_numel=0)
    init = run.run(2)
    check_run(run, init, 2, derive_w_tol=True)


def test_unaligned_tiny_and_empty_matrices():
    # offsets not multiples of 8 (pack / unpack path), cols not multiples of 8, m = 1,
    # an empty matrix, and both precisions in one set.
    shapes = [(1, 64), (64, 1), (3, 5), (100, 100), (0, 7), (33, 70), (70, 33), (96, 200),
              (130, 129)]
    run = DeviceRun(case_from_shapes(shapes, W=2, dtype=torch.bfloat16, grad_std=1e-2, n_tail=37,
                                  seed=5, gaps=True), split_max_numel=4000)
    assert 0 < run.runner.oset.split_count() < len(shapes) - 1
    init = run.run(2)
    check_run(run, init, 2, derive_w_tol=True)


def test_heavy_tailed_gradient_scales():
    # per-matrix gradient std from 1e-5 to 1e-1 (the skewed workload's dynamic range)
    shapes = [(128, 512)] * 4 + [(256, 256)] * 2
    stds = [1e-5, 1e-4, 1e-3, 1e-2, 1e-1, 3e-5]
    case = case_from_shapes(shapes, W=4, dtype=torch.bfloat16, seed=7)
    case.grad_std = stds
    run = DeviceRun(case, split_max_numel=0)
    init = run.run(2)
    check_run(run, init, 2, derive_w_tol=True)


def test_non_nesterov_and_match_rms():
    hp = Hyper(nesterov=False, lr_adjust="match_rms_adamw", lr=1e-3, momentum=0.5, ns_steps=2)
    run = DeviceRun(case_from_shapes([(256, 128), (128, 384)], W=2, dtype=torch.bfloat16,
                                  grad_std=1e-3, n_tail=64, seed=9, hyper=hp), split_max_numel=0)
    init = run.run(2)
    check_run(run, init, 2, derive_w_tol=True)


def test_newton_schulz_accuracy_on_gaussian_inputs():
    # Newton–Schulz alone on the kernel's own input, against the fp64 oracle, on Gaussian
    # gradients of ten shapes (tall and wide, ragged, bf16 operands and split ones).  Measured
    # 0.67-0.96 % (bf16, the a X term folded into B' = a I + B) and 2e-5 (split); the bounds
    # sit a quarter above that, inside the 2e-2 and 1e-3 acceptance bounds above.
    shapes = [(768, 2304), (768, 768), (3072, 768), (300, 700), (257, 1000), (1000, 257),
              (520, 520), (96, 400), (200, 300), (1024, 4096)]
    run = DeviceRun(case_from_shapes(shapes, W=1, dtype=torch.float32, grad_std=1e-3,
                                     n_tail=0, seed=13))
    run.run(1)
    split = _split_flags(run)
    assert sum(split) == 2
    h, hp = run.history[0], run.case.hyper
    for k, ((r, c), sp) in enumerate(zip(shapes, split)):
        U = run.mat(h["Uhat"], k)
        O = run.mat(h["O"], k)
        if sp:
            U = U + run.mat(h["Uhat_lo"], k)
            O = O + run.mat(h["O_lo"], k)
        ref = omuon.newton_schulz(U, hp.ns_steps, hp.ns_a, hp.ns_b, hp.ns_c, hp.ns_eps)
        err = rel(O, ref)
        assert err < (1e-4 if sp else 1.2e-2), ((r, c), sp, err)


def test_bitwise_deterministic():
    shapes = [(384, 640), (640, 384), (64, 64)]
    outs = []
    for _ in range(2):
        run = DeviceRun(case_from_shapes(shapes, W=4, dtype=torch.bfloat16, grad_std=1e-3,
                                      n_tail=100, seed=11))
        run.run(2)
        h = run.history[-1]
        outs.append((h["W"], h["nu"], h["O"], h["p"]))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_status_timeout_and_nonfinite():
    from matrix_optimizer_owner_gb300 import mfsdp
    assert mfsdp.mfsdp_query_status() == 0
    mfsdp.mfsdp_selftest_wait_timeout(2_000_000)  # 2 ms: the wait must run out
    assert mfsdp.mfsdp_query_status() == -7
    assert mfsdp.mfsdp_query_status() == 0        # read clears it
    # the context is still usable, and a non-finite gradient is reported
    run = DeviceRun(case_from_shapes([(64, 64)], W=1, dtype=torch.float32))
    contribs, _ = run.contributions(0)
    contribs[0][5] = float("inf")
    run.runner.reduce_momentum(contribs, run.case.hyper)
    assert mfsdp.mfsdp_query_status() == -8
    assert mfsdp.mfsdp_query_status() == 0


def test_argument_errors_on_device():
    from matrix_optimizer_owner_gb300 import mfsdp
    s = mfsdp.OwnerSet([(64, 128, 0)], split_max_numel=0)
    ws = torch.empty(s.workspace_bytes() - 256, dtype=torch.uint8, device="cuda")
    a = torch.zeros(64 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(64 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mfsdp.MfsdpError) as e:
        s.bind(ws, a, None, b, None)
    assert e.value.status == -5
    ws = torch.empty(s.workspace_bytes() + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(mfsdp.MfsdpError) as e:
        s.bind(ws[1:], a, None, b, None)
    assert e.value.status == -3
    with pytest.raises(mfsdp.MfsdpError) as e:
        s.bind(ws, a[1:], None, b, None)
    assert e.value.status == -3
    with pytest.raises(mfsdp.MfsdpError) as e:
        s.bind(ws, a, None, a, None)            # output aliases input
    assert e.value.status == -1
    s.bind(ws, a, None, b, None)
    norm = torch.zeros(1, device="cuda")
    with pytest.raises(mfsdp.MfsdpError) as e:  # not the bound output buffer
        mfsdp.mfsdp_newton_schulz(s, a, None, norm, 5, 3.4445, -4.775, 2.0315, 1e-7, a, None)
    assert e.value.status == -1
