"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against a closed form, an invariant, a library routine used as a
special case (``numpy.linalg.svd``), a hand-worked example or brute force — chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign, a transposed operand, a missing
normalisation) fails at least one of them.  ``test_planted_mistakes_are_caught`` plants such
slips in copies of the oracle's functions and checks that the pins reject them.
"""

import itertools
import math

import numpy as np
import pytest

from oracle import adamw, muon, plan
from oracle import step as ostep
from workloads import get_config

A, B, C = muon.NS_A, muon.NS_B, muon.NS_C


# ----------------------------------------------------------------------------- reduce
def test_reduce_integer_contributions_sum_exactly():
    rng = np.random.default_rng(1)
    ints = [rng.integers(-1000, 1000, size=(7, 5)) for _ in range(8)]
    contribs = [x.astype(np.float64) * 2.0 ** -10 for x in ints]
    exact = sum(x.astype(object) for x in ints)  # Python integers: no rounding at all
    got = muon.reduce_contributions(contribs)
    assert np.array_equal(got * 2 ** 10, np.array(exact, dtype=np.float64))
    got_q = muon.reduce_contributions(contribs, grad_scale=0.25)  # 1/W of W=4: data-parallel mean
    assert np.array_equal(got_q * 2 ** 12, np.array(exact, dtype=np.float64))


# ----------------------------------------------------------------------------- momentum
@pytest.mark.parametrize("mu", [0.95, 0.5])
def test_momentum_constant_gradient_closed_form(mu):
    # With G constant and B_0 = 0: B_t = (1 - mu^t) G and U_t = (1 - mu) G + mu (1 - mu^t) G.
    G = np.random.default_rng(2).normal(size=(4, 3))
    Bm = np.zeros_like(G)
    for t in range(1, 8):
        Bm = muon.momentum_update(Bm, G, mu)
        U = muon.nesterov_input(G, Bm, mu)
        np.testing.assert_allclose(Bm, (1 - mu ** t) * G, rtol=1e-14, atol=0)
        np.testing.assert_allclose(U, ((1 - mu) + mu * (1 - mu ** t)) * G, rtol=1e-14, atol=0)
        np.testing.assert_array_equal(muon.nesterov_input(G, Bm, mu, nesterov=False), Bm)


# ----------------------------------------------------------------------------- Newton–Schulz
def quintic(x, steps=5):
    """The scalar map the matrix iteration applies to each singular value: p(x)=ax+bx^3+cx^5."""
    for _ in range(steps):
        x = A * x + B * x ** 3 + C * x ** 5
    return x


def svd_prediction(U, steps=5, eps=1e-7):
    """NS is an odd matrix polynomial X q(X^T X): it keeps the singular vectors of U and maps
    each normalised singular value sigma/(||U||_F + eps) through the scalar quintic."""
    Us, s, Vt = np.linalg.svd(np.asarray(U, np.float64), full_matrices=False)
    nu = math.sqrt(float(np.sum(s ** 2)))
    return (Us * quintic(s / (nu + eps), steps)) @ Vt


def rel(x, y):
    return float(np.linalg.norm(np.asarray(x) - np.asarray(y)) / np.linalg.norm(np.asarray(y)))


SHAPES = [(1, 1), (1, 7), (7, 1), (5, 5), (6, 9), (9, 6), (16, 40), (40, 16), (64, 64), (33, 70)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("scale", [1e-5, 1.0, 30.0])
def test_newton_schulz_matches_svd_identity(shape, scale):
    U = np.random.default_rng(hash(shape) % 2 ** 32).normal(size=shape) * scale
    assert rel(muon.newton_schulz(U), svd_prediction(U)) < 1e-10


def test_newton_schulz_scalar_and_row_special_cases():
    # phi(1) = p(p(p(p(p(1))))) iterated by hand: 0.701, 1.11362..., 0.72071..., 1.08997..., 0.69644
    assert abs(quintic(1.0) - 0.6964364094697522) < 1e-13
    for u in (2.0, -0.3):
        O = muon.newton_schulz(np.array([[u]]))
        x = abs(u) / (abs(u) + 1e-7)
        assert abs(O[0, 0] - math.copysign(quintic(x), u)) < 1e-13
    x = np.random.default_rng(3).normal(size=(1, 50))
    n = np.linalg.norm(x)
    np.testing.assert_allclose(muon.newton_schulz(x), quintic(n / (n + 1e-7)) * x / n,
                               rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(muon.newton_schulz(x.T), (quintic(n / (n + 1e-7)) * x / n).T,
                               rtol=1e-12, atol=1e-15)


def test_newton_schulz_diagonal_and_orthogonal_cases():
    d = np.array([3.0, -1.0, 0.5, 2.0])
    nu = np.linalg.norm(d)
    O = muon.newton_schulz(np.diag(d))
    np.testing.assert_allclose(np.diag(O), np.sign(d) * quintic(np.abs(d) / (nu + 1e-7)),
                               rtol=1e-12)
    assert np.count_nonzero(O - np.diag(np.diag(O))) == 0
    Q, _ = np.linalg.qr(np.random.default_rng(4).normal(size=(12, 12)))
    k = 7.0
    sig = k / (k * math.sqrt(12) + 1e-7)
    np.testing.assert_allclose(muon.newton_schulz(k * Q), quintic(sig) * Q, rtol=1e-11, atol=1e-14)


def test_newton_schulz_transpose_symmetry_and_band():
    G = np.random.default_rng(5).normal(size=(20, 48))
    np.testing.assert_allclose(muon.newton_schulz(G.T), muon.newton_schulz(G).T, rtol=1e-12,
                               atol=1e-14)
    # For normalised singular values in [0.01, 1] the quintic keeps them in [0.68, 1.14]:
    xs = np.linspace(0.01, 1.0, 2000)
    ys = quintic(xs)
    assert ys.min() > 0.68 and ys.max() < 1.14
    s_out = np.linalg.svd(muon.newton_schulz(G), compute_uv=False)
    s_in = np.linalg.svd(G, compute_uv=False)
    np.testing.assert_allclose(np.sort(s_out), np.sort(quintic(s_in / (np.linalg.norm(G) + 1e-7))),
                               rtol=1e-10)


# ----------------------------------------------------------------------------- update
def test_update_closed_forms():
    rng = np.random.default_rng(6)
    lr, wd = 0.02, 0.01
    for (r, c), s in [((64, 64), 1.0), ((64, 256), 1.0), ((256, 64), 2.0), ((9, 4), 1.5)]:
        W0 = rng.normal(size=(r, c))
        W = W0
        for _ in range(5):
            W = muon.apply_update(W, np.zeros((r, c)), lr, wd)
        np.testing.assert_allclose(W, W0 * (1 - lr * wd) ** 5, rtol=1e-14)
        ones = np.ones((r, c))
        np.testing.assert_allclose(muon.apply_update(W0, ones, lr, wd),
                                   W0 * (1 - lr * wd) - lr * s, rtol=1e-14)


def test_update_scale_match_rms_adamw_hand_values():
    # MatrixFSDP §5.1 runs Muon with the match-RMS-to-AdamW learning-rate adjustment: the step
    # is scaled by 0.2 * sqrt(max(rows, cols)), independent of which side is longer.  Worked by
    # hand: sqrt(256) = 16, sqrt(9) = 3, sqrt(64) = 8, sqrt(2500) = 50, sqrt(1) = 1.
    for (r, c), s in [((256, 64), 3.2), ((64, 256), 3.2), ((9, 4), 0.6), ((4, 9), 0.6),
                      ((64, 64), 1.6), ((100, 2500), 10.0), ((1, 1), 0.2)]:
        assert abs(muon.update_scale(r, c, "match_rms_adamw") - s) <= 1e-15 * s, (r, c)
    # ...and the original scale sqrt(max(1, rows / cols)) on the same shapes
    for (r, c), s in [((256, 64), 2.0), ((64, 256), 1.0), ((9, 4), 1.5), ((4, 9), 1.0),
                      ((64, 64), 1.0), ((100, 2500), 1.0), ((2500, 100), 5.0)]:
        assert abs(muon.update_scale(r, c, "original") - s) <= 1e-15 * s, (r, c)
    # The whole update in that mode, by hand: W0 = 2, O = 1, lr 0.02, wd 0.01, (9, 4):
    # 2 * (1 - 0.0002) - 0.02 * 0.6 = 1.9996 - 0.012 = 1.9876; O = -0.5 on (256, 64):
    # 2 * 0.9998 + 0.02 * 3.2 * 0.5 = 1.9996 + 0.032 = 2.0316.
    W = muon.apply_update(np.full((9, 4), 2.0), np.ones((9, 4)), 0.02, 0.01, "match_rms_adamw")
    np.testing.assert_allclose(W, np.full((9, 4), 1.9876), rtol=1e-14)
    W = muon.apply_update(np.full((256, 64), 2.0), np.full((256, 64), -0.5), 0.02, 0.01,
                          "match_rms_adamw")
    np.testing.assert_allclose(W, np.full((256, 64), 2.0316), rtol=1e-14)


def test_update_scale_ratio_matches_torch_muon():
    """Third-party cross-check of both scales: torch.optim.Muon with weight decay 0 takes the
    same orthogonalised step under either adjustment, so the ratio of its two updates is
    s_match / s_original, whatever its own Newton–Schulz precision."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch.optim, "Muon"):
        pytest.skip("torch.optim.Muon not available")
    rng = np.random.default_rng(9)
    for r, c in [(256, 64), (64, 256), (96, 96)]:
        G = torch.tensor(rng.normal(size=(r, c)), dtype=torch.float32)
        steps = {}
        for mode in ("original", "match_rms_adamw"):
            t = torch.zeros(r, c, requires_grad=True)
            opt = torch.optim.Muon([t], lr=0.01, weight_decay=0.0, adjust_lr_fn=mode)
            t.grad = G.clone()
            opt.step()
            steps[mode] = t.detach().double().numpy()
        ratio = np.linalg.norm(steps["match_rms_adamw"]) / np.linalg.norm(steps["original"])
        want = muon.update_scale(r, c, "match_rms_adamw") / muon.update_scale(r, c, "original")
        assert abs(ratio - want) <= 1e-6 * want, (r, c, ratio, want)


# ----------------------------------------------------------------------------- AdamW
def test_adamw_hand_worked_single_element():
    # p0 = 1, lr 1e-3, wd 1e-2, betas (0.9, 0.95), eps 1e-8; gradients 0.5, -0.25, 0.
    # t=1: m = 0.05, v = 0.0125, m^ = 0.5, v^ = 0.25; p = 0.99999 - 1e-3*0.5/(0.5+1e-8)
    # t=2: m = 0.045-0.025 = 0.02, v = 0.011875+0.003125 = 0.015, m^ = 2/19, v^ = 2/13
    # t=3: m = 0.018, v = 0.01425, m^ = 0.018/0.271, v^ = 0.01425/0.142625
    # (exact decimal arithmetic, 40 digits, rounded here to 17 significant digits)
    expect = [(0.05, 0.0125, 0.99899000002),
              (0.02, 0.015, 0.99871164067875807),
              (0.018, 0.01425, 0.99849152088353600)]
    p, m, v = np.array([1.0]), np.array([0.0]), np.array([0.0])
    for t, (g, (em, ev, ep)) in enumerate(zip([0.5, -0.25, 0.0], expect), start=1):
        p, m, v = adamw.adamw_step(p, m, v, np.array([g]), t, 1e-3, 0.9, 0.95, 1e-8, 1e-2)
        assert m[0] == pytest.approx(em, rel=1e-14)
        assert v[0] == pytest.approx(ev, rel=1e-14)
        assert p[0] == pytest.approx(ep, rel=1e-15)


def test_adamw_first_step_identity():
    # At t = 1 bias correction gives m^ = g and v^ = g^2: the step is lr * g / (|g| + eps).
    rng = np.random.default_rng(7)
    p0, g = rng.normal(size=100), rng.normal(size=100) * 1e-3
    p1, _, _ = adamw.adamw_step(p0, np.zeros(100), np.zeros(100), g, 1, 1e-3, 0.9, 0.95, 1e-8, 1e-2)
    np.testing.assert_allclose(p1, p0 * (1 - 1e-5) - 1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-13)


def test_adamw_matches_torch_adamw_fp64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    p0 = rng.normal(size=64)
    grads = [rng.normal(size=64) * 1e-2 for _ in range(4)]
    t = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([t], lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=1e-2)
    p, m, v = p0, np.zeros(64), np.zeros(64)
    for k, g in enumerate(grads, start=1):
        t.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = adamw.adamw_step(p, m, v, g, k, 1e-3, 0.9, 0.95, 1e-8, 1e-2)
    np.testing.assert_allclose(t.detach().numpy(), p, rtol=1e-12)


def test_muon_matches_torch_muon_cross_check():
    """Third-party cross-check: torch.optim.Muon (its own bf16 Newton–Schulz) on the tiny set."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch.optim, "Muon"):
        pytest.skip("torch.optim.Muon not available")
    rng = np.random.default_rng(9)
    for shape in [(64, 64), (64, 256), (256, 64)]:
        W0 = rng.normal(size=shape) * 0.02
        t = torch.tensor(W0, dtype=torch.float32, requires_grad=True)
        opt = torch.optim.Muon([t], lr=0.02, weight_decay=0.01, momentum=0.95, nesterov=True,
                               adjust_lr_fn="original")
        Wo, Bo = W0, np.zeros(shape)
        for _ in range(3):
            g = rng.normal(size=shape) * 1e-2
            t.grad = torch.tensor(g, dtype=torch.float32)
            opt.step()
            r = ostep.muon_matrix_step(Wo, Bo, [g], momentum=0.95, nesterov=True, grad_scale=1.0,
                                       ns_steps=5, a=A, b=B, c=C, eps=1e-7, lr=0.02,
                                       weight_decay=0.01, lr_adjust="original")
            Wo, Bo = r["W"], r["B"]
            buf = opt.state[t]["momentum_buffer"].numpy()
            assert rel(buf, Bo) < 1e-6
        assert rel(t.detach().numpy() - W0, Wo - W0) < 3e-2


# ----------------------------------------------------------------------------- planted slips
def _ns_variant(kind):
    """A copy of the Newton–Schulz recursion with one deliberate slip."""
    def f(U, steps=5, eps=1e-7):
        X = np.asarray(U, np.float64)
        if kind != "no_norm":
            X = X / (np.linalg.norm(X) + eps)
        tr = X.shape[0] > X.shape[1]
        if tr:
            X = X.T
        for _ in range(steps):
            Am = X.T @ X if kind == "gram_transposed" else X @ X.T
            if kind == "b_sign":
                Bm = -B * Am + C * (Am @ Am)
            elif kind == "drop_c":
                Bm = B * Am
            elif kind == "A_not_A2":
                Bm = B * Am + C * Am
            else:
                Bm = B * Am + C * (Am @ Am)
            X = A * X + (X @ Bm if kind == "XB" else Bm @ X)
        return X.T if tr else X
    return f


@pytest.mark.parametrize("kind", ["b_sign", "drop_c", "A_not_A2", "no_norm", "XB", "gram_transposed"])
def test_planted_mistakes_are_caught(kind):
    U = np.random.default_rng(10).normal(size=(9, 9)) * 0.3
    with np.errstate(over="ignore", invalid="ignore"):  # a wrong sign or no norm diverges
        err = rel(_ns_variant(kind)(U), svd_prediction(U))
    assert not err <= 1e-3, err  # inf or NaN counts as caught
    assert rel(muon.newton_schulz(U), svd_prediction(U)) < 1e-10


def test_planted_momentum_and_adamw_mistakes_are_caught():
    G = np.ones((2, 2))
    mu = 0.95
    Bm = np.zeros_like(G)
    for _ in range(3):
        Bm = mu * Bm + G  # plain accumulation instead of the EMA: closed form rejects it
    assert not np.allclose(Bm, (1 - mu ** 3) * G)
    # bias correction dropped: the first-step identity rejects it
    p0, g = np.array([1.0]), np.array([0.5])
    m = 0.1 * g
    v = 0.05 * g * g
    wrong = p0 * (1 - 1e-5) - 1e-3 * m / (np.sqrt(v) + 1e-8)
    assert abs(wrong[0] - (p0[0] * (1 - 1e-5) - 1e-3 * 0.5 / (0.5 + 1e-8))) > 1e-5


# ----------------------------------------------------------------------------- planner
def _params(wl):
    return [plan.Param(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]


def _check_invariants(params, segs, W):
    roles = plan.roles_of(params)
    # every parameter has an owner; all members of a role share it
    for r in roles:
        assert len({segs[i].owner for i in r.members}) == 1
        assert all(segs[i].role == r.rid for i in r.members)
    # loads sum to the total
    assert sum(plan.rank_loads(segs, W)) == sum(p.numel for p in params)
    # block-local shards and rank buffers are gap-free and non-overlapping; roles contiguous
    for b in plan.block_order(params):
        for r in range(W):
            own = sorted((segs[i].local_offset, segs[i].numel, i) for i, p in enumerate(params)
                         if p.block == b and segs[i].owner == r)
            o = 0
            for off, n, _ in own:
                assert off == o
                o += n
    for r in roles:
        offs = [segs[i].local_offset for i in r.members]
        for a_, b_ in zip(r.members, r.members[1:]):
            assert segs[b_].local_offset == segs[a_].local_offset + segs[a_].numel
        assert offs == sorted(offs)
    for r in range(W):
        for is_mat in (True, False):
            own = sorted((segs[i].rank_offset, segs[i].numel) for i, p in enumerate(params)
                         if segs[i].owner == r and p.is_matrix == is_mat)
            o = 0
            for off, n in own:
                assert off == o
                o += n


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("policy", [plan.ROLE_GREEDY, plan.SCOPE_GREEDY])
def test_plan_invariants_on_workloads(cfg, policy):
    wl = get_config(cfg)
    ps = _params(wl)
    for W in sorted({1, 3, wl.world_size}):
        segs = plan.plan(ps, W, policy)
        _check_invariants(ps, segs, W)
        loads = plan.rank_loads(segs, W)
        # greedy list scheduling: max load <= average + largest role
        biggest = max(r.numel for r in plan.roles_of(ps))
        assert max(loads) <= sum(loads) / W + biggest


def test_plan_hand_worked_single_block():
    # One block: matrices of numel 5, 3, 3, 2 (declaration order) then a tail of 1 + 1.
    ps = [plan.Param(5, 1, 0, True), plan.Param(3, 1, 0, True), plan.Param(3, 1, 0, True),
          plan.Param(2, 1, 0, True), plan.Param(1, 1, 0, False), plan.Param(1, 1, 0, False)]
    # Largest first, least-loaded rank, ties to the lower rank:
    # 5 -> r0 (5,0); 3 -> r1 (5,3); 3 -> r1 (5,6); tail 2 (first index 4) vs matrix 2 (index 3):
    # matrix 2 first -> r0 (7,6); tail 2 -> r1 (7,8).
    segs = plan.plan(ps, 2)
    assert [s.owner for s in segs] == [0, 1, 1, 0, 1, 1]
    # r0 block shard: p0 @0, p3 @5.  r1 block shard: p1 @0, p2 @3, tail p4 @6, p5 @7.
    assert [s.local_offset for s in segs] == [0, 0, 3, 5, 6, 7]
    # rank matrix buffers: r0 = p0, p3 ; r1 = p1, p2 ; r1 tail buffer = p4, p5
    assert [s.rank_offset for s in segs] == [0, 0, 3, 5, 0, 1]


def test_plan_hand_worked_cumulative_blocks():
    # Block 0: one matrix of 4.  Block 1: a matrix of 4 and a tail of 1.  Two ranks.
    # RoleGreedy keeps the global load: b0: 4 -> r0; b1: 4 -> r1; tail 1 -> r0 (tie 4,4 -> r0).
    ps = [plan.Param(2, 2, 0, True), plan.Param(2, 2, 1, True), plan.Param(1, 1, 1, False)]
    assert [s.owner for s in plan.plan(ps, 2)] == [0, 1, 0]
    # ScopeGreedy pools: 4 (b0) -> r0, 4 (b1) -> r1, 1 -> r0: the same here
    assert [s.owner for s in plan.plan(ps, 2, plan.SCOPE_GREEDY)] == [0, 1, 0]
    # Three blocks where pooling changes the answer:
    # numels b0: [3], b1: [2, 2], b2: [3]; RoleGreedy: 3->r0; 2->r1, 2->r1; 3->r1?  loads (3,4):
    # r0 -> (6,4).  ScopeGreedy: 3 (b0)->r0, 3 (b2)->r1, 2->r0? loads (3,3) tie -> r0 (5,3),
    # 2 -> r1 (5,5).
    ps = [plan.Param(3, 1, 0, True), plan.Param(2, 1, 1, True), plan.Param(2, 1, 1, True),
          plan.Param(3, 1, 2, True)]
    assert [s.owner for s in plan.plan(ps, 2)] == [0, 1, 1, 0]
    assert [s.owner for s in plan.plan(ps, 2, plan.SCOPE_GREEDY)] == [0, 0, 1, 1]


def test_scope_greedy_lpt_bound_by_brute_force():
    # Pooled largest-first greedy is LPT: max load <= (4/3 - 1/(3W)) * optimum.
    rng = np.random.default_rng(11)
    for _ in range(40):
        n = int(rng.integers(2, 8))
        W = int(rng.integers(2, 4))
        ps = [plan.Param(int(rng.integers(1, 20)), 1, int(rng.integers(0, 3)), True)
              for _ in range(n)]
        sizes = [p.numel for p in ps]
        best = min(max(sum(s for s, a in zip(sizes, asg) if a == r) for r in range(W))
                   for asg in itertools.product(range(W), repeat=n))
        got = max(plan.rank_loads(plan.plan(ps, W, plan.SCOPE_GREEDY), W))
        assert got <= (4 / 3 - 1 / (3 * W)) * best + 1e-9


def test_plan_llama3_8b_rank0_share():
    """Regression against an independent computation of the 8-rank Llama-3-8B plan."""
    wl = get_config(2)
    ps = _params(wl)
    segs = plan.plan(ps, 8)
    loads = plan.rank_loads(segs, 8)
    assert [round(x / 1e6, 1) for x in loads] == [859.9, 868.2, 889.2, 859.9, 893.4, 864.1,
                                                  855.7, 889.2]
    mats, tails = plan.owned(ps, segs, 0)
    assert len(mats) == 28 and len(tails) == 6
    flat = plan.plan(ps, 8, plan.SCOPE_GREEDY)
    assert len(set(plan.rank_loads(flat, 8))) == 1


def test_gamma_model():
    # gamma_B = max_r O_{B,r} / (P_B / W): one owner holding everything gives W; even gives 1.
    ps = [plan.Param(4, 4, 0, True)]
    segs = plan.plan(ps, 4)
    assert plan.gamma(ps, segs, 4)[0] == pytest.approx(4.0)
    ps = [plan.Param(4, 4, 0, True) for _ in range(4)]
    assert plan.gamma(ps, plan.plan(ps, 4), 4)[0] == pytest.approx(1.0)


def test_score_plan_hand_worked():
    # One block: matrices 4x2 (8) and 2x3 (6), then a tail vector of 5.  Two ranks, RoleGreedy:
    # 8 -> r0; 6 -> r1; tail 5 -> r1 (6 < 8): O_{B,0} = 8, O_{B,1} = 11, P_B = 19.
    ps = [plan.Param(4, 2, 0, True), plan.Param(2, 3, 0, True), plan.Param(5, 1, 0, False)]
    segs = plan.plan(ps, 2)
    assert [s.owner for s in segs] == [0, 1, 1]
    r0, r1 = plan.score_plan(ps, segs, 2, param_bytes=2, grad_bytes=2, state_bytes=4,
                             ns_steps=5)
    # params/grads: owned numel x 2 B; state: matrices x 4 B + tail x 2 moments x 4 B
    assert (r0.param_bytes, r0.grad_bytes, r0.state_bytes) == (16, 16, 32)
    assert (r1.param_bytes, r1.grad_bytes, r1.state_bytes) == (22, 22, 64)
    # one collective: send (W-1) O + receive P - O, x 2 B: r0 (8 + 11) * 2, r1 (11 + 8) * 2
    assert r0.comm_bytes == 38 and r1.comm_bytes == 38
    # reduce receive buffers (W-1) O x 2 B
    assert r0.workspace_bytes == 16 and r1.workspace_bytes == 22
    # Newton-Schulz: 4x2 -> m=2, n=4: 5 (4*4*4 + 2*8) = 400; 2x3 -> m=2, n=3: 5 (48 + 16) = 320
    assert r0.optimizer_flops == 400.0 and r1.optimizer_flops == 320.0
    assert plan.gamma(ps, segs, 2)[0] == pytest.approx(22 / 19)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_score_plan_sums_over_ranks(cfg):
    wl = get_config(cfg)
    ps = _params(wl)
    total = sum(p.numel for p in ps)
    mats = sum(p.numel for p in ps if p.is_matrix)
    nominal = sum(5 * (4 * min(p.rows, p.cols) ** 2 * max(p.rows, p.cols)
                       + 2 * min(p.rows, p.cols) ** 3) for p in ps if p.is_matrix)
    for W in (1, 3, 8):
        for pol in (plan.ROLE_GREEDY, plan.SCOPE_GREEDY):
            sc = plan.score_plan(ps, plan.plan(ps, W, pol), W)
            assert sum(x.param_bytes for x in sc) == 2 * total
            assert sum(x.state_bytes for x in sc) == 4 * (mats + 2 * (total - mats))
            # every block's elements are sent W-1 times and received W-1 times in all
            assert sum(x.comm_bytes for x in sc) == 2 * (W - 1) * total * 2
            assert sum(x.optimizer_flops for x in sc) == pytest.approx(nominal, rel=1e-12)
            if W == 1:
                assert all(x.comm_bytes == 0 and x.workspace_bytes == 0 for x in sc)


def test_cost_aware_takes_scope_only_within_the_cap():
    wl = get_config(2)
    ps = _params(wl)
    role = plan.plan(ps, 8, plan.ROLE_GREEDY)
    scope = plan.plan(ps, 8, plan.SCOPE_GREEDY)
    ws_role = max(x.workspace_bytes for x in plan.score_plan(ps, role, 8))
    ws_scope = max(x.workspace_bytes for x in plan.score_plan(ps, scope, 8))
    assert ws_scope > ws_role  # pooling stacks more of one block on a rank
    assert plan.plan_cost_aware(ps, 8) == (role, plan.ROLE_GREEDY)
    assert plan.plan_cost_aware(ps, 8, ws_scope) == (scope, plan.SCOPE_GREEDY)
    assert plan.plan_cost_aware(ps, 8, ws_scope - 1) == (role, plan.ROLE_GREEDY)
    # a flatter plan with no workspace cost is taken
    same = [plan.Param(4, 4, b, True) for b in range(6)]
    assert plan.plan_cost_aware(same, 3)[1] == plan.SCOPE_GREEDY
    assert plan.imbalance([2.0, 2.0]) == 1.0 and plan.imbalance([3.0, 1.0]) == 1.5


# ----------------------------------------------------------------------------- repacking
def test_repack_hand_worked_layout():
    from oracle import repack
    # block 0: m0 4x2 (8) -> r0, m1 2x3 (6) -> r1, tail 5 -> r1; block 1: m3 3x3 (9) -> r0
    # (loads 8 < 11), tail 2 -> r1.  Shards: r0 = [m0 | m3], r1 = [m1, tail0 | tail1].
    ps = [plan.Param(4, 2, 0, True), plan.Param(2, 3, 0, True), plan.Param(5, 1, 0, False),
          plan.Param(3, 3, 1, True), plan.Param(2, 1, 1, False)]
    segs = plan.plan(ps, 2)
    assert [s.owner for s in segs] == [0, 1, 1, 0, 1]
    offs, size = repack.shard_offsets(ps, segs, 2)
    assert offs == [0, 0, 6, 8, 11] and size == [17, 13]
    canon = np.arange(30, dtype=np.int32)
    r0, r1 = repack.pack(ps, segs, 2, canon)
    assert r0.tolist() == list(range(0, 8)) + list(range(19, 28))
    assert r1.tolist() == list(range(8, 14)) + list(range(14, 19)) + list(range(28, 30))


@pytest.mark.parametrize("cfg", [0, 1])
def test_repack_round_trips(cfg):
    from oracle import repack
    ps = _params(get_config(cfg))
    total = sum(p.numel for p in ps)
    canon = np.random.default_rng(cfg).integers(0, 1 << 16, size=total).astype(np.uint16)
    for W in (1, 3, 8):
        segs = plan.plan(ps, W)
        shards = repack.pack(ps, segs, W, canon)
        assert sum(len(s) for s in shards) == total
        assert np.array_equal(repack.unpack(ps, segs, W, shards), canon)
    # reshard 8 -> 3 ranks under another policy equals packing the canonical buffer directly
    a = plan.plan(ps, 8, plan.ROLE_GREEDY)
    b = plan.plan(ps, 3, plan.SCOPE_GREEDY)
    out = repack.reshard(ps, a, 8, repack.pack(ps, a, 8, canon), b, 3)
    for x, y in zip(out, repack.pack(ps, b, 3, canon)):
        assert np.array_equal(x, y)


# ----------------------------------------------------------------------------- Shampoo
def test_shampoo_inverse_root_closed_forms():
    from oracle import shampoo
    lam = np.array([16.0, 1.0, 1e-4, 81.0])
    np.testing.assert_allclose(shampoo.inverse_root(np.diag(lam)), np.diag(lam ** -0.25),
                               rtol=1e-12)
    rng = np.random.default_rng(4)
    q, _ = np.linalg.qr(rng.normal(size=(6, 6)))
    lam = rng.uniform(1e-3, 10.0, size=6)
    a = (q * lam) @ q.T
    x = shampoo.inverse_root(a)
    np.testing.assert_allclose(x, (q * lam ** -0.25) @ q.T, rtol=1e-10, atol=1e-12)
    # X^4 A = I, and the square root variant is different (a planted -1/2 fails the pin)
    np.testing.assert_allclose(np.linalg.matrix_power(x, 4) @ a, np.eye(6), atol=1e-9)
    assert not np.allclose(shampoo.inverse_root(a, p=2) @ shampoo.inverse_root(a, p=2) @
                           shampoo.inverse_root(a, p=2) @ shampoo.inverse_root(a, p=2) @ a,
                           np.eye(6), atol=1e-3)


def test_shampoo_scalar_step_closed_form():
    # 1 x 1: L = R = eps + g^2, P = g / sqrt(eps + g^2); W = W (1 - lr wd) - lr P
    from oracle import shampoo
    eps, g, w = 1e-4, 0.03, 0.5
    out = shampoo.shampoo_matrix_step(np.array([[w]]), np.array([[eps]]), np.array([[eps]]),
                                      [np.array([[g / 2]]), np.array([[g / 2]])],
                                      grad_scale=1.0, lr=0.1, weight_decay=0.01)
    assert out["L"][0, 0] == pytest.approx(eps + g * g, rel=1e-14)
    assert out["P"][0, 0] == pytest.approx(g / math.sqrt(eps + g * g), rel=1e-12)
    assert out["W"][0, 0] == pytest.approx(w * (1 - 0.1 * 0.01) - 0.1 * g / math.sqrt(eps + g * g),
                                           rel=1e-12)


def test_shampoo_rank_one_and_orthogonal_invariance():
    from oracle import shampoo
    rng = np.random.default_rng(6)
    # G = s u v^T: L = eps I + s^2 u u^T, R = eps I + s^2 v v^T, so
    # P = s (eps + s^2)^{-1/2} u v^T exactly.
    u = rng.normal(size=5); u /= np.linalg.norm(u)
    v = rng.normal(size=7); v /= np.linalg.norm(v)
    s, eps = 0.2, 1e-3
    g = s * np.outer(u, v)
    l, r = shampoo.statistics_update(eps * np.eye(5), eps * np.eye(7), g)
    np.testing.assert_allclose(shampoo.preconditioned(l, r, g),
                               s / math.sqrt(eps + s * s) * np.outer(u, v), atol=1e-12)
    # rotating G on both sides rotates P the same way
    g = rng.normal(size=(5, 7))
    qa, _ = np.linalg.qr(rng.normal(size=(5, 5)))
    qb, _ = np.linalg.qr(rng.normal(size=(7, 7)))
    p1 = shampoo.preconditioned(*shampoo.statistics_update(eps * np.eye(5), eps * np.eye(7), g), g)
    g2 = qa @ g @ qb
    p2 = shampoo.preconditioned(*shampoo.statistics_update(eps * np.eye(5), eps * np.eye(7), g2),
                                g2)
    np.testing.assert_allclose(p2, qa @ p1 @ qb, atol=1e-10)


def test_coupled_newton_root_matches_the_definition():
    from oracle import shampoo
    rng = np.random.default_rng(8)
    for n, spread in ((8, 1e-2), (20, 1e-6), (33, 1e-8)):
        q, _ = np.linalg.qr(rng.normal(size=(n, n)))
        lam = np.exp(rng.uniform(np.log(spread), 0.0, size=n))
        a = (q * lam) @ q.T
        x = shampoo.coupled_newton_inverse_root(a, iters=30)
        ref = shampoo.inverse_root(a)
        assert np.linalg.norm(x - ref) / np.linalg.norm(ref) < 1e-9, n


# ----------------------------------------------------------------------------- SOAP
SOAP_HYPER = dict(grad_scale=1.0, lr=1e-3, weight_decay=1e-2, beta1=0.9, beta2=0.95, eps=1e-8,
                  beta_stats=0.95)


def _soap_run(gs, w0, **over):
    from oracle import soap
    h = dict(SOAP_HYPER, **over)
    rows, cols = gs[0].shape
    st = {"W": w0, "L": np.zeros((rows, rows)), "R": np.zeros((cols, cols)),
          "M": np.zeros((rows, cols)), "V": np.zeros((rows, cols))}
    outs = []
    for t, g in enumerate(gs, start=1):
        st = soap.soap_matrix_step(st["W"], st["L"], st["R"], st["M"], st["V"], [g], t=t, **h)
        outs.append(st)
    return outs


def test_soap_scalar_is_the_hand_worked_adamw_run():
    # 1 x 1: the eigenbasis is +-1, so SOAP is AdamW on the single element; p0 = 1,
    # lr 1e-3, wd 1e-2, betas (0.9, 0.95), eps 1e-8, gradients 0.5, -0.25, 0 (fp64 by hand)
    outs = _soap_run([np.array([[0.5]]), np.array([[-0.25]]), np.array([[0.0]])],
                     np.array([[1.0]]))
    expect = [(0.05, 0.0125, 0.99899000002), (0.02, 0.015, 0.99871164067875817),
              (0.018, 0.01425, 0.9984915208835361)]
    for o, (m, v, p) in zip(outs, expect):
        assert o["M"][0, 0] == pytest.approx(m, rel=1e-12)
        assert o["V"][0, 0] == pytest.approx(v, rel=1e-12)
        assert o["W"][0, 0] == pytest.approx(p, rel=1e-13)


def test_soap_diagonal_gradients_are_elementwise_adamw():
    # diagonal G with |g_11| > |g_22| > |g_33| at every step: L and R stay diagonal in that
    # order, the eigenbases are signed identities, and each diagonal entry runs its own AdamW
    # (the independent coordinate-wise oracle); off-diagonal entries only decay
    rng = np.random.default_rng(21)
    gs = [np.diag(np.array([3.0, 2.0, 1.0]) * rng.uniform(0.5, 0.6, 3) *
                  rng.choice([-1.0, 1.0], 3)) for _ in range(4)]
    w0 = rng.normal(size=(3, 3))
    outs = _soap_run(gs, w0)
    p, m, v = np.diag(w0).copy(), np.zeros(3), np.zeros(3)
    for t, (g, o) in enumerate(zip(gs, outs), start=1):
        p, m, v = adamw.adamw_step(p, m, v, np.diag(g), t, 1e-3, 0.9, 0.95, 1e-8, 1e-2)
        np.testing.assert_allclose(np.diag(o["W"]), p, rtol=1e-12)
        off = ~np.eye(3, dtype=bool)
        np.testing.assert_allclose(o["W"][off], w0[off] * (1 - 1e-5) ** t, rtol=1e-12)


def test_soap_rank_one_closed_form():
    # first step, G = s u v^T (unit u, v): the top eigenvectors are +-u and +-v, G' = +-s e1 e1^T,
    # N' = +-s / (s + eps) at (1, 1) and 0 elsewhere, so N = s / (s + eps) u v^T
    from oracle import soap
    rng = np.random.default_rng(22)
    u = rng.normal(size=5); u /= np.linalg.norm(u)
    v = rng.normal(size=7); v /= np.linalg.norm(v)
    s, eps = 0.2, 1e-3
    o = _soap_run([s * np.outer(u, v)], np.zeros((5, 7)), eps=eps)[0]
    np.testing.assert_allclose(o["N"], s / (s + eps) * np.outer(u, v), atol=1e-12)
    assert o["lamL"][0] == pytest.approx(0.05 * s * s, rel=1e-12)
    assert np.all(np.diff(o["lamL"]) <= 0) and np.all(np.diff(o["lamR"]) <= 0)


def test_soap_orthogonal_equivariance_and_transpose():
    # G -> A G B^T (A, B orthogonal) for every step and W0 -> A W0 B^T: W, M rotate the same
    # way, L -> A L A^T, R -> B R B^T, and V (eigenbasis coordinates) is unchanged.  G -> G^T
    # swaps L and R and transposes W, M and V.
    rng = np.random.default_rng(23)
    gs = [rng.normal(size=(5, 7)) * 1e-2 for _ in range(3)]
    w0 = rng.normal(size=(5, 7))
    a, _ = np.linalg.qr(rng.normal(size=(5, 5)))
    b, _ = np.linalg.qr(rng.normal(size=(7, 7)))
    base = _soap_run(gs, w0, eps=1e-6)
    rot = _soap_run([a @ g @ b.T for g in gs], a @ w0 @ b.T, eps=1e-6)
    tr = _soap_run([g.T for g in gs], w0.T, eps=1e-6)
    for o, orot, otr in zip(base, rot, tr):
        np.testing.assert_allclose(orot["W"], a @ o["W"] @ b.T, atol=1e-10)
        np.testing.assert_allclose(orot["M"], a @ o["M"] @ b.T, atol=1e-12)
        np.testing.assert_allclose(orot["L"], a @ o["L"] @ a.T, atol=1e-12)
        np.testing.assert_allclose(orot["V"], o["V"], rtol=1e-8, atol=1e-16)
        np.testing.assert_allclose(otr["W"], o["W"].T, atol=1e-10)
        np.testing.assert_allclose(otr["V"], o["V"].T, rtol=1e-8, atol=1e-16)
        np.testing.assert_allclose(otr["L"], o["R"], atol=1e-12)


def test_soap_direction_ignores_eigenvector_signs():
    from oracle import soap
    rng = np.random.default_rng(24)
    g, m, v = rng.normal(size=(4, 6)), rng.normal(size=(4, 6)), rng.uniform(size=(4, 6))
    ql, _ = np.linalg.qr(rng.normal(size=(4, 4)))
    qr, _ = np.linalg.qr(rng.normal(size=(6, 6)))
    kw = dict(t=3, beta1=0.9, beta2=0.95, eps=1e-8)
    n1, _, v1 = soap.soap_direction(g, m, v, ql, qr, **kw)
    sl, sr = np.array([1, -1, -1, 1]), np.array([-1, 1, 1, 1, -1, 1])
    n2, _, v2 = soap.soap_direction(g, m, v, ql * sl, qr * sr, **kw)
    np.testing.assert_allclose(n2, n1, atol=1e-12)
    np.testing.assert_allclose(v2, v1, rtol=1e-14)


def test_planted_soap_mistakes_are_caught():
    # back-rotation without the transpose, and the second moment kept in parameter
    # coordinates: both fail the rank-one closed form
    rng = np.random.default_rng(25)
    u = rng.normal(size=5); u /= np.linalg.norm(u)
    v = rng.normal(size=7); v /= np.linalg.norm(v)
    s, eps = 0.2, 1e-3
    g = s * np.outer(u, v)
    from oracle import soap
    _, ql = soap.eigenbasis(g @ g.T)
    _, qr = soap.eigenbasis(g.T @ g)
    want = s / (s + eps) * np.outer(u, v)
    n_rot = (ql.T @ g @ qr) / (np.abs(ql.T @ g @ qr) + eps)
    assert np.abs(ql @ n_rot @ qr - want).max() > 1e-2                  # Q_R instead of Q_R^T
    assert np.abs(ql @ n_rot @ qr.T - want).max() < 1e-12
    n_param = g / (np.abs(g) + eps)                                       # Adam in W coordinates
    assert np.abs(n_param - want).max() > 1e-2


def test_soap_without_refresh_keeps_the_basis():
    # refresh=False with the basis of the previous step is the same step as refresh=True when
    # the statistics' eigenvectors do not move (diagonal statistics in a fixed order), and
    # otherwise uses exactly the given basis
    from oracle import soap
    rng = np.random.default_rng(26)
    gs = [np.diag(np.array([3.0, 2.0, 1.0]) * rng.uniform(0.5, 0.6, 3)) for _ in range(2)]
    h = dict(SOAP_HYPER)
    o1 = soap.soap_matrix_step(np.eye(3), np.zeros((3, 3)), np.zeros((3, 3)), np.zeros((3, 3)),
                               np.zeros((3, 3)), [gs[0]], t=1, **h)
    basis = (o1["lamL"], o1["QL"], o1["lamR"], o1["QR"])
    a = soap.soap_matrix_step(o1["W"], o1["L"], o1["R"], o1["M"], o1["V"], [gs[1]], t=2, **h)
    b = soap.soap_matrix_step(o1["W"], o1["L"], o1["R"], o1["M"], o1["V"], [gs[1]], t=2,
                              refresh=False, basis=basis, **h)
    np.testing.assert_allclose(b["W"], a["W"], rtol=1e-13)
    g = rng.normal(size=(4, 5))
    ql, _ = np.linalg.qr(rng.normal(size=(4, 4)))
    qr, _ = np.linalg.qr(rng.normal(size=(5, 5)))
    c = soap.soap_matrix_step(np.zeros((4, 5)), np.zeros((4, 4)), np.zeros((5, 5)),
                              np.zeros((4, 5)), np.zeros((4, 5)), [g], t=1, refresh=False,
                              basis=(np.zeros(4), ql, np.zeros(5), qr), **dict(h, eps=1e-6))
    n_ref, _, _ = soap.soap_direction(g, 0.1 * g, np.zeros((4, 5)), ql, qr, t=1, beta1=0.9,
                                      beta2=0.95, eps=1e-6)
    np.testing.assert_allclose(c["N"], n_ref, atol=1e-14)
    assert c["QL"] is ql
