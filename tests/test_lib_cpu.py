"""Host-side tests of libmfsdp (CPU only): exported symbols, the C++ owner planner against the
oracle planner (bit-exact), argument validation and error codes.  Nothing here launches GPU
work."""

import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import plan as oplan
from workloads import get_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from matrix_optimizer_owner_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from matrix_optimizer_owner_gb300 import build
        build.build()
    return _lib.load()


def header_functions():
    with open(os.path.join(ROOT, "include", "mfsdp.h"), encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mfsdp_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    from matrix_optimizer_owner_gb300 import _lib
    names = header_functions()
    assert len(names) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert getattr(lib, n) is not None
    # the binding describes every declared entry point
    assert set(names) == set(_lib.SIGNATURES)


def test_version_and_status_strings(lib):
    from matrix_optimizer_owner_gb300 import mfsdp
    assert mfsdp.mfsdp_version() == 100
    assert mfsdp.mfsdp_status_string(-7) == "device wait timed out"
    assert mfsdp.mfsdp_status_string(12345) == "unknown status"


def _params(wl):
    return [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]


def _oracle(params, W, policy):
    ps = [oplan.Param(r, c, b, m) for r, c, b, m in params]
    segs = oplan.plan(ps, W, policy)
    brn = oplan.block_rank_numel(ps, segs, W)
    table = [[brn[(b, r)] for r in range(W)] for b in oplan.block_order(ps)]
    return [{"owner": s.owner, "role": s.role, "local_offset": s.local_offset,
             "rank_offset": s.rank_offset, "numel": s.numel} for s in segs], table


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("policy", [0, 1])
def test_planner_bit_exact_on_workloads(lib, cfg, policy):
    from matrix_optimizer_owner_gb300 import mfsdp
    wl = get_config(cfg)
    params = _params(wl)
    for W in sorted({1, 2, 3, 8, wl.world_size}):
        segs, table, nb = mfsdp.mfsdp_plan_owner_set(params, W, policy)
        osegs, otable = _oracle(params, W, policy)
        assert segs == osegs
        assert table == otable and nb == len(otable)


def test_planner_bit_exact_on_random_sets(lib):
    from matrix_optimizer_owner_gb300 import mfsdp
    rng = np.random.default_rng(123)
    for trial in range(300):
        n = int(rng.integers(0, 30))
        params = []
        for _ in range(n):
            is_mat = bool(rng.random() < 0.6)
            r = int(rng.integers(0, 9))
            c = int(rng.integers(0, 9)) if is_mat else 1
            params.append((r, c, int(rng.integers(0, 5)), is_mat))
        W = int(rng.integers(1, 6))
        for policy in (0, 1):
            segs, table, nb = mfsdp.mfsdp_plan_owner_set(params, W, policy)
            osegs, otable = _oracle(params, W, policy)
            assert segs == osegs, (trial, params, W, policy)
            assert table == otable


def _oracle_score(params, W, segs, **kw):
    ps = [oplan.Param(r, c, b, m) for r, c, b, m in params]
    osegs = [oplan.Segment(s["owner"], s["role"], s["local_offset"], s["rank_offset"],
                           s["numel"]) for s in segs]
    ranks = [x.__dict__ for x in oplan.score_plan(ps, osegs, W, **kw)]
    gam = oplan.gamma(ps, osegs, W)
    return ranks, [gam[b] for b in oplan.block_order(ps)]


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_scorer_and_cost_aware_bit_exact_on_workloads(lib, cfg):
    from matrix_optimizer_owner_gb300 import mfsdp
    wl = get_config(cfg)
    params = _params(wl)
    ps = [oplan.Param(r, c, b, m) for r, c, b, m in params]
    for W in sorted({1, 2, 3, 8, wl.world_size}):
        for policy in (0, 1):
            segs, _, _ = mfsdp.mfsdp_plan_owner_set(params, W, policy)
            for kw in ({}, dict(param_bytes=4, grad_bytes=4, state_bytes=8, ns_steps=2)):
                ranks, gam = mfsdp.mfsdp_score_plan(params, W, segs, **kw)
                oranks, ogam = _oracle_score(params, W, segs, **kw)
                assert ranks == oranks
                assert gam == ogam
        for cap in (0, 1, 1 << 40):
            segs, pol = mfsdp.mfsdp_plan_cost_aware(params, W, cap)
            osegs, opol = oplan.plan_cost_aware(ps, W, cap)
            assert pol == opol
            assert segs == [s.__dict__ for s in osegs]


def test_scorer_bit_exact_on_random_sets(lib):
    from matrix_optimizer_owner_gb300 import mfsdp
    rng = np.random.default_rng(321)
    for trial in range(200):
        n = int(rng.integers(0, 25))
        params = []
        for _ in range(n):
            is_mat = bool(rng.random() < 0.6)
            r = int(rng.integers(0, 300))
            c = int(rng.integers(0, 300)) if is_mat else 1
            params.append((r, c, int(rng.integers(0, 4)), is_mat))
        W = int(rng.integers(1, 6))
        segs, _, _ = mfsdp.mfsdp_plan_owner_set(params, W, int(rng.integers(0, 2)))
        ranks, gam = mfsdp.mfsdp_score_plan(params, W, segs)
        assert (ranks, gam) == _oracle_score(params, W, segs), trial
        ps = [oplan.Param(r, c, b, m) for r, c, b, m in params]
        cap = int(rng.integers(0, 4000))
        segs, pol = mfsdp.mfsdp_plan_cost_aware(params, W, cap)
        osegs, opol = oplan.plan_cost_aware(ps, W, cap)
        assert pol == opol and segs == [s.__dict__ for s in osegs], trial


def test_scorer_error_codes(lib):
    from matrix_optimizer_owner_gb300 import _lib as L
    pd = (L.ParamDesc * 1)(L.ParamDesc(2, 2, 0, 1))
    seg = (L.Segment * 1)(L.Segment(0, 0, 0, 0, 4))
    out = (L.RankResources * 2)()
    good = L.CostModel(2, 2, 4, 5)
    assert lib.mfsdp_score_plan(pd, 1, 2, seg, C.byref(good), out, None, None) == 0
    assert lib.mfsdp_score_plan(pd, 1, 2, seg, None, out, None, None) == -1       # no model
    bad_model = L.CostModel(0, 2, 4, 5)
    assert lib.mfsdp_score_plan(pd, 1, 2, seg, C.byref(bad_model), out, None, None) == -1
    bad_owner = (L.Segment * 1)(L.Segment(2, 0, 0, 0, 4))
    assert lib.mfsdp_score_plan(pd, 1, 2, bad_owner, C.byref(good), out, None, None) == -1
    bad_numel = (L.Segment * 1)(L.Segment(0, 0, 0, 0, 5))
    assert lib.mfsdp_score_plan(pd, 1, 2, bad_numel, C.byref(good), out, None, None) == -2
    assert lib.mfsdp_plan_cost_aware(pd, 1, 0, C.byref(good), 0, seg, None) == -1  # world size
    assert lib.mfsdp_plan_cost_aware(pd, 1, 2, None, 0, seg, None) == -1           # no model


def test_repack_validation_before_any_launch(lib):
    from matrix_optimizer_owner_gb300 import _lib as L
    pd = (L.ParamDesc * 2)(L.ParamDesc(2, 2, 0, 1), L.ParamDesc(3, 1, 0, 0))
    seg = (L.Segment * 2)(L.Segment(0, 0, 0, 0, 4), L.Segment(1, 1, 0, 0, 3))
    sh = (C.c_void_p * 2)(1 << 20, 2 << 20)     # never dereferenced: every case fails first
    canon, ws = C.c_void_p(3 << 20), C.c_void_p(4 << 20)
    need = C.c_size_t(0)
    assert lib.mfsdp_repack_workspace_bytes(2, C.byref(need)) == 0 and need.value >= 64
    assert lib.mfsdp_repack_workspace_bytes(-1, C.byref(need)) == -1
    pack, unpack = lib.mfsdp_pack_owner_shards, lib.mfsdp_unpack_owner_shards
    assert pack(pd, 2, seg, 0, 2, canon, sh, ws, need.value, None) == -1        # world size
    assert pack(pd, 2, seg, 2, 3, canon, sh, ws, need.value, None) == -1        # element size
    assert pack(pd, 2, seg, 2, 2, None, sh, ws, need.value, None) == -1         # no canonical
    assert unpack(pd, 2, seg, 2, 2, None, canon, ws, need.value, None) == -1    # no shards
    bad_owner = (L.Segment * 2)(L.Segment(0, 0, 0, 0, 4), L.Segment(2, 1, 0, 0, 3))
    assert pack(pd, 2, bad_owner, 2, 2, canon, sh, ws, need.value, None) == -1
    bad_numel = (L.Segment * 2)(L.Segment(0, 0, 0, 0, 5), L.Segment(1, 1, 0, 0, 3))
    assert pack(pd, 2, bad_numel, 2, 2, canon, sh, ws, need.value, None) == -2
    outside = (L.Segment * 2)(L.Segment(0, 0, 1, 0, 4), L.Segment(1, 1, 0, 0, 3))
    assert pack(pd, 2, outside, 2, 2, canon, sh, ws, need.value, None) == -2    # past its shard
    assert pack(pd, 2, seg, 2, 2, canon, sh, None, need.value, None) == -5      # no workspace
    assert pack(pd, 2, seg, 2, 2, canon, sh, ws, 8, None) == -5                 # too small
    assert pack(None, 0, None, 2, 2, None, None, None, 0, None) == 0            # empty model


def test_planner_error_codes(lib):
    from matrix_optimizer_owner_gb300 import _lib as L
    pd = (L.ParamDesc * 1)(L.ParamDesc(2, 2, 0, 1))
    seg = (L.Segment * 1)()
    assert lib.mfsdp_plan_owner_set(pd, 1, 0, 0, seg, None, None) == -1      # world size
    assert lib.mfsdp_plan_owner_set(pd, 1, 2, 7, seg, None, None) == -1      # policy
    assert lib.mfsdp_plan_owner_set(None, 1, 2, 0, seg, None, None) == -1    # null params
    bad = (L.ParamDesc * 1)(L.ParamDesc(-1, 2, 0, 1))
    assert lib.mfsdp_plan_owner_set(bad, 1, 2, 0, seg, None, None) == -2     # negative dim
    huge = (L.ParamDesc * 1)(L.ParamDesc(1 << 40, 1 << 40, 0, 1))
    assert lib.mfsdp_plan_owner_set(huge, 1, 2, 0, seg, None, None) == -2    # numel overflow
    assert lib.mfsdp_plan_owner_set(None, 0, 2, 0, None, None, None) == 0    # empty model


def test_owner_set_validation_and_workspace(lib):
    from matrix_optimizer_owner_gb300 import mfsdp
    s = mfsdp.OwnerSet([(64, 64, 0), (64, 256, 4096), (256, 64, 20480), (128, 128, 36864)],
                       split_max_numel=32768)
    assert s.split_count() == 4
    ws = s.workspace_bytes()
    assert ws > 0 and ws % 256 == 0
    big = mfsdp.OwnerSet([(2304, 768, 0)], split_max_numel=0)
    assert big.split_count() == 0
    # m x m Gram + polynomial buffers and the ping X buffer are in the workspace
    assert big.workspace_bytes() >= 2304 * 768 * 2 + 2 * 768 * 768 * 2
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.OwnerSet([(4, 4, 0), (4, 4, 8)])                         # overlapping ranges
    assert e.value.status == -2
    with pytest.raises(mfsdp.MfsdpError) as e:
        mfsdp.OwnerSet([(-4, 4, 0)])
    assert e.value.status == -2
    empty = mfsdp.OwnerSet([])
    assert empty.workspace_bytes() > 0
    # step calls on an unbound set are rejected before anything is launched
    nul = C.c_void_p(0)
    ptrs = (C.c_void_p * 1)(256)
    assert lib.mfsdp_owner_reduce_momentum(s.handle, ptrs, 1, 1, 1.0, 0.9, 1, 256, 512, 768,
                                           None, 1024, nul) == -1
    assert lib.mfsdp_newton_schulz(s.handle, 256, 512, 1024, 5, 3.4, -4.7, 2.0, 1e-7, 768, 1024,
                                   nul) == -1
    assert lib.mfsdp_apply_update(s.handle, 256, 512, None, 0.02, 0.01, 0, nul) == -1
    # AdamW argument checks (no launch: they fail first)
    assert lib.mfsdp_adamw_tail(ptrs, 1, 1, 1.0, 16, 256, 512, 768, 0, 1e-3, 0.9, 0.95, 1e-8,
                                0.01, nul) == -1                         # step 0
    assert lib.mfsdp_adamw_tail(ptrs, 0, 1, 1.0, 16, 256, 512, 768, 1, 1e-3, 0.9, 0.95, 1e-8,
                                0.01, nul) == -1                         # W = 0
    assert lib.mfsdp_adamw_tail(ptrs, 1, 1, 1.0, 16, 258, 512, 768, 1, 1e-3, 0.9, 0.95, 1e-8,
                                0.01, nul) == -3                         # misaligned
    assert lib.mfsdp_adamw_tail(ptrs, 1, 1, 1.0, 0, 0, 0, 0, 1, 1e-3, 0.9, 0.95, 1e-8,
                                0.01, nul) == 0                          # empty tail


def test_shampoo_validation_before_any_launch(lib):
    from matrix_optimizer_owner_gb300 import _lib as L
    mats = (L.Matrix * 2)(L.Matrix(4, 3, 0), L.Matrix(2, 5, 12))
    h = C.c_void_p()
    assert lib.mfsdp_shampoo_set_create(mats, 2, C.byref(h)) == 0
    ws, ln, rn = C.c_size_t(0), C.c_int64(0), C.c_int64(0)
    assert lib.mfsdp_shampoo_set_sizes(h, C.byref(ws), C.byref(ln), C.byref(rn)) == 0
    assert (ln.value, rn.value) == (16 + 4, 9 + 25)
    # 7 root buffers per side, P and Y, norms and tables; the split-bf16 mode's buffers (hi and
    # lo halves, rows padded to 8 elements) and its tensor maps (8 per buffer) fit as well
    assert ws.value >= 4 * (7 * (16 + 9 + 4 + 25) + 2 * 22)
    assert ws.value >= 4 * 7 * (4 * 8 + 3 * 8 + 2 * 8 + 5 * 8) + 128 * 8 * (7 * 4 + 3 * 2)
    p = C.c_void_p(1 << 20)  # never dereferenced: every case fails first
    st = lib.mfsdp_shampoo_step
    for prec in (0, 1):
        assert st(h, None, p, p, p, 0.1, 0.0, 30, prec, p, ws.value, None) == -1  # no gradient
        assert st(h, p, p, p, p, 0.1, 0.0, 0, prec, p, ws.value, None) == -1      # iterations
        assert st(h, p, p, p, p, 0.1, 0.0, 30, prec, None, ws.value, None) == -5  # no workspace
        assert st(h, p, p, p, p, 0.1, 0.0, 30, prec, p, ws.value - 1, None) == -5  # too small
    assert st(h, p, p, p, p, 0.1, 0.0, 30, 2, p, ws.value, None) == -1          # precision
    assert st(h, p, p, p, p, 0.1, 0.0, 30, -1, p, ws.value, None) == -1
    assert lib.mfsdp_shampoo_init_state(h, 0.0, p, p, p, ws.value, None) == -1  # eps
    assert lib.mfsdp_shampoo_set_destroy(h) == 0
    bad = (L.Matrix * 1)(L.Matrix(0, 3, 0))
    assert lib.mfsdp_shampoo_set_create(bad, 1, C.byref(h)) == -2
    assert lib.mfsdp_shampoo_set_create(None, 1, C.byref(h)) == -1


def test_soap_validation_before_any_launch(lib):
    from matrix_optimizer_owner_gb300 import _lib as L
    mats = (L.Matrix * 2)(L.Matrix(4, 3, 0), L.Matrix(2, 70, 12))
    h = C.c_void_p()
    assert lib.mfsdp_soap_set_create(mats, 2, C.byref(h)) == 0
    ws, ln, rn, el, er = (C.c_size_t(0), C.c_int64(0), C.c_int64(0), C.c_int64(0),
                          C.c_int64(0))
    assert lib.mfsdp_soap_set_sizes(h, C.byref(ws), C.byref(ln), C.byref(rn), C.byref(el),
                                    C.byref(er)) == 0
    assert (ln.value, rn.value, el.value, er.value) == (16 + 4, 9 + 4900, 4 + 2, 3 + 70)
    # per side a padded working matrix and basis (dims rounded up to 64: 64, 64, 64, 128)
    assert ws.value >= 4 * 2 * (3 * 64 * 64 + 128 * 128)
    p = C.c_void_p(1 << 20)  # never dereferenced: every case fails first
    st = L.SoapState(*([p.value] * 8))
    good = L.SoapHyper(1e-3, 0.9, 0.95, 0.95, 1e-8, 0.01, 10, 0.0, 1)
    step = lib.mfsdp_soap_step
    assert step(h, None, p, C.byref(st), 1, C.byref(good), None, p, ws.value, None) == -1
    assert step(h, p, p, None, 1, C.byref(good), None, p, ws.value, None) == -1
    assert step(h, p, p, C.byref(st), 0, C.byref(good), None, p, ws.value, None) == -1  # t
    for field, bad in (("max_sweeps", 0), ("max_sweeps", 101), ("beta1", 1.0),
                       ("beta2", -0.1), ("beta_stats", 1.0), ("eps", -1.0),
                       ("jacobi_tol", -1e-6), ("jacobi_tol", 0.5), ("refresh", 2)):
        hb = L.SoapHyper(1e-3, 0.9, 0.95, 0.95, 1e-8, 0.01, 10, 0.0, 1)
        setattr(hb, field, bad)
        assert step(h, p, p, C.byref(st), 1, C.byref(hb), None, p, ws.value, None) == -1, field
    assert step(h, p, p, C.byref(st), 1, C.byref(good), None, None, ws.value, None) == -5
    assert step(h, p, p, C.byref(st), 1, C.byref(good), None, p, ws.value - 1, None) == -5
    missing = L.SoapState(*([p.value] * 7 + [None]))
    assert step(h, p, p, C.byref(missing), 1, C.byref(good), None, p, ws.value, None) == -1
    assert lib.mfsdp_soap_init_state(h, C.byref(missing), p, ws.value, None) == -1
    assert lib.mfsdp_soap_init_state(h, C.byref(st), p, ws.value - 1, None) == -5
    assert lib.mfsdp_soap_set_destroy(h) == 0
    bad = (L.Matrix * 1)(L.Matrix(3, 0, 0))
    assert lib.mfsdp_soap_set_create(bad, 1, C.byref(h)) == -2
    assert lib.mfsdp_soap_set_create(None, 1, C.byref(h)) == -1
    # the empty set is a no-op
    assert lib.mfsdp_soap_set_create(None, 0, C.byref(h)) == 0
    assert step(h, p, p, C.byref(st), 1, C.byref(good), None, None, 0, None) == 0
    assert lib.mfsdp_soap_set_destroy(h) == 0
