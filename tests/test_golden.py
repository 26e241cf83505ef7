"""The stored fixtures of tests/golden (written by tests/golden/make_golden.py from the oracle).

They anchor the oracle against accidental change, and the planner fixtures pin the C
library's planner bit for bit without the oracle in the loop.
"""

import os

import numpy as np
import pytest

from oracle import muon, plan, soap
from workloads import get_config

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load_golden():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _read_matrix(name):
    rows, shape = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("# shape"):
                shape = tuple(int(x) for x in line.split()[2:])
            elif not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    m = np.array(rows)
    assert m.shape == shape
    return m


def _read_plan(name):
    loads, rows = None, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("# loads"):
                loads = [int(x) for x in line.split()[2:]]
            elif not line.startswith("#"):
                rows.append(tuple(int(x) for x in line.split()))
    return rows, loads


PLANS = [("plan_llama3_8b_w8_rolegreedy.txt", 2, 8, plan.ROLE_GREEDY),
         ("plan_gpt2_small_w8_scopegreedy.txt", 1, 8, plan.SCOPE_GREEDY)]


@pytest.mark.parametrize("name,cfg,world,policy", PLANS)
def test_plan_fixture_oracle_and_library(name, cfg, world, policy):
    rows, loads = _read_plan(name)
    mg = _load_golden()
    orows, oloads = mg.plan_rows(cfg, world, policy)
    assert orows == rows and oloads == loads
    from matrix_optimizer_owner_gb300 import _lib, mfsdp
    if not os.path.exists(_lib.LIB_PATH):
        pytest.skip("library not built")
    wl = get_config(cfg)
    params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
    segs, _, _ = mfsdp.mfsdp_plan_owner_set(params, world, policy)
    got = [(i, s["owner"], s["role"], s["local_offset"], s["numel"]) for i, s in enumerate(segs)]
    assert got == rows


def test_newton_schulz_fixture():
    mg = _load_golden()
    np.testing.assert_allclose(muon.newton_schulz(mg.ns_input()),
                               _read_matrix("newton_schulz_8x12_seed3.txt"), rtol=0, atol=1e-15)


def test_soap_fixture():
    mg = _load_golden()
    gs, w0 = mg.soap_inputs()
    st = {"W": w0, "L": np.zeros((5, 5)), "R": np.zeros((7, 7)), "M": np.zeros((5, 7)),
          "V": np.zeros((5, 7))}
    for t, g in enumerate(gs, start=1):
        st = soap.soap_matrix_step(st["W"], st["L"], st["R"], st["M"], st["V"], [g], t=t,
                                   **mg.SOAP_HYPER)
    np.testing.assert_allclose(st["W"], _read_matrix("soap_5x7_3steps_seed5.txt"), rtol=0,
                               atol=1e-12)


def test_shampoo_fixture():
    mg = _load_golden()
    np.testing.assert_allclose(mg.shampoo_run(), _read_matrix("shampoo_6x4_3steps_seed7.txt"),
                               rtol=0, atol=1e-12)
