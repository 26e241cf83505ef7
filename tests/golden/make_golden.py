"""Writes the stored fixtures of this folder from the oracle (and only the oracle).

    python tests/golden/make_golden.py

Each fixture starts with comment lines naming the passage it follows and the inputs it was
computed from; tests/test_golden.py recomputes every value with the oracle and checks the
planner fixture against the C library as well.
"""

from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import muon, plan, shampoo, soap  # noqa: E402
from workloads import get_config  # noqa: E402

SOURCE = ('"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter '
          'sharding"')


def ns_input():
    return np.random.default_rng(3).normal(size=(8, 12)) * 0.1


def soap_inputs():
    rng = np.random.default_rng(5)
    return [rng.normal(size=(5, 7)) * 1e-2 for _ in range(3)], rng.normal(size=(5, 7)) * 0.02


def shampoo_inputs():
    rng = np.random.default_rng(7)
    return [rng.normal(size=(6, 4)) * 1e-2 for _ in range(3)], rng.normal(size=(6, 4)) * 0.02


SHAMPOO_EPS = 1e-6
SHAMPOO_HYPER = dict(grad_scale=1.0, lr=0.02, weight_decay=1e-2)


def shampoo_run():
    gs, w = shampoo_inputs()
    l, r = SHAMPOO_EPS * np.eye(6), SHAMPOO_EPS * np.eye(4)
    for g in gs:
        o = shampoo.shampoo_matrix_step(w, l, r, [g], **SHAMPOO_HYPER)
        w, l, r = o["W"], o["L"], o["R"]
    return w


SOAP_HYPER = dict(grad_scale=1.0, lr=1e-3, weight_decay=1e-2, beta1=0.9, beta2=0.95, eps=1e-6,
                  beta_stats=0.95)


def plan_rows(cfg: int, world: int, policy: int):
    wl = get_config(cfg)
    ps = [plan.Param(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
    segs = plan.plan(ps, world, policy)
    return [(i, s.owner, s.role, s.local_offset, s.numel) for i, s in enumerate(segs)], \
        plan.rank_loads(segs, world)


def write_plan(path, cfg, world, policy, name):
    rows, loads = plan_rows(cfg, world, policy)
    with open(path, "w") as f:
        f.write(f"# {SOURCE}, §4.1 (owner assignment, {name}) and §4.2 (segment layout)\n")
        f.write(f"# workload config {cfg}, world size {world}; columns: parameter owner role "
                f"local_offset numel\n")
        f.write("# loads " + " ".join(str(x) for x in loads) + "\n")
        for r in rows:
            f.write(" ".join(str(x) for x in r) + "\n")


def write_matrix(path, header, m):
    with open(path, "w") as f:
        for h in header:
            f.write(f"# {h}\n")
        f.write(f"# shape {m.shape[0]} {m.shape[1]}\n")
        for row in m:
            f.write(" ".join(repr(float(x)) for x in row) + "\n")


def main():
    write_plan(os.path.join(HERE, "plan_llama3_8b_w8_rolegreedy.txt"), 2, 8, plan.ROLE_GREEDY,
               "RoleGreedy")
    write_plan(os.path.join(HERE, "plan_gpt2_small_w8_scopegreedy.txt"), 1, 8,
               plan.SCOPE_GREEDY, "ScopeGreedy")
    write_matrix(os.path.join(HERE, "newton_schulz_8x12_seed3.txt"),
                 [f"{SOURCE}, §2: Muon's quintic Newton-Schulz, 5 steps, (a, b, c) = "
                  "(3.4445, -4.7750, 2.0315), X0 = U / (||U||_F + 1e-7)",
                  "input: numpy default_rng(3).normal(size=(8, 12)) * 0.1"],
                 muon.newton_schulz(ns_input()))
    write_matrix(os.path.join(HERE, "shampoo_6x4_3steps_seed7.txt"),
                 [f"{SOURCE}, §5.7: Shampoo (full left and right preconditioners, inverse "
                  "fourth roots), W after 3 steps",
                  "inputs: numpy default_rng(7): three normal(size=(6, 4)) * 1e-2 gradients, "
                  "then W0 = normal(size=(6, 4)) * 0.02; L = 1e-6 I, R = 1e-6 I",
                  "lr 0.02, wd 1e-2, grad_scale 1"],
                 shampoo_run())
    gs, w0 = soap_inputs()
    st = {"W": w0, "L": np.zeros((5, 5)), "R": np.zeros((7, 7)), "M": np.zeros((5, 7)),
          "V": np.zeros((5, 7))}
    for t, g in enumerate(gs, start=1):
        st = soap.soap_matrix_step(st["W"], st["L"], st["R"], st["M"], st["V"], [g], t=t,
                                   **SOAP_HYPER)
    write_matrix(os.path.join(HERE, "soap_5x7_3steps_seed5.txt"),
                 [f"{SOURCE}, §5.7: SOAP (Adam in the Shampoo eigenbasis), W after 3 steps",
                  "inputs: numpy default_rng(5): three normal(size=(5, 7)) * 1e-2 gradients, "
                  "then W0 = normal(size=(5, 7)) * 0.02; L = R = M = V = 0",
                  "lr 1e-3, wd 1e-2, beta1 0.9, beta2 0.95, beta_stats 0.95, eps 1e-6"],
                 st["W"])


if __name__ == "__main__":
    main()
