"""Shared machinery of the GPU parity tests: build a workload's owned set on the device, draw
its seeded inputs there, run owner steps through the C ABI, and run the CPU oracle on exactly
the same input values (copied back from the device)."""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

from oracle import step as ostep
from workloads import synth
from workloads.configs import Hyper, Workload

from matrix_optimizer_owner_gb300 import owner_step


def rel(x, y) -> float:
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / d) if d > 0 else float(np.linalg.norm(x))


def max_rel(x, y) -> float:
    """max |x - y| / max |y|: catches a few wrong elements that a norm would average away."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    m = np.max(np.abs(y)) if y.size else 0.0
    return float(np.max(np.abs(x - y)) / m) if m > 0 else float(np.max(np.abs(x), initial=0.0))


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != torch.float64 \
        else t.detach().cpu().numpy()


@dataclass
class Case:
    """An owned set: shapes, flat offsets, tail length, and how contributions are drawn."""
    shapes: List[Tuple[int, int]]
    offsets: List[int]
    n_tail: int
    W: int
    dtype: torch.dtype
    hyper: Hyper
    grad_std: List[float]           # per matrix
    tail_grad_std: float
    weight_std: float = 0.02
    seed: int = 0
    wl: Optional[Workload] = None
    mat_params: Optional[List[int]] = None   # parameter indices, when built from a workload
    tail_params: Optional[List[int]] = None
    tail_offsets: Optional[List[int]] = None


def case_from_shapes(shapes, W=4, dtype=torch.float32, grad_std=1e-2, n_tail=0, seed=0,
                     hyper=None, gaps=False) -> Case:
    offs, o = [], 0
    for (r, c) in shapes:
        offs.append(o)
        o += r * c + (3 if gaps else 0)  # gaps make offsets ragged (unaligned)
    return Case(list(shapes), offs, n_tail, W, dtype, hyper or Hyper(), [grad_std] * len(shapes),
                grad_std, seed=seed)


def case_from_workload(wl: Workload) -> Case:
    params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
    lay = owner_step.owned_layout(params, wl.world_size, wl.rank)
    shapes = [(wl.params[i].rows, wl.params[i].cols) for i in lay.matrices]
    return Case(shapes, lay.matrix_offsets, lay.n_tail, wl.W, synth.torch_dtype(wl.contrib_dtype),
                wl.hyper, [synth.grad_std(wl, i) for i in lay.matrices], wl.grad_std,
                wl.weight_std, wl.index, wl, lay.matrices, lay.tails, lay.tail_offsets)


class DeviceRun:
    """Runs owner steps on the device and keeps host copies of every intermediate."""

    def __init__(self, case: Case, split_max_numel=owner_step.DEFAULT_SPLIT_MAX_NUMEL,
                 device="cuda"):
        self.case = case
        self.split_max_numel = split_max_numel
        self.dev = torch.device(device)
        self.runner = owner_step.OwnerStep(case.shapes, case.offsets, case.n_tail,
                                           split_max_numel=split_max_numel, device=self.dev)
        n = self.runner.n
        self.grad = torch.zeros(n, dtype=torch.float32, device=self.dev)
        # initial weights and tail parameters
        for k, ((r, c), off) in enumerate(zip(case.shapes, case.offsets)):
            self.runner.weights[off:off + r * c] = self._draw(r * c, case.weight_std,
                                                              (synth.KIND_WEIGHT, k), torch.float32)
        if case.n_tail:
            self.runner.tail_p.copy_(self._draw(case.n_tail, case.weight_std,
                                                (synth.KIND_WEIGHT, 10 ** 6), torch.float32))
        self.history: List[Dict] = []

    def _draw(self, n, std, key, dtype):
        return synth.normal(n, std, synth.seed_of(1000 + self.case.seed, *key), self.dev, dtype)

    def contributions(self, step: int):
        c = self.case
        out = []
        for w in range(c.W):
            buf = torch.zeros(self.runner.n, dtype=c.dtype, device=self.dev)
            for k, ((r, cc), off) in enumerate(zip(c.shapes, c.offsets)):
                buf[off:off + r * cc] = self._draw(r * cc, c.grad_std[k],
                                                   (synth.KIND_CONTRIB, step, k, w), c.dtype)
            out.append(buf)
        tail = [self._draw(c.n_tail, c.tail_grad_std, (synth.KIND_CONTRIB, step, 10 ** 6, w),
                           c.dtype) for w in range(c.W)] if c.n_tail else []
        return out, tail

    def run(self, steps: int):
        c = self.case
        r = self.runner
        init = {"W": host(r.weights), "p": host(r.tail_p) if c.n_tail else None}
        for t in range(steps):
            contribs, tail = self.contributions(t)
            W_before = host(r.weights)
            r.step(contribs, tail, c.hyper, reduced_grad=self.grad)
            torch.cuda.synchronize()
            rec = {
                "contrib": [host(x) for x in contribs],
                "tail_contrib": [host(x) for x in tail],
                "G": host(self.grad), "B": host(r.momentum), "Uhat": host(r.ns_input),
                "Uhat_lo": host(r.ns_input_lo) if r.ns_input_lo is not None else None,
                "nu": host(r.norm), "O": host(r.ortho),
                "O_lo": host(r.ortho_lo) if r.ortho_lo is not None else None,
                "W_before": W_before, "W": host(r.weights),
            }
            if c.n_tail:
                rec.update({"p": host(r.tail_p), "m": host(r.tail_m), "v": host(r.tail_v)})
            self.history.append(rec)
        return init

    def mat(self, arr: np.ndarray, k: int) -> np.ndarray:
        (rr, cc), off = self.case.shapes[k], self.case.offsets[k]
        return arr[off:off + rr * cc].reshape(rr, cc)


def oracle_matrix(run: DeviceRun, init, k: int, steps: int):
    """The oracle's trajectory of matrix k on the same (device-drawn) inputs."""
    c = run.case
    W0 = run.mat(init["W"], k)
    contribs_at = lambda t: [run.mat(x, k) for x in run.history[t]["contrib"]]
    return ostep.muon_trajectory(W0, contribs_at, steps, c.hyper)


def oracle_tail(run: DeviceRun, init, steps: int):
    c = run.case
    return ostep.adamw_trajectory(init["p"], lambda t: run.history[t]["tail_contrib"], steps,
                                  c.hyper)
