"""Seeded synthetic inputs: weights, per-rank gradient contributions, tail vectors.

Every draw is keyed by (workload, kind, step, parameter index, contribution index) through a
splitmix64 mix, so any single parameter's inputs can be regenerated on their own (the
full-size parity tests rebuild the inputs of a sample of matrices for the oracle).

Values are drawn in fp32 with ``torch.randn`` and then rounded to the contribution dtype
(round-to-nearest-even for bf16).  The rounded value *is* the input: the oracle upcasts it
exactly to fp64.  On a CUDA device torch uses its counter-based Philox generator, on the CPU
its Mersenne twister, so host and device draws differ; parity tests therefore always copy
the device draw to the host rather than re-drawing it there.
"""

from __future__ import annotations

import math
from typing import List, Sequence

import numpy as np
import torch

from .configs import ParamSpec, Workload

KIND_WEIGHT = 1
KIND_CONTRIB = 2
KIND_STD = 3

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def seed_of(*keys: int) -> int:
    """Deterministic 63-bit seed from a tuple of small non-negative integers."""
    h = 0x243F6A8885A308D3
    for k in keys:
        h = _splitmix64(h ^ (int(k) & _MASK64))
    return h & ((1 << 63) - 1)


_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def normal(n: int, std: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """``n`` draws of N(0, std^2): fp32 draw, scaled in fp32, then rounded to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    x.mul_(std)
    return x.to(dtype)


def grad_std(wl: Workload, p_index: int) -> float:
    """Gradient std of parameter ``p_index``; per-matrix log-uniform where the workload says so."""
    if wl.grad_std_loguniform is None:
        return wl.grad_std
    lo, hi = wl.grad_std_loguniform
    rng = np.random.default_rng(seed_of(wl.index, KIND_STD, p_index))
    return float(10.0 ** rng.uniform(math.log10(lo), math.log10(hi)))


def weight(wl: Workload, p_index: int, device="cpu") -> torch.Tensor:
    p = wl.params[p_index]
    return normal(p.numel, wl.weight_std, seed_of(wl.index, KIND_WEIGHT, p_index), device)


def contribution(wl: Workload, step: int, p_index: int, w: int, device="cpu") -> torch.Tensor:
    p = wl.params[p_index]
    return normal(p.numel, grad_std(wl, p_index),
                  seed_of(wl.index, KIND_CONTRIB, step, p_index, w), device,
                  torch_dtype(wl.contrib_dtype))


def flat_offsets(params: Sequence[ParamSpec]) -> List[int]:
    """Offsets of ``params`` packed back to back (no padding) in one flat buffer."""
    offs, o = [], 0
    for p in params:
        offs.append(o)
        o += p.numel
    return offs


def fill_flat(buf: torch.Tensor, indices: Sequence[int], offsets: Sequence[int],
              make) -> torch.Tensor:
    """Write ``make(p_index)`` into ``buf[offset : offset + numel]`` for each owned parameter."""
    for pi, off in zip(indices, offsets):
        v = make(pi)
        buf[off:off + v.numel()].copy_(v)
    return buf
