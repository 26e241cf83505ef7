"""The five owner-step workloads, as parameter lists with FSDP blocks.

Shapes follow the transformer shapes each workload names (weights stored as
``rows x cols`` = ``out_features x in_features``).  Where a workload leaves a choice open,
the choice is written next to it:

* weights and tail parameters are drawn from N(0, 0.02^2) in fp32;
* tail (non-2D) contributions use the workload's gradient std and contribution dtype;
* the GPT-2-small tail per layer is ln_1.{weight,bias}, attn.c_proj.bias, ln_2.{weight,bias},
  mlp.c_proj.bias (768 each) and mlp.c_fc.bias (3072): the lengths the workload lists;
* the Llama-3-8B tail per layer is the two RMSNorm weights (4096 each);
* the skewed batch and the Llama-3-70B share have no tail;
* the skewed batch draws one gradient std per matrix, log-uniform over [1e-5, 1e-1].

"MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding",
§3 (owner-shaped placement: one role per 2D matrix and one packed non-2D tail per FSDP unit)
and §5.1 (AdamW lr 1e-3, weight decay 1e-2 for the tail; Muon uses weight decay 1e-2).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple


@dataclass(frozen=True)
class ParamSpec:
    """One model parameter.  ``cols == 1`` and ``is_matrix == False`` for vectors."""

    name: str
    rows: int
    cols: int
    block: int
    is_matrix: bool

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Hyper:
    lr: float = 0.02
    momentum: float = 0.95
    nesterov: bool = True
    weight_decay: float = 0.01
    ns_steps: int = 5
    ns_a: float = 3.4445
    ns_b: float = -4.7750
    ns_c: float = 2.0315
    ns_eps: float = 1e-7
    lr_adjust: str = "original"  # sqrt(max(1, rows/cols)); "match_rms_adamw" = 0.2*sqrt(max(rows, cols))
    grad_scale: float = 1.0  # contributions are summed (1/W would average them)
    adam_lr: float = 1e-3
    adam_betas: Tuple[float, float] = (0.9, 0.95)
    adam_eps: float = 1e-8
    adam_wd: float = 1e-2


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    params: Tuple[ParamSpec, ...]  # the whole model, in declaration order
    world_size: int  # simulated data-parallel ranks the planner spreads owners over
    rank: int  # the rank whose owned set runs on this GPU
    W: int  # gradient contributions per parameter (simulated rank-local gradients)
    contrib_dtype: str  # "f32" or "bf16"
    grad_std: float
    weight_std: float = 0.02
    steps: int = 3
    grad_std_loguniform: Optional[Tuple[float, float]] = None  # per-matrix std range
    hyper: Hyper = field(default_factory=Hyper)

    @property
    def matrices(self) -> List[ParamSpec]:
        return [p for p in self.params if p.is_matrix]


def _mat(name, r, c, block):
    return ParamSpec(name, r, c, block, True)


def _vec(name, n, block):
    return ParamSpec(name, n, 1, block, False)


def _tiny() -> Tuple[ParamSpec, ...]:
    ps = [_mat("w0", 64, 64, 0), _mat("w1", 64, 256, 0), _mat("w2", 256, 64, 0),
          _mat("w3", 128, 128, 0)]
    ps += [_vec(f"v{i}", 256, 0) for i in range(3)]
    return tuple(ps)


def _gpt2_small() -> Tuple[ParamSpec, ...]:
    ps = []
    for l in range(12):
        ps += [
            _vec(f"h{l}.ln_1.weight", 768, l),
            _vec(f"h{l}.ln_1.bias", 768, l),
            _mat(f"h{l}.attn.c_attn.weight", 2304, 768, l),
            _mat(f"h{l}.attn.c_proj.weight", 768, 768, l),
            _vec(f"h{l}.attn.c_proj.bias", 768, l),
            _vec(f"h{l}.ln_2.weight", 768, l),
            _vec(f"h{l}.ln_2.bias", 768, l),
            _mat(f"h{l}.mlp.c_fc.weight", 3072, 768, l),
            _vec(f"h{l}.mlp.c_fc.bias", 3072, l),
            _mat(f"h{l}.mlp.c_proj.weight", 768, 3072, l),
            _vec(f"h{l}.mlp.c_proj.bias", 768, l),
        ]
    return tuple(ps)


def _llama3_8b() -> Tuple[ParamSpec, ...]:
    ps = []
    for l in range(32):
        ps += [
            _mat(f"layers.{l}.self_attn.q_proj.weight", 4096, 4096, l),
            _mat(f"layers.{l}.self_attn.k_proj.weight", 1024, 4096, l),
            _mat(f"layers.{l}.self_attn.v_proj.weight", 1024, 4096, l),
            _mat(f"layers.{l}.self_attn.o_proj.weight", 4096, 4096, l),
            _mat(f"layers.{l}.mlp.gate_proj.weight", 14336, 4096, l),
            _mat(f"layers.{l}.mlp.up_proj.weight", 14336, 4096, l),
            _mat(f"layers.{l}.mlp.down_proj.weight", 4096, 14336, l),
            _vec(f"layers.{l}.input_layernorm.weight", 4096, l),
            _vec(f"layers.{l}.post_attention_layernorm.weight", 4096, l),
        ]
    return tuple(ps)


def _skewed() -> Tuple[ParamSpec, ...]:
    ps = [_mat(f"s{i}", 128, 512, 0) for i in range(256)]
    ps += [_mat(f"m{i}", 1024, 1024, 1) for i in range(64)]
    ps += [_mat(f"l{i}", 8192, 28672, 2 + i) for i in range(4)]
    return tuple(ps)


def _llama3_70b_share() -> Tuple[ParamSpec, ...]:
    ps = []
    for i in range(24):
        r, c = (28672, 8192) if i % 2 == 0 else (8192, 28672)
        ps.append(_mat(f"mlp{i}", r, c, i))
    ps += [_mat(f"attn{i}", 8192, 8192, 24 + i) for i in range(16)]
    return tuple(ps)


CONFIGS: Tuple[Workload, ...] = (
    Workload(0, "tiny: 64x64, 64x256, 256x64, 128x128 + 3x256 tail, W=4 fp32", _tiny(),
             world_size=1, rank=0, W=4, contrib_dtype="f32", grad_std=1e-2, steps=3),
    Workload(1, "gpt2-small: 12 layers, hidden 768, 48 matrices, W=8 bf16", _gpt2_small(),
             world_size=1, rank=0, W=8, contrib_dtype="bf16", grad_std=1e-3, steps=3),
    Workload(2, "llama3-8b owner share: rank 0 of 8, W=8 bf16", _llama3_8b(),
             world_size=8, rank=0, W=8, contrib_dtype="bf16", grad_std=1e-3, steps=3),
    Workload(3, "skewed: 256x(128x512) + 64x(1024^2) + 4x(8192x28672), W=4 bf16", _skewed(),
             world_size=1, rank=0, W=4, contrib_dtype="bf16", grad_std=1e-3, steps=3,
             grad_std_loguniform=(1e-5, 1e-1)),
    Workload(4, "llama3-70b share: 24 MLP (28672x8192 / 8192x28672) + 16 x 8192^2, W=2 bf16",
             _llama3_70b_share(), world_size=1, rank=0, W=2, contrib_dtype="bf16",
             grad_std=1e-3, steps=5),
)


def get_config(i: int) -> Workload:
    return CONFIGS[i]
