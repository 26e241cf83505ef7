"""Workload shapes and seeded synthetic inputs for the owner-local Muon step.

This package describes *what* is optimised (parameter shapes, FSDP blocks, gradient
statistics, hyperparameters) and draws the seeded random inputs.  It holds none of the
optimizer arithmetic: both the CUDA path (through the binding) and the CPU oracle consume
exactly the arrays drawn here.
"""

from .configs import CONFIGS, Hyper, ParamSpec, Workload, get_config  # noqa: F401
