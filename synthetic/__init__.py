"""Seeded synthetic inputs for the MoE layer forward.

This package is the only code shared by the CUDA path's tests/benchmark and
the CPU oracle.  It draws random tensors and holds no arithmetic of the MoE
method itself (no router, no top-k, no permutation, no expert MLP).  The one
non-trivial routine here, `calibrate_gate_bias`, solves a probability problem
about i.i.d. Gaussian logits to pick a gate-logit bias that gives a requested
expected expert load; it never looks at the generated tensors.
"""

from .workloads import Workload, WORKLOADS, scaled
from .generate import (
    generate,
    redraw_x_rows,
    expert_weights,
    calibrate_gate_bias,
    target_probabilities,
    logit_std,
)

__all__ = [
    "Workload",
    "WORKLOADS",
    "scaled",
    "generate",
    "redraw_x_rows",
    "expert_weights",
    "calibrate_gate_bias",
    "target_probabilities",
    "logit_std",
]
