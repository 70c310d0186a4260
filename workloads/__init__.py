"""Seeded synthetic GDPA workloads.

This package only draws random numbers: jagged lengths, offset arrays and
input tensors with the shapes and value distributions of the five GDPA
workloads (jagged self-attention, user-ad cross-attention, PMA pooling, a
training step, and a tiny correctness case).  It holds none of the attention
arithmetic, so both the CUDA path and the float64 oracle can take their inputs
from it without sharing any of the method's code.
"""

from .configs import (  # noqa: F401
    CONFIGS,
    Workload,
    draw_lengths,
    get_config,
    make_inputs,
    offsets_from_lengths,
    small_case,
)
