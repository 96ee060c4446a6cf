"""Seeded synthetic workloads for the Titans/ATLAS memory-layer forward.

This package holds workload shapes and seeded input generators only.  It
contains none of the memory layer's arithmetic, so both the CPU oracle and
the CUDA path (through its Python binding) can draw identical inputs from it.
"""
from .configs import PROLOGUES, WORKLOADS, Prologue, Workload, get_workload  # noqa: F401
from .inputs import (  # noqa: F401
    bf16_round,
    bf16_bits,
    bf16_from_bits,
    make_inputs,
    make_prologue_inputs,
    unit_slice,
)
