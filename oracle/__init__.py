"""fp64 CPU oracle of the Titans/ATLAS memory-layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may.  It shares no code with the CUDA library.
"""
from .atlas_oracle import (  # noqa: F401
    NS_COEFFS,
    NS_EPS,
    features,
    forward,
    forward_unit,
    memory_apply,
    newton_schulz,
    poly_features,
    token_gradients,
    unit_inputs,
)
from .prologue import prologue_row  # noqa: F401,E402
