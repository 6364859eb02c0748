"""fp64 CPU oracle for batched quintic Newton–Schulz and the Muon step around it.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the product library.  It
shares no code with the CUDA path.
"""
from .ns_fp64 import (  # noqa: F401
    DEFAULT_COEFFS,
    DEFAULT_EPS,
    DEFAULT_STEPS,
    frobenius_norm,
    gram,
    newton_schulz,
    newton_schulz_batched,
    newton_schulz_trace,
    normalize,
    poly,
    update,
)
from .muon_step import (  # noqa: F401
    apply_update,
    default_scale,
    momentum_update,
    muon_step,
    ns_input,
    round_bf16,
)
