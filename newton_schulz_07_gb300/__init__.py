"""Batched quintic Newton–Schulz orthogonalisation for GB300 (sm_103a).

The compute path is the CUDA library libmuon_ns.so (C ABI in
include/muon_ns.h); this package is its thin PyTorch binding.
"""
from ._lib import LIB_PATH, MuonNSError, lib  # noqa: F401
from .ns import (  # noqa: F401
    DEFAULT_COEFFS,
    DEFAULT_EPS,
    alloc_workspace,
    default_scale,
    error_status,
    launches_per_call,
    muon_ns,
    muon_ns_check,
    muon_ns_f32,
    f32_workspace_region,
    f32_workspace_size,
    muon_ns_gram,
    muon_ns_grouped,
    grouped_workspace_size,
    inject_stall,
    host_chunk,
    host_plan,
    host_workspace_size,
    muon_ns_host,
    muon_ns_normalize,
    muon_ns_normalize_static,
    muon_ns_poly,
    muon_ns_update,
    muon_apply,
    muon_momentum,
    muon_step,
    muon_step_grouped,
    read_error,
    set_wait_budget,
    step_grouped_workspace_size,
    step_launches,
    step_workspace_size,
    workspace_region,
    workspace_size,
)

__version__ = "0.1.0"
