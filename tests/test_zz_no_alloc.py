"""The allocation-free normalisation entry point, muon_ns_normalize_static.

It exists for callers that cannot allocate device memory (a plugin handed
only its buffers, a host whose allocator forbids cudaMalloc, a loop that cannot
take cudaMalloc's synchronisation); its scratch is a fixed 1 MiB device array
inside the library.  Here it is called through the C ABI twice in a row, each
time against muon_ns_normalize (which takes a caller-allocated workspace) on
the same input, within the per-element bound the kernel tests use (one bf16
rounding, 2^-8 relative).  The second call checks that the scratch left over
from the first (tickets, partial sums) is cleared where it must be.

This file is collected last on purpose, so a failure here cannot hide any
other test in a run that stops at the first failure.
"""
import ctypes

import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import ns_inputs
import oracle
from newton_schulz_07_gb300 import _lib
from nsutil import random_bits, to_bits, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _static_call(G, X, eps=1e-7):
    b, r, c = G.shape
    return _lib.lib().muon_ns_normalize_static(
        ctypes.c_void_p(G.data_ptr()), ctypes.c_void_p(X.data_ptr()), b, r, c, ctypes.c_float(eps),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(4, 256, 512), (3, 264, 136)])
def test_static_scratch_matches_workspace_entry_point_two_calls(shape):
    for call in range(2):
        bits = random_bits(shape, seed=1000 * call + sum(shape), scale=0.02 * (1 + 9 * call))
        G = to_dev(bits)
        X_static = torch.empty_like(G)
        assert _static_call(G, X_static) == _lib.OK
        ws = ns.alloc_workspace(*shape)
        X_ref = ns.muon_ns_normalize(G, ws)
        torch.cuda.synchronize()
        got, ref = to_f64(X_static), to_f64(X_ref)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
        # Same kernels, same fixed reduction order: identical bits.
        np.testing.assert_array_equal(to_bits(X_static), to_bits(X_ref))
        # And against the definition, G / (||G||_F + eps) in fp64: one bf16
        # rounding (2^-8 relative) on top of an fp32 norm (1e-4 is ample).
        g = ns_inputs.bf16_bits_to_f64(bits)
        exact = np.stack([oracle.normalize(g[k], 1e-7) for k in range(shape[0])])
        assert np.all(np.abs(got - exact) <= (2.0 ** -8 + 1e-4) * np.abs(exact) + 1e-30)


def test_static_scratch_rejects_problems_beyond_its_size():
    # 1 MiB holds about 4 * batch * (chunks + 2) bytes, chunks = rows * cols / 16384;
    # 256 matrices of 8192 x 8192 need 256 * (4096 + 2) * 4 bytes (4 MiB).  The
    # call is rejected on the host before anything is launched, so the small
    # buffer passed here is never touched.
    G = torch.empty((1, 8, 8), dtype=torch.bfloat16, device="cuda")
    b, r, c = 256, 8192, 8192
    s = _lib.lib().muon_ns_normalize_static(ctypes.c_void_p(G.data_ptr()), ctypes.c_void_p(G.data_ptr()), b, r, c,
                                            ctypes.c_float(1e-7), None)
    assert s == _lib.ERR_WORKSPACE


def test_static_scratch_rejects_a_null_output():
    # Its norms stay in the library's private array, so a call without X
    # would compute nothing the caller can read: rejected before any launch.
    G = torch.empty((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    s = _lib.lib().muon_ns_normalize_static(ctypes.c_void_p(G.data_ptr()), None, 2, 64, 128,
                                            ctypes.c_float(1e-7), None)
    assert s == _lib.ERR_INVALID_ARG
