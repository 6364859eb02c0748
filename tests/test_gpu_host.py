"""The host-buffer path (muon_ns_host): a stack held in host memory is
uploaded, orthogonalised and downloaded in chunks, the copies of one chunk
overlapping the compute of its neighbours.  The matrices of a stack are
independent and the kernels are batch-invariant, so the result must equal the
device call on the whole stack bit for bit, for any chunking (ragged last
chunk, one matrix per chunk, chunk larger than the stack), in place, from
pageable memory, and with a workspace reused by back-to-back calls."""
import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import ns_inputs
import oracle
from nsutil import NS_TOL, per_matrix_rel, random_bits, to_bits, to_dev

pytestmark = pytest.mark.gpu


def host(bits, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).clone()
    return t.pin_memory() if pinned else t


def host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def device_ref(bits, steps=5):
    # Own workspace: the library-cached one must not grow here (a later test
    # relies on its size).
    return to_bits(ns.muon_ns(to_dev(bits), steps=steps, workspace=ns.alloc_workspace(*bits.shape)))


@pytest.mark.parametrize("chunk", [0, 1, 3, 4, 9, 100])
def test_host_path_equals_device_call_bitwise(chunk):
    # Largest chunk 3: chunks of 2, 3, 3, 2; 4: 2, 4, 2, 2; 9: 5, 5.
    bits = random_bits((10, 136, 264), seed=51)
    G = host(bits)
    out = ns.muon_ns_host(G, chunk=chunk)
    np.testing.assert_array_equal(host_bits(out), device_ref(bits))


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 4, 5, 7])
def test_host_path_tall_input_and_step_counts(steps):
    # Chunks of 1, 2, 1, 1 matrices (single-matrix chunks wait for whole
    # kernels, the other one through counters); odd and even step counts end
    # the iterate in different buffers of a chunk's slot.
    bits = random_bits((5, 264, 136), seed=52)
    G = host(bits)
    out = ns.muon_ns_host(G, steps=steps, chunk=2)
    np.testing.assert_array_equal(host_bits(out), device_ref(bits, steps))


def test_host_path_in_place_and_pageable():
    bits = random_bits((6, 256, 512), seed=53)
    ref = device_ref(bits)
    G = host(bits)
    ns.muon_ns_host(G, out=G, chunk=2)  # in place, pinned
    np.testing.assert_array_equal(host_bits(G), ref)
    Gp = host(bits, pinned=False)
    out = ns.muon_ns_host(Gp, chunk=4)  # pageable: same result, no overlap
    np.testing.assert_array_equal(host_bits(out), ref)


def test_host_path_expert_stack_vs_device_and_oracle():
    w = ns_inputs.WORKLOADS["experts_16x1536x2048"]
    bits = ns_inputs.stack_bits(w)
    G = host(bits)
    got = host_bits(ns.muon_ns_host(G))  # default: chunks of 4, 8, 4 matrices
    np.testing.assert_array_equal(got, device_ref(bits))
    for k in (0, 15):
        ref = oracle.newton_schulz(ns_inputs.bf16_bits_to_f64(bits[k]))
        assert per_matrix_rel(ns_inputs.bf16_bits_to_f64(got[k]), ref)[0] <= NS_TOL


def test_host_path_reused_workspace_and_error_word():
    bits = random_bits((4, 256, 512), seed=54)
    ws = torch.empty(ns.host_workspace_size(4, 256, 512, 1), dtype=torch.uint8, device="cuda")
    G1, G2 = host(bits), host(bits)
    a = ns.muon_ns_host(G1, chunk=1, workspace=ws, sync=False)
    b = ns.muon_ns_host(G2, chunk=1, workspace=ws, sync=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(a), host_bits(b))
    np.testing.assert_array_equal(host_bits(a), device_ref(bits))
    assert ns.read_error(ws) == 0


def test_host_path_workspace_too_small():
    G = host(random_bits((4, 256, 512), seed=55))
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(ns.MuonNSError):
        ns.muon_ns_host(G, workspace=ws)


def test_host_path_stack_beyond_the_grid_y_limit():
    # 70,000 matrices in one chunk: the norm pass, which runs on the upload
    # stream, loops past the grid's y limit; same bits as the device call.
    bits = random_bits((70000, 8, 16), seed=56)
    out = ns.muon_ns_host(host(bits))
    np.testing.assert_array_equal(host_bits(out), device_ref(bits))
