"""Failure detection on the GPU without a fault: a bounded wait runs out.

The library's host-side injection gives the first step's polynomial kernel a
per-matrix completion target one unit above what the Gram kernel signals, so
the producer's counter wait runs out after a short budget.  The kernel must
report it through the device error word (MUON_NS_ERR_TIMEOUT), every later
kernel of the call must give up when it sees the word, and the context must
stay usable: the next call, without the injection, gives the normal result.
Nothing here faults or hangs the GPU; every wait involved is bounded.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
from nsutil import random_bits, to_bits, to_dev

pytestmark = pytest.mark.gpu

BUDGET = 20_000_000  # SM clock cycles per wait, about 10 ms


# Short contractions (CTA pairs sharing a multicast panel) and long ones
# (2-SM MMAs).
@pytest.mark.parametrize("shape", [(2, 256, 512), (2, 1040, 1280)])
def test_counter_wait_that_runs_out_reports_timeout(shape):
    G = to_dev(random_bits(shape, seed=700))
    ws = ns.alloc_workspace(*shape)
    ref = ns.muon_ns(G, workspace=ns.alloc_workspace(*shape))
    torch.cuda.synchronize()
    ns.set_wait_budget(BUDGET)
    ns.inject_stall(True)
    try:
        t0 = time.monotonic()
        ns.muon_ns(G, workspace=ws)
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
    finally:
        ns.inject_stall(False)
        ns.set_wait_budget(0)
    assert ns.read_error(ws, clear=True) != 0
    # One wait ran out; the rest gave up on the error word.
    assert elapsed < 5.0
    # The context is usable and the workspace reusable.
    out = ns.muon_ns(G, workspace=ws)
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    np.testing.assert_array_equal(to_bits(out), to_bits(ref))


def test_check_inside_a_captured_graph_reports_timeout():
    # muon_ns_check enqueues the error word's copy into pinned host memory
    # without synchronising, so it is captured with the call.  A clean graph
    # reads 0; a graph captured while the stall is injected (its kernels carry
    # the unreachable target and the short budget) reads the timeout bit, and
    # the word maps to MUON_NS_ERR_TIMEOUT.
    shape = (2, 256, 512)
    G = to_dev(random_bits(shape, seed=701))
    ws = ns.alloc_workspace(*shape)
    out = torch.empty_like(G)
    word = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):  # first launches (per-device set-up) outside any capture
        ns.muon_ns(G, out=out, workspace=ws)
        ns.muon_ns_check(ws, word)
    cur.wait_stream(side)
    torch.cuda.synchronize()
    assert word.item() == 0

    def capture():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ns.muon_ns(G, out=out, workspace=ws)
            ns.muon_ns_check(ws, word)
        return g

    clean = capture()
    ns.set_wait_budget(BUDGET)
    ns.inject_stall(True)
    try:
        stalled = capture()
    finally:
        ns.inject_stall(False)
        ns.set_wait_budget(0)
    word.fill_(-1)
    clean.replay()
    torch.cuda.synchronize()
    assert word.item() == 0 and ns.error_status(word.item()) == ns._lib.OK
    t0 = time.monotonic()
    stalled.replay()
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 5.0
    assert word.item() & ns._lib.DEVERR_WAIT_TIMEOUT
    assert ns.error_status(word.item()) == ns._lib.ERR_TIMEOUT
    # The clean graph still runs clean on the same workspace afterwards.
    word.fill_(-1)
    clean.replay()
    torch.cuda.synchronize()
    assert word.item() == 0


def test_check_rejects_pageable_host_memory():
    ws = ns.alloc_workspace(2, 64, 128)
    pageable = torch.zeros(1, dtype=torch.int32)
    s = ns._lib.lib().muon_ns_check(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(pageable.data_ptr()), None)
    assert s == ns._lib.ERR_INVALID_ARG
