"""The whole call under CUDA-graph capture and on concurrent streams.

muon_ns_ws takes a caller-owned workspace and neither allocates nor
synchronises, so it can be captured into a CUDA graph and replayed; muon_ns
with the library's cached workspace refuses to grow that cache while the
stream is being captured.  Calls on different streams with their own
workspaces do not interfere.
"""
import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
from nsutil import random_bits, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(4, 256, 512), (3, 264, 136)])
def test_graph_capture_and_replay_matches_eager(shape):
    bits = random_bits(shape, seed=77)
    G = to_dev(bits)
    ws = ns.alloc_workspace(*shape)
    eager = ns.muon_ns(G, workspace=ws).clone()
    out = torch.empty_like(G)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ns.muon_ns(G, out=out, workspace=ws)  # warm-up on a side stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ns.muon_ns(G, out=out, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(out), to_bits(eager))
    # Replay on new input data in the same buffers.
    G.copy_(to_dev(random_bits(shape, seed=78)))
    g.replay()
    ref = ns.muon_ns(G, workspace=ns.alloc_workspace(*shape))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(out), to_bits(ref))
    assert ns.read_error(ws) == 0


# The refused call launches nothing, so the capture ends empty.
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_cached_workspace_does_not_grow_during_capture():
    big = (2, 2048, 3072)  # larger than anything the cache has held in this test process
    G = torch.zeros(big, dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with pytest.raises(ns.MuonNSError) as exc:
        with torch.cuda.graph(g):
            ns.muon_ns(G)
    assert exc.value.status == ns._lib.ERR_WORKSPACE


def test_concurrent_streams_with_own_workspaces():
    shape = (8, 384, 640)
    inputs = [to_dev(random_bits(shape, seed=90 + i)) for i in range(2)]
    refs = [ns.muon_ns(x, workspace=ns.alloc_workspace(*shape)).clone() for x in inputs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [ns.alloc_workspace(*shape) for _ in range(2)]
    outs = [torch.empty_like(x) for x in inputs]
    for _ in range(3):
        for x, o, w, st in zip(inputs, outs, wss, streams):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                ns.muon_ns(x, out=o, workspace=w)
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        np.testing.assert_array_equal(to_bits(o), to_bits(r))
