"""muon_ns_grouped: several stacks of different shapes in one call.

Each tile of a launch depends only on its own matrix and contraction length,
so a grouped call must give results bit-identical to one muon_ns_ws call per
stack; and the mixed tall-stack workload (32 x 7168 x 2048 with
128 x 2048 x 768, one optimizer step's NS) is checked against the oracle on
sampled matrices.
"""
import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import ns_inputs
import oracle
from nsutil import NS_TOL, per_matrix_rel, random_bits, to_bits, to_dev, to_f64

pytestmark = pytest.mark.gpu

MIXED = [(3, 136, 264), (2, 264, 136), (4, 256, 512), (1, 392, 392), (2, 1040, 520), (1, 8, 8)]


def alone(G, steps=5):
    ws = ns.alloc_workspace(*([1] + list(G.shape) if G.dim() == 2 else G.shape))
    out = ns.muon_ns(G, steps=steps, workspace=ws)
    assert ns.read_error(ws) == 0
    return out


@pytest.mark.parametrize("steps", [5, 2])
def test_grouped_equals_separate_calls_bitwise(steps):
    Gs = [to_dev(random_bits(s, seed=300 + i)) for i, s in enumerate(MIXED)]
    ws = torch.empty(ns.grouped_workspace_size(Gs), dtype=torch.uint8, device="cuda")
    outs = ns.muon_ns_grouped(Gs, steps=steps, workspace=ws)
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    for G, o in zip(Gs, outs):
        np.testing.assert_array_equal(to_bits(o), to_bits(alone(G, steps)))


def test_grouped_long_contractions_mixed_batches_bitwise():
    # Contractions above 1024 (2-SM pairs) with a single-matrix stack in the
    # same launches as multi-matrix stacks: the latter order their products
    # through per-matrix counters, the former through whole kernels.
    shapes = [(2, 1040, 1280), (1, 1032, 1032), (3, 1280, 1040)]
    Gs = [to_dev(random_bits(s, seed=320 + i)) for i, s in enumerate(shapes)]
    ws = torch.empty(ns.grouped_workspace_size(Gs), dtype=torch.uint8, device="cuda")
    outs = ns.muon_ns_grouped(Gs, steps=3, workspace=ws)
    torch.cuda.synchronize()
    assert ns.read_error(ws) == 0
    for G, o in zip(Gs, outs):
        np.testing.assert_array_equal(to_bits(o), to_bits(alone(G, 3)))


def test_grouped_more_than_eight_stacks_and_in_place():
    shapes = [(2, 128 + 8 * i, 256) for i in range(10)] + [(1, 512, 256), (1, 264, 136)]
    Gs = [to_dev(random_bits(s, seed=400 + i)) for i, s in enumerate(shapes)]
    refs = [alone(G) for G in Gs]
    ns.muon_ns_grouped(Gs, outs=Gs)  # in place: 10 wide stacks (two launches) and 2 tall ones
    torch.cuda.synchronize()
    for G, r in zip(Gs, refs):
        np.testing.assert_array_equal(to_bits(G), to_bits(r))


def test_grouped_skips_empty_stacks():
    Gs = [torch.empty((0, 256, 512), dtype=torch.bfloat16, device="cuda"),
          to_dev(random_bits((2, 256, 512), seed=5))]
    outs = ns.muon_ns_grouped(Gs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(outs[1]), to_bits(alone(Gs[1])))


def test_mixed_tall_stacks_workload_vs_oracle():
    names = ["stack_32x7168x2048", "stack_128x2048x768"]
    bits = [ns_inputs.stack_bits(ns_inputs.WORKLOADS[n]) for n in names]
    Gs = [to_dev(b) for b in bits]
    outs = ns.muon_ns_grouped(Gs)
    torch.cuda.synchronize()
    for b, o, sample in zip(bits, outs, ([0, 31], [0, 127])):
        got = to_f64(o[sample])
        errs = [per_matrix_rel(got[i], oracle.newton_schulz(ns_inputs.bf16_bits_to_f64(b[k])))[0]
                for i, k in enumerate(sample)]
        assert max(errs) <= NS_TOL, errs
