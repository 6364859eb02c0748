"""Checks of the seeded input generator and of the stored golden values."""
import glob
import os

import numpy as np
import pytest
import torch

import ns_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(path):
    rec = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#"):
                continue
            key, _, rest = line.strip().partition(" ")
            rec[key] = rest.split()
    shape = tuple(int(v) for v in rec["shape"])
    bits = np.array([int(v, 16) for v in rec["input_bf16_hex"]], dtype=np.uint16).reshape(shape)
    out = np.array([float(v) for v in rec["output_f64"]]).reshape(shape)
    return bits, out


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "ns_*.txt"))))
def test_golden_oracle_outputs(path):
    bits, expect = _read_golden(path)
    got = oracle.newton_schulz(ns_inputs.bf16_bits_to_f64(bits))
    assert np.max(np.abs(got - expect)) <= 1e-13 * np.max(np.abs(expect))


def test_golden_inputs_regenerate_bitwise():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    for name, batch, rows, cols, seed in mg.CASES:
        bits, _ = _read_golden(os.path.join(GOLDEN, f"ns_{name}.txt"))
        w = ns_inputs.Workload(name, batch, rows, cols, "iid", seed=seed)
        np.testing.assert_array_equal(ns_inputs.stack_bits(w), bits)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 0.02,
        rng.standard_normal(1000).astype(np.float32) * 1e30,
        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3.0e-39, 65504.0], dtype=np.float32),
        # exact ties: low 16 bits 0x8000 with even and odd bf16 mantissas
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF], dtype=np.uint32).view(np.float32),
    ])
    ours = ns_inputs.fp32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # Widening is exact.
    np.testing.assert_array_equal(ns_inputs.bf16_bits_to_f32(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_per_matrix_seeding_is_independent_of_batch():
    w = ns_inputs.WORKLOADS["tiny_4x256x512"]
    full = ns_inputs.stack_bits(w)
    np.testing.assert_array_equal(full[2], ns_inputs.matrix_bits(w, 2))
    np.testing.assert_array_equal(ns_inputs.stack_bits(w, batch=2), full[:2])


def test_distributions():
    w = ns_inputs.WORKLOADS["tiny_4x256x512"]
    g = ns_inputs.matrix_f32(w, 0)
    assert abs(g.std() - 0.02) < 0.001 and abs(g.mean()) < 0.001
    e = ns_inputs.Workload("e", 8, 64, 64, "expert", seed=3)
    scales = [ns_inputs.matrix_f32(e, k).std() / 0.02 for k in range(8)]
    assert all(0.09 < s < 11 for s in scales) and max(scales) / min(scales) > 1.5
    r = ns_inputs.Workload("r", 1, 512, 384, "rank64", seed=4)
    sv = np.linalg.svd(ns_inputs.matrix_f32(r, 0).astype(np.float64), compute_uv=False)
    # 64 dominant singular values in about [1e-3, 1], then the noise floor.
    assert sv[0] < 2.0 and sv[0] > 0.2
    assert sv[70] < 0.02


def test_workloads_cover_the_pages_shapes():
    shapes = set()
    with open(os.path.join(GOLDEN, "pages_h200_ns_microbench.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, r, c = (int(v) for v in line.split()[:3])
            shapes.add((b, r, c))
    ours = {(w.batch, w.rows, w.cols) for w in ns_inputs.WORKLOADS.values()}
    assert shapes <= ours


def test_flop_model():
    w = ns_inputs.WORKLOADS["square_4096"]
    assert w.dense_flops() == 5 * (4 * 4096 ** 3 + 2 * 4096 ** 3)
    # The pages' H200 4096^2 QuACK time, 2.71 ms, is 761 dense-equivalent TFLOP/s.
    assert abs(w.dense_flops() / 2.71e-3 / 1e12 - 761) < 1
    t = ns_inputs.WORKLOADS["stack_128x2048x768"]
    assert (t.m, t.n, t.transposed) == (768, 2048, True)
