"""fp32 NS (muon_ns_ws_f32): fp32 in and out, fp32 storage of X, A and B
rounded to tf32, tf32 tensor cores, fp32 epilogues.

Tolerance, from the CPU rounding model of exactly this path
(tests/rounding_model.py with storage="tf32": tf32 round-to-nearest storage of
the product operands, step 1's G read truncated to tf32, fp32 epilogues): it
gives 7.8e-4 to 9.9e-4 relative Frobenius error on the shapes below from
24 x 40 up, and 4.0e-3 on the 8 x 8 one.  The tests use 3e-3 and, below 64
rows or columns, 1.5 times the model's error on the same input when that is
larger (nsutil.model_tols).  The fp32 path must also beat the bf16 path on
the same input.
"""
import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
import ns_inputs
import oracle
from nsutil import model_tols, per_matrix_rel, random_bits, to_f64, to_dev

pytestmark = pytest.mark.gpu


F32_TOL = 3e-3


def f32_tols(x):
    return model_tols(np.asarray(x, dtype=np.float64), F32_TOL, "tf32")


def rand_f32(shape, seed, scale=0.02):
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(scale)


def run_f32(x, steps=5):
    G = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    shape = x.shape if x.ndim == 3 else (1,) + x.shape
    ws = torch.empty(ns.f32_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    out = ns.muon_ns_f32(G, steps=steps, workspace=ws)
    assert ns.read_error(ws) == 0
    return out, ws


def errs_vs_oracle(out, x, steps=5):
    return per_matrix_rel(out.double().cpu().numpy(), oracle.newton_schulz(x.astype(np.float64), steps))


@pytest.mark.parametrize("shape", [(4, 256, 512), (4, 512, 256), (3, 136, 264), (2, 264, 136), (1, 392, 392),
                                   (1, 8, 8), (2, 40, 24), (1, 1000, 776)])
def test_f32_vs_oracle(shape):
    x = rand_f32(shape, seed=sum(shape))
    out, _ = run_f32(x)
    e = errs_vs_oracle(out, x)
    tols = f32_tols(x)
    assert all(v <= t for v, t in zip(e, tols)), (e, tols)


@pytest.mark.parametrize("steps", [0, 1, 3])
def test_f32_step_counts(steps):
    x = rand_f32((2, 136, 264), seed=50 + steps)
    out, _ = run_f32(x, steps=steps)
    e = errs_vs_oracle(out, x, steps)
    assert max(e) <= (1e-6 if steps == 0 else F32_TOL), e


def test_f32_more_accurate_than_bf16():
    w = ns_inputs.WORKLOADS["tiny_4x256x512"]
    bits = ns_inputs.stack_bits(w)
    x = ns_inputs.bf16_bits_to_f32(bits)  # the same values for both paths
    e32 = errs_vs_oracle(run_f32(x)[0], x)
    e16 = per_matrix_rel(to_f64(ns.muon_ns(to_dev(bits))), oracle.newton_schulz(x.astype(np.float64)))
    assert max(e32) < min(e16) / 3, (e32, e16)


def test_f32_gram_and_poly_bit_symmetric():
    shape = (3, 264, 520)
    x = rand_f32(shape, seed=7)
    _, ws = run_f32(x, steps=1)
    torch.cuda.synchronize()
    m = min(shape[1:])
    for region in (ns._lib.WS_GRAM, ns._lib.WS_POLY):
        off, nb = ns.f32_workspace_region(*shape, region)
        a = ws[off:off + nb].view(torch.int32).cpu().numpy().reshape(shape[0], m, m)
        np.testing.assert_array_equal(a, np.swapaxes(a, 1, 2))
        # stored rounded to tf32: the low 13 mantissa bits are zero
        assert np.all((a.view(np.uint32) & 0x1FFF) == 0)


def test_f32_batched_equals_per_matrix_and_in_place():
    x = rand_f32((4, 256, 384), seed=11)
    whole = run_f32(x)[0].cpu().numpy()
    for k in range(4):
        np.testing.assert_array_equal(run_f32(x[k:k + 1])[0].cpu().numpy()[0], whole[k])
    G = torch.from_numpy(x).cuda()
    ns.muon_ns_f32(G, out=G)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(G.cpu().numpy(), whole)


@pytest.mark.parametrize("name,sample", [("experts_128x1536x2048", [0, 127]), ("stack_128x2048x768", [0, 64]),
                                         ("square_4096", [0])])
def test_f32_full_size_sampled(name, sample):
    w = ns_inputs.WORKLOADS[name]
    x = np.stack([ns_inputs.matrix_f32(w, k) for k in range(w.batch)])
    out, _ = run_f32(x)
    got = out[sample].double().cpu().numpy()
    e = [per_matrix_rel(got[i], oracle.newton_schulz(x[k].astype(np.float64)))[0] for i, k in enumerate(sample)]
    print(name, "fp32 rel errors", e)
    assert max(e) <= F32_TOL, e


def test_f32_error_tracks_the_rounding_model():
    # As for the bf16 path: the fp32 mode's error against the oracle agrees
    # with the CPU rounding model of tf32 storage on the same input.
    import rounding_model

    x = rand_f32((2, 256, 512), seed=77)
    e = errs_vs_oracle(run_f32(x)[0], x)
    model = [per_matrix_rel(rounding_model.model_ns(x[k].astype(np.float64), storage="tf32"),
                            oracle.newton_schulz(x[k].astype(np.float64)))[0] for k in range(2)]
    for v, vm in zip(e, model):
        assert abs(v - vm) <= 0.15 * vm, (e, model)
