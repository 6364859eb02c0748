"""The CPU rounding model behind the GPU tests' tolerances (tests/rounding_model.py).

  * With every rounding switched off the model must equal the fp64 oracle
    (itself pinned to the SVD closed form), for the fused first step, the
    scaled-copy chain and the fp32 mode, wide and tall: so its arithmetic has
    no dropped term, wrong scale or transposed operand.
  * Its error figures back the two tolerance regimes: from 24 x 40 up the
    bf16 path stays well inside the 1.5e-2 bar (and the tf32 path inside
    3e-3), while random 8 x 8 matrices have a heavy tail well above it.
  * The per-input bounds that the GPU ragged-shape tests derive from it stay
    modest (the looser bound cannot hide a broken kernel).
"""
import numpy as np
import pytest

import ns_inputs
import oracle
import rounding_model as rm
from nsutil import NS_TOL, SMALL_MARGIN, model_tols, ns_tols, random_bits, rel_fro


def _no_rounding(monkeypatch):
    ident = lambda x: np.asarray(x, dtype=np.float64)  # noqa: E731
    for name in ("bf16", "f32", "tf32", "tf32_trunc"):
        monkeypatch.setattr(rm, name, ident)


@pytest.mark.parametrize("shape", [(8, 16), (24, 8), (16, 16), (40, 24)])
@pytest.mark.parametrize("variant", [dict(), dict(scaled_copy=True), dict(storage="tf32")])
@pytest.mark.parametrize("steps", [1, 5])
def test_without_rounding_equals_oracle(monkeypatch, shape, variant, steps):
    g = np.random.default_rng(sum(shape) + steps).standard_normal(shape) * 0.02
    _no_rounding(monkeypatch)
    got = rm.model_ns(g, steps=steps, **variant)
    assert rel_fro(got, oracle.newton_schulz(g, steps=steps)) < 1e-12


def test_rounding_helpers():
    x = np.array([1.0, 1.0 + 2.0 ** -9, 1.0 + 3 * 2.0 ** -9, -3.0e-3, 0.0])
    # bf16 keeps 7 stored mantissa bits (ulp 2^-7 at 1): 1 + 2^-9 rounds down, 1 + 3 * 2^-9 up.
    np.testing.assert_array_equal(rm.bf16(x)[:3], [1.0, 1.0, 1.0 + 2.0 ** -7])
    # tf32 keeps 10 (ulp 2^-10): 1 + 2^-11 is a tie (to even: 1), 1 + 3 * 2^-12 rounds up,
    # and truncation drops both.
    y = np.array([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -12])
    np.testing.assert_array_equal(rm.tf32(y), [1.0, 1.0 + 2.0 ** -10])
    np.testing.assert_array_equal(rm.tf32_trunc(y), [1.0, 1.0])
    assert rm.bf16(x)[4] == 0.0 and abs(rm.bf16(x)[3] + 3.0e-3) <= 2.0 ** -8 * 3.0e-3


def _errs(shape, seed, storage="bf16"):
    if storage == "bf16":
        g = ns_inputs.bf16_bits_to_f64(random_bits(shape, seed=seed))
    else:
        g = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32).astype(np.float64) * 0.02
    return np.array([rel_fro(rm.model_ns(g[k], storage=storage), oracle.newton_schulz(g[k]))
                     for k in range(shape[0])])


@pytest.mark.parametrize("shape", [(6, 24, 40), (6, 32, 64), (3, 64, 64), (2, 64, 128)])
def test_bf16_model_inside_the_bar_from_small_sizes_up(shape):
    e = _errs(shape, seed=31)
    assert e.max() < 0.75 * NS_TOL, e
    assert e.min() > 3e-3, e  # bf16 storage does cost something: the model is not a no-op


def test_tiny_squares_have_a_heavy_tail():
    e = _errs((200, 8, 8), seed=7)
    assert 5e-3 < np.median(e) < NS_TOL
    assert np.quantile(e, 0.99) > 1.5 * NS_TOL  # a flat 1.5e-2 cannot hold for 8 x 8


@pytest.mark.parametrize("shape", [(4, 24, 40), (2, 64, 128)])
def test_tf32_model_inside_its_bar(shape):
    e = _errs(shape, seed=41, storage="tf32")
    assert e.max() < 1.2e-3, e


# The ragged shapes of the bf16 GPU parity test (same inputs: random_bits with
# seed = sum(shape)) and the bounds they get.
RAGGED = [(1, 8, 8), (1, 8, 2048), (1, 2048, 8), (2, 40, 24)]


@pytest.mark.parametrize("shape", RAGGED)
def test_ragged_gpu_bounds_stay_modest(shape):
    bits = random_bits(shape, seed=sum(shape))
    tols = ns_tols(bits)
    assert all(NS_TOL <= t <= 2.5e-2 for t in tols), tols


def test_model_tols_regimes():
    big = np.zeros((2, 64, 64))
    assert model_tols(big, 7e-3) == [7e-3, 7e-3]
    g = ns_inputs.bf16_bits_to_f64(random_bits((1, 8, 8), seed=16))
    e = rel_fro(rm.model_ns(g[0]), oracle.newton_schulz(g[0]))
    assert model_tols(g, 1e-9) == [SMALL_MARGIN * e]
