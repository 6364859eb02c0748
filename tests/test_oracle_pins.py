"""Pins for the fp64 oracle: checks against what the mathematics fixes, never
against the oracle's own formula retyped.

  * closed form: for X = U S V^T, one NS step maps X to U p(S) V^T with
    p(s) = a s + b s^3 + c s^5, so NS(G) = U p^{o steps}(S / (||G||_F + eps)) V^T
    (thin SVD from LAPACK, a library routine independent of the oracle);
  * special cases with scalar closed forms (scaled partial isometry, rank one,
    zero matrix, steps = 0);
  * invariants (exact symmetry of A and B, transpose invariance, batched equals
    per-matrix, orthogonal invariance, internal m <= n orientation);
  * planted mistakes: each plausible error in the oracle makes a pin fail.
"""
import numpy as np
import pytest

import oracle
from oracle import ns_fp64 as ns_mod

COEFFS = oracle.DEFAULT_COEFFS
EPS = oracle.DEFAULT_EPS


def closed_form(G, steps=5, coeffs=COEFFS, eps=EPS):
    G = np.asarray(G, dtype=np.float64)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    nu = np.sqrt(np.sum(S * S))  # ||G||_F from the singular values
    s = S / (nu + eps)
    for _ in range(steps):
        s = coeffs[0] * s + coeffs[1] * s ** 3 + coeffs[2] * s ** 5
    return (U * s[None, :]) @ Vt


def rel_err(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


SHAPES = [(8, 16), (16, 16), (24, 8), (5, 40), (33, 17), (1, 9), (9, 1)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [0, 1, 2, 5, 7])
def test_closed_form_svd(shape, steps):
    G = rand(shape, seed=hash((shape, steps)) % 1000)
    got = oracle.newton_schulz(G, steps=steps)
    ref = closed_form(G, steps=steps)
    assert got.shape == G.shape
    assert rel_err(got, ref) < 1e-12


@pytest.mark.parametrize("coeffs", [COEFFS, (2.0, -1.5, 0.5), (1.875, -1.25, 0.375)])
def test_closed_form_other_coefficients(coeffs):
    G = rand((12, 20), seed=7, scale=0.3)
    assert rel_err(oracle.newton_schulz(G, coeffs=coeffs), closed_form(G, coeffs=coeffs)) < 1e-12


def test_closed_form_batched_stack_with_per_matrix_scales():
    rng = np.random.default_rng(3)
    G = rng.standard_normal((3, 12, 20)) * np.array([0.01, 1.0, 100.0])[:, None, None]
    got = oracle.newton_schulz(G)
    for k in range(3):
        assert rel_err(got[k], closed_form(G[k])) < 1e-12


def test_scaled_partial_isometry():
    # G = sigma * Q with orthonormal rows: every singular value is sigma and
    # ||G||_F = sigma sqrt(m), so NS(G) = p^5(sigma / (sigma sqrt(m) + eps)) Q.
    m, n, sigma = 6, 10, 0.37
    Qfull, _ = np.linalg.qr(rand((n, n), seed=11))
    Q = Qfull[:m, :]
    got = oracle.newton_schulz(sigma * Q)
    s0 = sigma / (sigma * np.sqrt(m) + EPS)
    s = s0
    for _ in range(5):
        s = 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5
    assert rel_err(got, s * Q) < 1e-13


def test_rank_one():
    u = rand(7, seed=1)
    v = rand(13, seed=2)
    G = np.outer(u, v)
    nu = np.linalg.norm(u) * np.linalg.norm(v)
    s = nu / (nu + EPS)
    for _ in range(5):
        s = 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5
    expect = s * np.outer(u / np.linalg.norm(u), v / np.linalg.norm(v))
    assert rel_err(oracle.newton_schulz(G), expect) < 1e-13
    # Tall rank one goes through the transposed branch.
    assert rel_err(oracle.newton_schulz(G.T), expect.T) < 1e-13


def test_zero_matrix_gives_zero():
    out = oracle.newton_schulz(np.zeros((4, 8, 16)))
    assert np.all(out == 0.0)
    assert np.all(np.isfinite(out))


def test_steps_zero_is_normalisation():
    G = rand((9, 14), seed=5)
    out = oracle.newton_schulz(G, steps=0)
    np.testing.assert_array_equal(out, G / (np.sqrt(np.sum(G * G)) + EPS))


def test_frobenius_norm_matches_lapack():
    G = rand((17, 23), seed=9)
    assert abs(oracle.frobenius_norm(G) - np.linalg.norm(G, "fro")) < 1e-12 * np.linalg.norm(G)
    assert abs(oracle.frobenius_norm(G) - np.linalg.norm(np.linalg.svd(G, compute_uv=False))) < 1e-12 * np.linalg.norm(G)


@pytest.mark.parametrize("shape", [(8, 16), (16, 16), (24, 8)])
def test_gram_and_poly_are_exactly_symmetric(shape):
    tr = oracle.newton_schulz_trace(rand(shape, seed=4))
    for A, B in zip(tr["A"], tr["B"]):
        assert np.array_equal(A, A.T)
        assert np.array_equal(B, B.T)


@pytest.mark.parametrize("shape", [(8, 16), (24, 8), (16, 16), (30, 12)])
def test_internal_orientation_rows_le_cols(shape):
    tr = oracle.newton_schulz_trace(rand(shape, seed=8))
    m = min(shape)
    assert tr["transposed"] == (shape[0] > shape[1])
    assert tr["X0"].shape == (m, max(shape))
    assert all(A.shape == (m, m) for A in tr["A"])


@pytest.mark.parametrize("shape", [(8, 16), (24, 8), (5, 40)])
def test_transpose_invariance_bitwise_non_square(shape):
    G = rand(shape, seed=12)
    np.testing.assert_array_equal(oracle.newton_schulz(G.T), oracle.newton_schulz(G).T)


def test_transpose_invariance_square():
    G = rand((16, 16), seed=13)
    assert rel_err(oracle.newton_schulz(G.T), oracle.newton_schulz(G).T) < 1e-12


def test_batched_equals_per_matrix_bitwise():
    G = rand((5, 10, 18), seed=14)
    got = oracle.newton_schulz(G)
    for k in range(5):
        np.testing.assert_array_equal(got[k], oracle.newton_schulz(G[k]))


def test_orthogonal_invariance():
    G = rand((10, 16), seed=15)
    Q, _ = np.linalg.qr(rand((10, 10), seed=16))
    P, _ = np.linalg.qr(rand((16, 16), seed=17))
    assert rel_err(oracle.newton_schulz(Q @ G @ P), Q @ oracle.newton_schulz(G) @ P) < 1e-12


# ---------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail.
# ---------------------------------------------------------------------------

def _closed_form_pins_pass():
    try:
        for shape, seed in [((8, 16), 21), ((16, 16), 22), ((24, 8), 23)]:
            G = rand(shape, seed=seed)
            if rel_err(oracle.newton_schulz(G), closed_form(G)) > 1e-12:
                return False
    except ValueError:  # shape mismatch from a transposed operand
        return False
    return True


def _orientation_pin_passes():
    tr = oracle.newton_schulz_trace(rand((24, 8), seed=24))
    return tr["A"][0].shape == (8, 8)


MISTAKES = {
    "dropped_cAA": ("poly", lambda A, b, c: b * A),
    "sign_flip_c": ("poly", lambda A, b, c: b * A - c * (A @ A)),
    "swapped_bc": ("poly", lambda A, b, c: c * A + b * (A @ A)),
    "dropped_aX": ("update", lambda X, B, a: B @ X),
    "right_multiply": ("update", lambda X, B, a: a * X + X @ B),
    "gram_transposed": ("gram", lambda X: X.T @ X),
    "no_eps": ("normalize", lambda G, eps: np.asarray(G, np.float64) / np.sqrt(np.sum(np.asarray(G, np.float64) ** 2))),
    "norm_squared": ("normalize", lambda G, eps: np.asarray(G, np.float64) / (np.sum(np.asarray(G, np.float64) ** 2) + eps)),
    "spectral_norm": ("normalize", lambda G, eps: np.asarray(G, np.float64) / (np.linalg.norm(G, 2) + eps)),
}


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(monkeypatch, name):
    assert _closed_form_pins_pass()
    attr, fn = MISTAKES[name]
    monkeypatch.setattr(ns_mod, attr, fn)
    assert not _closed_form_pins_pass(), f"planted mistake {name} went unnoticed"


def test_planted_missing_transpose_is_caught(monkeypatch):
    # Skipping the transpose gives the same exact result (the SVD closed form is
    # orientation-free), so it is the orientation pin that must catch it.
    assert _orientation_pin_passes()

    def trace_without_transpose(G, steps=5, coeffs=COEFFS, eps=EPS):
        a, b, c = coeffs
        X = ns_mod.normalize(G, eps)
        As = []
        for _ in range(steps):
            A = ns_mod.gram(X)
            X = ns_mod.update(X, ns_mod.poly(A, b, c), a)
            As.append(A)
        return {"A": As}

    monkeypatch.setattr(oracle, "newton_schulz_trace", trace_without_transpose)
    assert not _orientation_pin_passes()
