"""Pins for the Muon-step oracle (oracle/muon_step.py), against what the
mathematics fixes rather than the oracle's formulas retyped.

  * closed form: for G = sigma Q and M = tau Q with Q having orthonormal rows,
    every quantity is a multiple of Q, NS(c Q) = p^{o5}(c / (c sqrt(m) + eps)) Q,
    so W', M' and O have scalar closed forms;
  * exact Nesterov and plain-momentum inputs on values whose fp64 arithmetic
    is exact, and the momentum recurrence over two steps;
  * bf16 rounding against ties and against torch's conversion;
  * lr = 0 leaves W unchanged, and the change of W is linear in lr;
  * planted mistakes: each plausible error in the step makes a pin fail.
"""
import importlib

import numpy as np
import pytest
import torch

import oracle

ms = importlib.import_module("oracle.muon_step")  # the module (the package exports its function of that name)

COEFFS = oracle.DEFAULT_COEFFS
EPS = oracle.DEFAULT_EPS


def rel(x, y, den=None):
    d = np.linalg.norm(y) if den is None else den
    return float(np.linalg.norm(np.asarray(x) - np.asarray(y)) / max(d, 1e-300))


def p5(s, steps=5):
    a, b, c = COEFFS
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def hadamard_rows(m, n):
    """m orthonormal rows of length n (n a power of two), entries +-1/sqrt(n)."""
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H[:m] / np.sqrt(n)


def bf16_exact(shape, seed, bits=4):
    """Random values with few significant bits, so fp64 sums and products of
    them (and of mu = 0.5) are exact and bf16-representable."""
    rng = np.random.default_rng(seed)
    return rng.integers(-(2 ** bits), 2 ** bits, size=shape).astype(np.float64) / 2 ** bits


# ------------------------------------------------------------------- pins --

def pin_isometry(mu=0.5, lr=0.1, wd=0.5, scale=1.7, nesterov=True):
    m, n = 4, 16
    Q = hadamard_rows(m, n)  # entries +-1/4: bf16-exact multiples below
    sigma, tau = 1.0, 2.0
    G, M = sigma * Q, tau * Q
    W = np.random.default_rng(3).standard_normal((m, n))
    Wn, Mn, O = oracle.muon_step(W, M, G, lr, mu, nesterov=nesterov, weight_decay=wd, scale=scale)
    m_c = mu * tau + sigma
    u_c = sigma + mu * m_c if nesterov else m_c
    o_c = p5(u_c / (u_c * np.sqrt(m) + EPS))
    ok = rel(Mn, m_c * Q) < 1e-14
    ok &= rel(O, o_c * Q) < 1e-12
    ok &= rel(Wn, (1 - lr * wd) * W - lr * scale * o_c * Q, den=lr * scale * np.linalg.norm(O)) < 1e-12
    return ok


def pin_inputs_exact(nesterov):
    mu = 0.5
    G, M = bf16_exact((6, 10), 1), bf16_exact((6, 10), 2)
    _, _, O = oracle.muon_step(np.zeros((6, 10)), M, G, 0.0, mu, nesterov=nesterov)
    U = (1 + mu) * G + mu * mu * M if nesterov else mu * M + G
    return np.array_equal(O, oracle.newton_schulz(U))


def pin_two_steps(nesterov=True):
    mu, rng = 0.9, np.random.default_rng(4)
    M0, G1, G2 = (rng.standard_normal((5, 7)) for _ in range(3))
    W = rng.standard_normal((5, 7))
    W1, M1, _ = oracle.muon_step(W, M0, G1, 1e-2, mu, nesterov=nesterov)
    _, M2, _ = oracle.muon_step(W1, M1, G2, 1e-2, mu, nesterov=nesterov)
    return rel(M2, mu * mu * M0 + mu * G1 + G2) < 1e-14


def pin_bf16_ties():
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 * 2.0 ** -130 * 2 ** 10, 0.0])
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 3 * 2.0 ** -120, 0.0])
    return np.array_equal(oracle.round_bf16(x), want)


def all_pins_pass():
    return (pin_isometry() and pin_isometry(nesterov=False, wd=0.0, scale=1.0) and pin_inputs_exact(True)
            and pin_inputs_exact(False) and pin_two_steps() and pin_bf16_ties())


def test_isometry_closed_form():
    assert pin_isometry()
    assert pin_isometry(nesterov=False, wd=0.0, scale=1.0)
    assert pin_isometry(mu=0.0, lr=3e-3, wd=0.1, scale=1.0)


@pytest.mark.parametrize("nesterov", [True, False])
def test_ns_input_exact(nesterov):
    assert pin_inputs_exact(nesterov)


def test_momentum_two_steps():
    assert pin_two_steps(True) and pin_two_steps(False)


def test_bf16_rounding_ties_and_torch():
    assert pin_bf16_ties()
    x = (np.random.default_rng(5).standard_normal(20000) * 10.0 ** np.random.default_rng(6).integers(-20, 20, 20000))
    x = x.astype(np.float32).astype(np.float64)  # torch rounds through fp32; these are fp32 values already
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)


def test_lr_zero_and_linearity():
    rng = np.random.default_rng(7)
    W, M, G = (rng.standard_normal((2, 8, 12)) for _ in range(3))
    W0, M0, _ = oracle.muon_step(W, M, G, 0.0, 0.95, weight_decay=0.3)
    np.testing.assert_array_equal(W0, W)
    d1 = W - oracle.muon_step(W, M, G, 1e-3, 0.95, weight_decay=0.3)[0]
    d2 = W - oracle.muon_step(W, M, G, 2e-2, 0.95, weight_decay=0.3)[0]
    assert rel(d2, 20 * d1) < 1e-12
    np.testing.assert_array_equal(oracle.muon_step(W, M, G, 2e-2, 0.95)[1], M0)


def test_batched_equals_per_matrix_and_default_scale():
    rng = np.random.default_rng(8)
    W, M, G = (rng.standard_normal((3, 12, 8)) for _ in range(3))
    Wn, Mn, O = oracle.muon_step(W, M, G, 0.02, 0.9)
    for k in range(3):
        wk, mk, ok = oracle.muon_step(W[k], M[k], G[k], 0.02, 0.9)
        np.testing.assert_array_equal(Wn[k], wk)
        np.testing.assert_array_equal(O[k], ok)
    assert oracle.default_scale(2048, 768) == np.sqrt(2048 / 768)
    assert oracle.default_scale(768, 2048) == 1.0 and oracle.default_scale(64, 64) == 1.0
    # A tall matrix gets the larger factor in the update.
    assert rel(W[0] - Wn[0], 0.02 * np.sqrt(12 / 8) * O[0]) < 1e-12


MISTAKES = {
    "dampened_momentum": ("momentum_update", lambda M, G, mu: mu * (np.asarray(M) + np.asarray(G))),
    "nesterov_old_momentum": ("ns_input", lambda G, Mn, mu, nest: np.asarray(G) + mu * (np.asarray(Mn) - np.asarray(G)) / mu
                              if nest and mu else np.asarray(Mn)),
    "plain_uses_gradient": ("ns_input", lambda G, Mn, mu, nest: np.asarray(G) + mu * np.asarray(Mn) if nest else np.asarray(G)),
    "update_sign": ("apply_update", lambda W, O, lr, wd, s: (1 - lr * wd) * np.asarray(W) + lr * s * np.asarray(O)),
    "decay_after_update": ("apply_update", lambda W, O, lr, wd, s: (np.asarray(W) - lr * s * np.asarray(O)) * (1 - lr * wd)),
    "scale_dropped": ("apply_update", lambda W, O, lr, wd, s: (1 - lr * wd) * np.asarray(W) - lr * np.asarray(O)),
    "bf16_truncated": ("round_bf16", lambda x: np.ldexp(np.trunc(np.ldexp(np.frexp(x)[0], 8)), np.frexp(x)[1] - 8)),
}


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(monkeypatch, name):
    assert all_pins_pass()
    attr, fn = MISTAKES[name]
    monkeypatch.setattr(ms, attr, fn)
    if attr == "round_bf16":
        monkeypatch.setattr(oracle, "round_bf16", fn)
    assert not all_pins_pass(), f"planted mistake {name} went unnoticed"
