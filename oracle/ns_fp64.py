"""Plain fp64 CPU oracle for the quintic Newton–Schulz (NS) orthogonalisation.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA library.

What it computes (the algorithm's steps, in the pages' order and notation):

  1. X <- G / (||G||_F + eps)                      (Frobenius normalisation)
  2. if rows > cols: X <- X^T                      (so that X is m x n, m <= n)
  3. repeat `steps` times:
        A = X X^T                                   (the Gram matrix)
        B = b A + c A A
        X = a X + B X
  4. if transposed in step 2: X <- X^T

The three products of step 3 are the ones named by prime-rl PR #3873, Summary
item 1 ("Symmetric-GEMM Newton–Schulz"): X·X^T, b·A + c·A·A and a·X + B·X,
inside Dion's dense zeropower_via_newtonschulz5.  The step count 5 is the
`ns_steps` default of param-decomp PR #978 ("stacked-NS Muon", What).  The
batch semantics (the leading axis of a 3-D stack is a batch of independent
matrices) are prime-rl PR #3873, Summary item 2, and param-decomp PR #978,
What (leaves of one shape are stacked into a single NS).

The pages name this function but do not print its constants.  The readings
taken here, which the rest of the pages support:
  * (a, b, c) = (3.4445, -4.7750, 2.0315), the standard Muon quintic, the same
    for every step;
  * normalisation divides by ||G||_F + eps with eps = 1e-7;
  * the transpose is taken iff rows > cols (square inputs are not transposed);
  * every step runs in fp64 with no intermediate rounding.  prime-rl PR #3873
    (Results) measures bf16 NS against an fp32 NS that uses the same
    coefficients; fp64 is the stricter reference.

Each step is a module-level function so that a test can replace one of them
with a planted mistake and check that the pins catch it.  The matrix products
use numpy's matmul (a library primitive); there is no blocking, fusion or
reordering beyond the definition above.
"""
from __future__ import annotations

import numpy as np

DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)
DEFAULT_EPS = 1e-7
DEFAULT_STEPS = 5

__all__ = [
    "DEFAULT_COEFFS",
    "DEFAULT_EPS",
    "DEFAULT_STEPS",
    "frobenius_norm",
    "normalize",
    "gram",
    "poly",
    "update",
    "newton_schulz",
    "newton_schulz_trace",
    "newton_schulz_batched",
]


def frobenius_norm(G: np.ndarray) -> float:
    """||G||_F = sqrt(sum of squared entries), in fp64."""
    g = np.asarray(G, dtype=np.float64)
    return float(np.sqrt(np.sum(g * g)))


def normalize(G: np.ndarray, eps: float) -> np.ndarray:
    """Step 1: X = G / (||G||_F + eps)."""
    g = np.asarray(G, dtype=np.float64)
    return g / (frobenius_norm(g) + eps)


def gram(X: np.ndarray) -> np.ndarray:
    """A = X X^T (m x m) for X of shape m x n."""
    return X @ X.T


def poly(A: np.ndarray, b: float, c: float) -> np.ndarray:
    """B = b A + c A A."""
    return b * A + c * (A @ A)


def update(X: np.ndarray, B: np.ndarray, a: float) -> np.ndarray:
    """X' = a X + B X."""
    return a * X + B @ X


def newton_schulz_trace(G: np.ndarray, steps: int = DEFAULT_STEPS,
                        coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS):
    """Run NS on one 2-D matrix and return every intermediate.

    Returns a dict with keys
      "transposed": bool, "X0": the normalised (and possibly transposed) input,
      "A", "B", "X": lists with one entry per step (internal orientation),
      "out": the result in the input's orientation.
    """
    G = np.asarray(G, dtype=np.float64)
    if G.ndim != 2:
        raise ValueError("newton_schulz_trace takes one 2-D matrix")
    a, b, c = (float(v) for v in coeffs)
    X = normalize(G, eps)
    transposed = G.shape[0] > G.shape[1]
    if transposed:
        X = X.T
    X0 = X
    As, Bs, Xs = [], [], []
    for _ in range(int(steps)):
        A = gram(X)
        B = poly(A, b, c)
        X = update(X, B, a)
        As.append(A)
        Bs.append(B)
        Xs.append(X)
    out = X.T if transposed else X
    return {"transposed": transposed, "X0": X0, "A": As, "B": Bs, "X": Xs,
            "out": np.ascontiguousarray(out)}


def newton_schulz(G: np.ndarray, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
                  eps: float = DEFAULT_EPS) -> np.ndarray:
    """NS of one 2-D matrix, or of every matrix of a 3-D stack (leading axis =
    batch).  Returns fp64 in the input's shape."""
    G = np.asarray(G, dtype=np.float64)
    if G.ndim == 3:
        return newton_schulz_batched(G, steps, coeffs, eps)
    return newton_schulz_trace(G, steps, coeffs, eps)["out"]


def newton_schulz_batched(G: np.ndarray, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
                          eps: float = DEFAULT_EPS) -> np.ndarray:
    """NS applied independently to each matrix of a (batch, rows, cols) stack."""
    G = np.asarray(G, dtype=np.float64)
    if G.ndim != 3:
        raise ValueError("newton_schulz_batched takes a 3-D stack")
    out = np.empty_like(G)
    for k in range(G.shape[0]):
        out[k] = newton_schulz_trace(G[k], steps, coeffs, eps)["out"]
    return out

