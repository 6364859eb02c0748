"""Plain fp64 CPU oracle for the Muon optimizer step around Newton–Schulz.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: nothing on the product
path may import, call or execute it; it shares no code with the CUDA library.

The pages name the step but print no formula for it.  prime-rl PR #3873
(Summary) speeds up "the Muon optimizer step" whose inner loop is the NS of
oracle/ns_fp64.py; param-decomp PR #978 (What, the `ns_dtype` setting) runs
that NS in bf16 while "masters/momentum stay fp32".  The reading taken here,
per matrix W (fp32 master, rows x cols) with gradient G (fp32) and momentum
buffer M (fp32):

  1. M' = mu M + G                                   (momentum)
  2. U  = G + mu M'  (Nesterov)   or   U = M'         (plain momentum)
  3. O  = NS(bf16(U))                                 (bf16 NS, ns_dtype bfloat16)
  4. W' = (1 - lr wd) W - lr scale O                  (decoupled weight decay,
                                                       shape factor `scale`)

with `scale` defaulting to sqrt(max(1, rows / cols)) (the update of a tall
matrix is scaled up so that its per-entry size matches that of a wide one).
Steps 1, 2 and 4 run in fp64 with no rounding; the NS input is U rounded once
to the nearest bf16 (ties to even), because the NS precision is part of the
method's setting; the NS itself is the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np

from .ns_fp64 import DEFAULT_COEFFS, DEFAULT_EPS, DEFAULT_STEPS, newton_schulz

__all__ = ["default_scale", "round_bf16", "momentum_update", "ns_input", "apply_update", "muon_step"]


def default_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows / cols))."""
    return math.sqrt(max(1.0, rows / cols))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round each value to the nearest bfloat16 (8 significant bits, ties to
    even), returned as fp64.  Exact for every finite value of magnitude at
    least 2^-126 (the smallest normal bf16); zero stays zero."""
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)  # x = f 2^e, 0.5 <= |f| < 1
    return np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)  # rint rounds half to even


def momentum_update(M: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Step 1: M' = mu M + G."""
    return mu * np.asarray(M, dtype=np.float64) + np.asarray(G, dtype=np.float64)


def ns_input(G: np.ndarray, M_new: np.ndarray, mu: float, nesterov: bool) -> np.ndarray:
    """Step 2: U = G + mu M' with Nesterov momentum, else U = M'."""
    M_new = np.asarray(M_new, dtype=np.float64)
    return np.asarray(G, dtype=np.float64) + mu * M_new if nesterov else M_new


def apply_update(W: np.ndarray, O: np.ndarray, lr: float, weight_decay: float, scale: float) -> np.ndarray:
    """Step 4: W' = (1 - lr wd) W - lr scale O."""
    return (1.0 - lr * weight_decay) * np.asarray(W, dtype=np.float64) - lr * scale * np.asarray(O, dtype=np.float64)


def muon_step(W, M, G, lr: float, momentum: float, nesterov: bool = True, weight_decay: float = 0.0,
              scale: float | None = None, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
              eps: float = DEFAULT_EPS):
    """One Muon step of a matrix or a (batch, rows, cols) stack.

    Returns (W', M', O) in fp64, O being the orthogonalised update NS(bf16(U)).
    """
    W = np.asarray(W, dtype=np.float64)
    rows, cols = W.shape[-2], W.shape[-1]
    s = default_scale(rows, cols) if scale is None else float(scale)
    M_new = momentum_update(M, G, momentum)
    U = ns_input(G, M_new, momentum, nesterov)
    O = newton_schulz(round_bf16(U), steps, coeffs, eps)
    return apply_update(W, O, lr, weight_decay, s), M_new, O
