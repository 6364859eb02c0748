"""Helpers shared by the GPU tests: moving raw bf16 bits between numpy and
torch, and the per-matrix relative Frobenius error."""
import numpy as np
import torch

import ns_inputs

NS_TOL = 1.5e-2  # relative Frobenius error per matrix, GPU NS vs the fp64 oracle
# Matrices with fewer than 64 rows or columns have too few singular values for
# bf16 rounding noise to average out, and their error depends strongly on the
# matrix: the CPU rounding model of tests/rounding_model.py gives, on random
# 8 x 8 matrices, a median of 1.0e-2 but a 99th percentile of 3.0e-2
# (tests/test_rounding_model.py).  Such edge-case shapes are held to
# SMALL_MARGIN times the model's own error on the same input (at least
# NS_TOL); every benchmark workload is >= 256 on each side and keeps NS_TOL.
SMALL_MARGIN = 1.5
SMALL_DIM = 64


def model_tols(g: np.ndarray, base: float, storage: str = "bf16", steps: int = 5) -> list:
    """Per-matrix tolerance of a stack g [batch][rows][cols] (the input values
    as fp64): `base`, or for small shapes SMALL_MARGIN times the rounding
    model's error on the same matrix when that is larger."""
    g = g if g.ndim == 3 else g[None]
    if min(g.shape[1], g.shape[2]) >= SMALL_DIM:
        return [base] * g.shape[0]
    import oracle
    import rounding_model

    out = []
    for k in range(g.shape[0]):
        e = rel_fro(rounding_model.model_ns(g[k], steps=steps, storage=storage),
                    oracle.newton_schulz(g[k], steps=steps))
        out.append(max(base, SMALL_MARGIN * e))
    return out


def ns_tols(bits: np.ndarray, steps: int = 5) -> list:
    """Per-matrix tolerance of the bf16 path for a stack of bf16 bits."""
    return model_tols(ns_inputs.bf16_bits_to_f64(bits), NS_TOL, "bf16", steps)


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return ns_inputs.bf16_bits_to_f64(to_bits(t))


def rel_fro(x: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


def per_matrix_rel(x: np.ndarray, ref: np.ndarray) -> list:
    if x.ndim == 2:
        return [rel_fro(x, ref)]
    return [rel_fro(x[k], ref[k]) for k in range(x.shape[0])]


def random_bits(shape, seed, scale=0.02) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return ns_inputs.fp32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def symmetric_bits(batch, m, seed, scale=0.05) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, m, m), dtype=np.float32) * np.float32(scale)
    bits = ns_inputs.fp32_to_bf16_bits(x)
    lower = np.tril(bits)
    return lower + np.transpose(np.tril(bits, -1), (0, 2, 1))
