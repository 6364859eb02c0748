"""Helpers shared by the GPU tests: moving raw bf16 bits between numpy and
torch, and the per-matrix relative Frobenius error."""
import numpy as np
import torch

import ns_inputs

NS_TOL = 1.5e-2  # relative Frobenius error per matrix, GPU NS vs the fp64 oracle
# Matrices with fewer than 64 rows or columns have too few singular values for
# bf16 rounding noise to average out: a CPU model of the kernels' rounding
# (bf16 storage of A, O and X, exact fp32 products) gave up to 1.9e-2 (fused
# first step) and 3.7e-2 (scaled copy of G) on 40 random 8 x 8 matrices, and
# 2.8e-2 on 16 x 16, against at most 1.01e-2 from 32 x 64 upward.  Such
# edge-case shapes are held to 5e-2; every benchmark workload is >= 768.
NS_TOL_SMALL = 5e-2


def ns_tol(rows: int, cols: int) -> float:
    return NS_TOL if min(rows, cols) >= 64 else NS_TOL_SMALL


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
