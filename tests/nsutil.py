"""Helpers shared by the GPU tests: moving raw bf16 bits between numpy and
torch, and the per-matrix relative Frobenius error."""
import numpy as np
import torch

import ns_inputs

NS_TOL = 1.5e-2  # relative Frobenius error per matrix, GPU NS vs the fp64 oracle


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
