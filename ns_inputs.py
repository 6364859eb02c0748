"""Seeded synthetic inputs for batched Newton–Schulz (NS) orthogonalisation.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA
side (tests, bench): it generates matrices and nothing else.  It holds none of
the method's arithmetic (no norms, no products, no polynomial); it only draws
random numbers, applies the stated distribution, and rounds fp32 to bf16.

Workload shapes follow the pages:
  * prime-rl PR #3873, "NS microbenchmark on one H200" table: 4096x4096,
    8192x8192, 4096x14336, 128x1536x2048, 128x2048x768, 32x7168x2048;
  * prime-rl PR #3873, Summary item 2: the local expert-shard stack
    (16, 1536, 2048) next to Dion's padded (128, 1536, 2048).
The distributions (i.i.d. Gaussian gradients, a rank-64 spectrum plus noise,
per-expert log-uniform scales) are synthetic stand-ins for the pages' "random
grads"; no dataset is involved.

Every matrix k of a stack is drawn from its own generator seeded with
(seed, k), so any single matrix can be regenerated alone (sampled parity at full
size) and a stack's contents do not depend on how many matrices it holds.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "fp32_to_bf16_bits",
    "bf16_bits_to_f64",
    "bf16_bits_to_f32",
    "matrix_f32",
    "matrix_bits",
    "stack_bits",
]


@dataclass(frozen=True)
class Workload:
    """One NS workload: a stack of `batch` matrices of `rows` x `cols`.

    dist:
      "iid"      entries i.i.d. N(0, sigma^2)
      "expert"   i.i.d. N(0, sigma^2) times a per-matrix scale drawn
                 log-uniform in [scale_lo, scale_hi]
      "rank64"   U diag(s) V^T + N(0, noise^2), U (rows x 64) and V (cols x 64)
                 with i.i.d. N(0, 1/rows) and N(0, 1/cols) entries so that the
                 columns are close to unit norm and s are close to the singular
                 values of the low-rank part; s log-uniform in [1e-3, 1]
    """

    name: str
    batch: int
    rows: int
    cols: int
    dist: str = "iid"
    sigma: float = 0.02
    scale_lo: float = 0.1
    scale_hi: float = 10.0
    rank: int = 64
    noise: float = 1e-4
    seed: int = 1234
    note: str = field(default="", compare=False)

    @property
    def transposed(self) -> bool:
        return self.rows > self.cols

    @property
    def m(self) -> int:
        return min(self.rows, self.cols)

    @property
    def n(self) -> int:
        return max(self.rows, self.cols)

    def dense_flops(self, steps: int = 5) -> float:
        """Dense-GEMM-equivalent FLOPs of one NS call: per matrix and step,
        X X^T (2 m^2 n) + A A (2 m^3) + B X (2 m^2 n)."""
        m, n = float(self.m), float(self.n)
        return steps * self.batch * (4.0 * m * m * n + 2.0 * m * m * m)

    def useful_flops(self, steps: int = 5) -> float:
        """FLOPs when the two symmetric products compute one triangle only:
        m(m+1)n for X X^T, m^2(m+1) for A A, 2 m^2 n for B X."""
        m, n = float(self.m), float(self.n)
        return steps * self.batch * (m * (m + 1) * n + m * m * (m + 1) + 2.0 * m * m * n)

    def with_batch(self, batch: int) -> "Workload":
        return Workload(self.name, batch, self.rows, self.cols, self.dist, self.sigma,
                        self.scale_lo, self.scale_hi, self.rank, self.noise, self.seed, self.note)


# The workloads, named by what they are.  Seeds are fixed per workload.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_4x256x512", 4, 256, 512, "iid", seed=1234,
                 note="tiny batched case, wide"),
        Workload("tiny_4x512x256", 4, 512, 256, "iid", seed=1235,
                 note="tiny batched case, tall (transposed internally)"),
        Workload("square_4096", 1, 4096, 4096, "rank64", seed=1236,
                 note="single square matrix, rank-64 spectrum plus noise"),
        Workload("wide_4096x14336", 1, 4096, 14336, "iid", seed=1237,
                 note="single wide MLP-projection matrix"),
        Workload("square_8192", 1, 8192, 8192, "rank64", seed=1238,
                 note="single large square matrix, rank-64 spectrum plus noise"),
        Workload("experts_128x1536x2048", 128, 1536, 2048, "expert", seed=1239,
                 note="MoE expert stack (all 128 experts)"),
        Workload("experts_16x1536x2048", 16, 1536, 2048, "expert", seed=1240,
                 note="MoE expert stack, local 16-expert shard"),
        Workload("stack_32x7168x2048", 32, 7168, 2048, "iid", seed=1241,
                 note="tall stack, transposed internally to 2048x7168"),
        Workload("stack_128x2048x768", 128, 2048, 768, "iid", seed=1242,
                 note="tall stack, transposed internally to 768x2048"),
    ]
}


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns the
    raw 16-bit patterns as uint16.  Inputs here are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 patterns exactly to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 patterns exactly to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def matrix_f32(w: Workload, k: int, rows: int | None = None, cols: int | None = None) -> np.ndarray:
    """Matrix k of workload w as float32 (before the bf16 cast)."""
    R = w.rows if rows is None else rows
    C = w.cols if cols is None else cols
    rng = np.random.default_rng((w.seed, k))
    if w.dist == "iid":
        return rng.standard_normal((R, C), dtype=np.float32) * np.float32(w.sigma)
    if w.dist == "expert":
        g = rng.standard_normal((R, C), dtype=np.float32) * np.float32(w.sigma)
        scale = np.exp(rng.uniform(np.log(w.scale_lo), np.log(w.scale_hi)))
        return g * np.float32(scale)
    if w.dist == "rank64":
        r = w.rank
        U = rng.standard_normal((R, r), dtype=np.float32) / np.float32(np.sqrt(R))
        V = rng.standard_normal((C, r), dtype=np.float32) / np.float32(np.sqrt(C))
        s = np.exp(rng.uniform(np.log(1e-3), np.log(1.0), size=r)).astype(np.float32)
        low = (U * s[None, :]) @ V.T
        return (low + rng.standard_normal((R, C), dtype=np.float32) * np.float32(w.noise)).astype(np.float32)
    raise ValueError(f"unknown distribution {w.dist!r}")


def matrix_bits(w: Workload, k: int, rows: int | None = None, cols: int | None = None) -> np.ndarray:
    """Matrix k of workload w as raw bf16 bits, shape (rows, cols)."""
    return fp32_to_bf16_bits(matrix_f32(w, k, rows, cols))


def stack_bits(w: Workload, batch: int | None = None) -> np.ndarray:
    """The whole stack as raw bf16 bits, shape (batch, rows, cols)."""
    B = w.batch if batch is None else batch
    out = np.empty((B, w.rows, w.cols), dtype=np.uint16)
    for k in range(B):
        out[k] = matrix_bits(w, k)
    return out
