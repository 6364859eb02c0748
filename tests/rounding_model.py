"""CPU model of where the CUDA path rounds, used to size test tolerances.

This is not the oracle: the oracle (oracle/ns_fp64.py) runs NS in fp64 with no
rounding at all.  This model runs the same steps with the rounding placement
that the library documents for its whole-call bf16 path, so that the error a
correct kernel must show against the oracle can be predicted on the CPU:

  * G arrives in bf16; its norm is an fp32 value, s = fp32(1 / (nu + eps));
  * every tensor-core product is taken as exact (fp32 accumulation of bf16
    products, modelled in fp64: the accumulation error is far below one bf16
    ulp of the stored results);
  * step 1 reads G itself: A = bf16(s^2 (G G^T)) and
    X1 = bf16(s (O G) + (a + D_i) s G);
  * every step stores A in bf16, splits B = b A + c A A (an fp32 epilogue)
    into D = diag(B) in fp32 and O = B - diag(B) in bf16, and stores
    X' = bf16(O X + (a + D_i) X);
  * `scaled_copy=True` models the per-step chain instead, which first stores
    X0 = bf16(s G) and then runs every step on bf16 iterates;
  * `storage="tf32"` models the fp32 mode: G arrives in fp32, the iterates A,
    O and X are stored rounded to tf32 (10-bit mantissa, nearest, ties to
    even), the tensor cores read step 1's raw G truncated to tf32, and the
    last iterate is stored in full fp32.

Tall inputs (rows > cols) run in their transposed, wide orientation: rounding
is elementwise, so the orientation changes nothing in the model.
"""
from __future__ import annotations

import numpy as np

import ns_inputs

COEFFS = (3.4445, -4.7750, 2.0315)


def bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as fp64."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    return ns_inputs.bf16_bits_to_f64(ns_inputs.fp32_to_bf16_bits(x32))


def f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _tf32_bits(x: np.ndarray, nearest: bool) -> np.ndarray:
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    if nearest:
        u = u + 0xFFF + ((u >> 13) & 1)
    return (u & 0xFFFFE000).astype(np.uint32).view(np.float32).astype(np.float64)


def tf32(x: np.ndarray) -> np.ndarray:
    """Round to the nearest tf32 (ties to even), kept as fp64."""
    return _tf32_bits(x, True)


def tf32_trunc(x: np.ndarray) -> np.ndarray:
    """What a tf32 tensor-core read keeps of an fp32 value: the top 10 mantissa bits."""
    return _tf32_bits(x, False)


def model_ns(g: np.ndarray, steps: int = 5, coeffs=COEFFS, eps: float = 1e-7,
             scaled_copy: bool = False, storage: str = "bf16") -> np.ndarray:
    """Rounding model of one matrix's NS (g: the input's values as fp64, rows x cols)."""
    if storage not in ("bf16", "tf32"):
        raise ValueError(storage)
    rnd = bf16 if storage == "bf16" else tf32
    a, b, c = (float(v) for v in coeffs)
    g = np.asarray(g, dtype=np.float64)
    tall = g.shape[0] > g.shape[1]
    x = g.T if tall else g
    nu = f32(np.sqrt(np.sum(x * x)))
    s = f32(1.0 / (nu + f32(eps)))
    if scaled_copy:
        x = rnd(s * x)
        s = 1.0
    for k in range(steps):
        first = k == 0 and not scaled_copy
        last = k + 1 == steps
        xm = tf32_trunc(x) if (first and storage == "tf32") else x  # what the tensor cores read
        acc = xm @ xm.T
        A = rnd(f32(s * s) * acc) if first else rnd(acc)
        Bf = f32(c * (A @ A) + b * A)
        D = np.diag(Bf).copy()
        O = rnd(Bf - np.diag(D))
        out_rnd = f32 if (last and storage == "tf32") else rnd
        if first:
            x = out_rnd(s * (O @ xm) + f32((a + D) * s)[:, None] * x)
        else:
            x = out_rnd(O @ xm + f32(a + D)[:, None] * x)
    return x.T if tall else x
