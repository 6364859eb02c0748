"""Writes the stored expected values under tests/golden/.

Calls only the oracle and the seeded input generator; no value here comes from
the CUDA library.  Re-run with `python tests/golden/make_golden.py` from the
repository root; the files are committed.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import ns_inputs  # noqa: E402
import oracle  # noqa: E402

CASES = [
    # name, batch, rows, cols, seed: tiny i.i.d. N(0, 0.02^2) matrices, bf16 at input
    ("wide_2x6x10", 2, 6, 10, 501),
    ("tall_1x10x6", 1, 10, 6, 502),
    ("square_1x8x8", 1, 8, 8, 503),
]


def write_case(name, batch, rows, cols, seed):
    w = ns_inputs.Workload(name, batch, rows, cols, "iid", seed=seed)
    bits = ns_inputs.stack_bits(w)
    out = oracle.newton_schulz(ns_inputs.bf16_bits_to_f64(bits))
    path = os.path.join(HERE, f"ns_{name}.txt")
    with open(path, "w") as f:
        f.write(f"# fp64 oracle output of 5-step quintic NS, coeffs {oracle.DEFAULT_COEFFS}, eps {oracle.DEFAULT_EPS}\n")
        f.write("# written by tests/golden/make_golden.py (oracle only)\n")
        f.write(f"shape {batch} {rows} {cols}\n")
        f.write("input_bf16_hex " + " ".join(f"{int(v):04x}" for v in bits.ravel()) + "\n")
        f.write("output_f64 " + " ".join(repr(float(v)) for v in out.ravel()) + "\n")


if __name__ == "__main__":
    for case in CASES:
        write_case(*case)
