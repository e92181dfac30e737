"""Writes the golden fixtures in this folder.  Calls only the oracle and the
seeded input generator; run from the repository root:

    python tests/golden/make_golden.py

Fixtures (one value per line after a '#' header; row-major C):
  small_int_12x10x9.txt   C = A x B for the small-integer pattern of
                          "matmul_registers.cu" (fillInputs), FP16 inputs.
                          Every value is an exact integer.
  mod_pattern_16.txt      C = A x B, M = N = K = 16, for the fractional input
                          pattern of the "04-wmma-matmul" code example (its
                          main(): (7i+1) mod 13 / 13 - 1/2 and (5i+3) mod 11 /
                          11 - 1/2 over the flat index), rounded to FP16, with
                          the oracle's double sums printed to 17 digits.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dense_gemm_tensor_tcgen05_gb300 import inputs  # noqa: E402

FIXTURES = {
    "small_int_12x10x9.txt": ("small_int", 12, 10, 9),
    "mod_pattern_16.txt": ("mod_pattern", 16, 16, 16),
}


def compute(dist, M, N, K):
    A = inputs.make(dist, "f16", M, K, 0, 0)
    B = inputs.make(dist, "f16", K, N, 0, 1)
    return oracle.gemm("f16", A, B, M, N, K, K, N, nthreads=1)


def main():
    for name, (dist, M, N, K) in FIXTURES.items():
        C = compute(dist, M, N, K)
        with open(os.path.join(HERE, name), "w") as f:
            f.write(f"# {dist} FP16 inputs, M={M} N={N} K={K}; C row-major, oracle double sums\n")
            for v in C.ravel():
                f.write(f"{float(v)!r}\n")


if __name__ == "__main__":
    main()
