"""Golden fixtures built from the pages' deterministic input patterns.

The fixtures are written by tests/golden/make_golden.py, which calls only the
oracle.  Here they are pinned by something other than the oracle: exact
integer arithmetic for the small-integer pattern and exact rational
arithmetic for the fractional pattern."""
import os
from fractions import Fraction

import numpy as np

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import _pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name, M, N):
    vals = [float(l) for l in open(os.path.join(GOLDEN, name)) if not l.startswith("#")]
    return np.array(vals, dtype=np.float64).reshape(M, N)


def test_small_int_fixture_is_exact_integer_product():
    C = load("small_int_12x10x9.txt", 12, 10)
    assert np.array_equal(C, _pins.small_int_exact(12, 10, 9))


def test_mod_pattern_fixture_against_exact_rationals():
    C = load("mod_pattern_16.txt", 16, 16)
    A = inputs.make("mod_pattern", "f16", 16, 16, 0, 0)
    B = inputs.make("mod_pattern", "f16", 16, 16, 0, 1)
    Av = A.view(np.float16).astype(np.float64)
    Bv = B.view(np.float16).astype(np.float64)
    for i in range(16):
        for j in range(16):
            exact = sum((Fraction(float(Av[i, p])) * Fraction(float(Bv[p, j])) for p in range(16)),
                        Fraction(0))
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(16, 2 ** 52) * 16 / 4


def test_fixtures_reproduce_from_oracle():
    for name, (dist, M, N, K) in {"small_int_12x10x9.txt": ("small_int", 12, 10, 9),
                                  "mod_pattern_16.txt": ("mod_pattern", 16, 16, 16)}.items():
        A = inputs.make(dist, "f16", M, K, 0, 0)
        B = inputs.make(dist, "f16", K, N, 0, 1)
        assert np.array_equal(load(name, M, N), oracle.gemm("f16", A, B, nthreads=1))


def test_mod_pattern_first_values():
    # The pattern's first inputs, worked by hand from its formula:
    # a_0 = 1/13 - 1/2, a_1 = 8/13 - 1/2, b_0 = 3/11 - 1/2, b_1 = 8/11 - 1/2.
    A = inputs.make("mod_pattern", "f32", 1, 2, 0, 0)
    B = inputs.make("mod_pattern", "f32", 1, 2, 0, 1)
    assert np.allclose(A[0], [1 / 13 - 0.5, 8 / 13 - 0.5], atol=1e-7)
    assert np.allclose(B[0], [3 / 11 - 0.5, 8 / 11 - 0.5], atol=1e-7)
