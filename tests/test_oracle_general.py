"""Pins for the oracle's general form alpha * AB + beta * C_in (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import _pins


def test_beta_zero_ignores_c_in_even_nan():
    A = inputs.make("small_int", "f16", 5, 7, 0, 0)
    B = inputs.make("small_int", "f16", 7, 4, 0, 1)
    Cin = np.full((5, 4), np.nan, dtype=np.float32)
    out = oracle.gemm_general("f16", A, B, Cin, 1.0, 0.0)
    assert np.array_equal(out, _pins.small_int_exact(5, 4, 7))


def test_alpha_scales_and_beta_adds_exactly_on_integers():
    M, N, K = 6, 9, 11
    A = inputs.make("small_int", "bf16", M, K, 0, 0)
    B = inputs.make("small_int", "bf16", K, N, 0, 1)
    Cin = (np.arange(M * N).reshape(M, N) % 7 - 3).astype(np.float32)
    exact = _pins.small_int_exact(M, N, K)
    out = oracle.gemm_general("bf16", A, B, Cin, -2.0, 3.0)
    assert np.array_equal(out, -2.0 * exact + 3.0 * Cin)


def test_alpha_minus_one_beta_one_cancels_the_product():
    M, N, K = 8, 8, 16
    A = inputs.make("small_int", "f32", M, K, 0, 0)
    B = inputs.make("small_int", "f32", K, N, 0, 1)
    Cin = _pins.small_int_exact(M, N, K).astype(np.float32)
    out = oracle.gemm_general("f32", A, B, Cin, -1.0, 1.0)
    assert np.all(out == 0.0)


def test_identity_operand_closed_form():
    # A = I: alpha * B + beta * C
    M = K = 10
    N = 6
    I = inputs.make("identity", "f16", M, K, 0, 0)
    B = inputs.make("uniform", "f16", K, N, 3, 1)
    Cin = inputs.uniform_f32(4, 2, (M, N))
    out = oracle.gemm_general("f16", I, B, Cin, 0.5, -1.25)
    Bv = B.view(np.float16).astype(np.float64)
    assert np.array_equal(out, 0.5 * Bv + -1.25 * Cin.astype(np.float64))


def test_fraction_bruteforce_with_scalars():
    M, N, K = 3, 4, 5
    A = inputs.make("uniform", "f16", M, K, 9, 0)
    B = inputs.make("uniform", "f16", K, N, 9, 1)
    Cin = inputs.uniform_f32(9, 2, (M, N))
    alpha, beta = np.float32(0.75), np.float32(-0.3)
    out = oracle.gemm_general("f16", A, B, Cin, float(alpha), float(beta))
    Av, Bv = A.view(np.float16).astype(np.float64), B.view(np.float16).astype(np.float64)
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(float(Av[i, k])) * Fraction(float(Bv[k, j])) for k in range(K)), Fraction(0))
            want = Fraction(float(alpha)) * s + Fraction(float(beta)) * Fraction(float(Cin[i, j]))
            assert abs(Fraction(out[i, j]) - want) <= Fraction(1, 2 ** 45) * (abs(want) + 1)


def test_padded_c_in_rows():
    M, N, K = 4, 3, 5
    A = inputs.make("small_int", "f16", M, K, 0, 0)
    B = inputs.make("small_int", "f16", K, N, 0, 1)
    Cin = np.full((M, N + 5), 1e30, dtype=np.float32)
    Cin[:, :N] = 2.0
    out = oracle.gemm_general("f16", A, B, Cin, 1.0, 0.5, ldc_in=N + 5)
    assert np.array_equal(out, _pins.small_int_exact(M, N, K) + 1.0)
