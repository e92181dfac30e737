"""Pins for oracle.general_bounds, the tolerance of C = alpha * (A x B) + beta * C.

The kernels form the product in FP32 (covered by the standard bound
1e-3 sqrt(K) max|A| max|B|, scaled by |alpha|), then compute
fmaf(alpha, acc, beta * c): two more FP32 roundings (beta * c, and the fused
multiply-add), each at most 2^-24 of a value no larger than
|alpha| K max|A| max|B| + |beta| max|C|.  The bound adds 2^-21 of that, eight
such roundings.  These tests replay those FP32 steps exactly (numpy float32
for beta * c; the fused multiply-add as one exact double sum rounded once)
and check that (a) the bound covers them on random and adversarial data and
(b) its rounding term is needed: without it, large beta * C fails."""
import math

import numpy as np

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs


def epilogue_fp32(acc32, alpha, beta, c32):
    """fmaf(alpha, acc, beta * c) in FP32, step by step."""
    a = np.float32(alpha)
    bc = (np.float32(beta) * c32).astype(np.float32)             # one FP32 rounding
    exact = a.astype(np.float64) * acc32.astype(np.float64) + bc.astype(np.float64)
    return exact.astype(np.float32)                                # the FMA's one rounding


def case(M, N, K, alpha, beta, c_scale, seed):
    A = inputs.make("uniform", "f16", M, K, seed, 0)
    B = inputs.make("uniform", "f16", K, N, seed, 1)
    C = inputs.uniform_f32(seed, 2, (M, N)) * np.float32(c_scale)
    R = oracle.gemm("f16", A, B)                                  # exact in double here
    want = oracle.gemm_general("f16", A, B, C, alpha, beta)
    # an FP32 accumulator: the product rounded to FP32 and pushed by up to the
    # standard bound in the direction that hurts most
    amax, bmax = inputs.bits_abs_max(A, "f16"), inputs.bits_abs_max(B, "f16")
    prod_bound = oracle.ABS_COEF * math.sqrt(K) * amax * bmax
    push = np.sign(R) * np.sign(alpha) * np.float32(prod_bound * 0.999)
    acc32 = (R.astype(np.float32) + push.astype(np.float32)).astype(np.float32)
    got = epilogue_fp32(acc32, alpha, beta, C)
    bound = oracle.general_bounds(K, amax, bmax, alpha, beta, float(np.abs(C).max()))
    return np.abs(got.astype(np.float64) - want), bound, abs(alpha) * prod_bound


def test_bound_covers_the_fp32_epilogue_on_random_data():
    for seed, (alpha, beta, cs) in enumerate([(1.5, -0.75, 1.0), (0.5, 0.0, 1.0), (1.0, 1.0, 3.0),
                                              (-2.0, 0.25, 100.0), (1e3, -1e3, 1e2)]):
        err, bound, _ = case(33, 47, 300, alpha, beta, cs, seed)
        assert err.max() <= bound, (alpha, beta, err.max(), bound)


def test_rounding_term_is_needed_for_large_beta_c():
    # beta * C of order 1e9: its FP32 rounding (~2^-24 * 1e9 ~ 60) dwarfs the
    # product's own bound (~1e-2), so a bound without the rounding term fails
    err, bound, product_only = case(16, 16, 64, 1.0, 3.0e4, 3.0e4, 11)
    assert err.max() > product_only
    assert err.max() <= bound

