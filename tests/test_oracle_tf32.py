"""Pins for oracle.tf32_cut, the two readings of how FP32 operands become TF32
(10 fraction bits): dropping the 13 low fraction bits, or rounding them to
nearest with ties to even.  CPU only."""
import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs


def cut(v, mode):
    return float(oracle.tf32_cut(np.array([v], dtype=np.float32), mode)[0])


@pytest.mark.parametrize("v,trunc,rne", [
    (1.0, 1.0, 1.0),
    (1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10),            # kept exactly
    (1.0 + 2.0 ** -11, 1.0, 1.0),                                       # tie, even is 1
    (1.0 + 2.0 ** -10 + 2.0 ** -11, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -9),  # tie, rounds to even
    (1.0 + 2.0 ** -11 + 2.0 ** -23, 1.0, 1.0 + 2.0 ** -10),            # just above the tie
    (2.0 - 2.0 ** -11, 2.0 - 2.0 ** -10, 2.0),                          # carry into the exponent
    (-(1.0 + 2.0 ** -10 + 2.0 ** -11), -(1.0 + 2.0 ** -10), -(1.0 + 2.0 ** -9)),   # sign kept
    (3.0 * 2.0 ** -130, 3.0 * 2.0 ** -130, 3.0 * 2.0 ** -130),         # subnormal, high bits only
    (0.0, 0.0, 0.0),
])
def test_textbook_values(v, trunc, rne):
    assert cut(v, "trunc") == trunc
    assert cut(v, "rne") == rne


@pytest.mark.parametrize("mode,rel", [("trunc", 2.0 ** -10), ("rne", 2.0 ** -11)])
def test_ten_fraction_bits_and_error_bound(mode, rel):
    x = np.concatenate([inputs.uniform_f32(3, 0, (4096,)),
                        inputs.uniform_f32(3, 1, (4096,)) * np.float32(1e6),
                        inputs.uniform_f32(3, 2, (4096,)) * np.float32(1e-6)])
    y = oracle.tf32_cut(x, mode)
    assert np.all((y.view(np.uint32) & 0x1FFF) == 0)              # 10 fraction bits left
    assert np.array_equal(np.signbit(y), np.signbit(x))            # sign kept
    err = np.abs(y.astype(np.float64) - x.astype(np.float64))
    assert np.all(err <= rel * np.abs(x.astype(np.float64)))      # relative error bound
    assert np.array_equal(oracle.tf32_cut(y, mode), y)            # idempotent
    if mode == "trunc":
        assert np.all(np.abs(y) <= np.abs(x))                     # toward zero


def test_round_is_nearest_of_the_two_neighbours():
    x = inputs.uniform_f32(8, 0, (20000,)).astype(np.float32)
    down = oracle.tf32_cut(x, "trunc").astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(x).astype(np.float64))[1] - 11)   # TF32 spacing at |x|
    up = down + np.sign(x) * ulp
    r = oracle.tf32_cut(x, "rne").astype(np.float64)
    xd = x.astype(np.float64)
    best = np.minimum(np.abs(down - xd), np.abs(up - xd))
    assert np.all(np.abs(r - xd) == best)
