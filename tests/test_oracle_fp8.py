"""Pins for the oracle's 8-bit decoders and low-precision products (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import _pins


def test_e4m3_textbook_values():
    L = oracle.lib()
    cases = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x7E: 448.0, 0x01: 2.0 ** -9,
             0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9, 0x3C: 1.5}
    for b, v in cases.items():
        assert L.oracle_e4m3_to_f64(b) == v, hex(b)
    assert math.isnan(L.oracle_e4m3_to_f64(0x7F)) and math.isnan(L.oracle_e4m3_to_f64(0xFF))


def test_e5m2_textbook_values():
    L = oracle.lib()
    cases = {0x00: 0.0, 0x3C: 1.0, 0xBC: -1.0, 0x7B: 57344.0, 0x01: 2.0 ** -16,
             0x04: 2.0 ** -14, 0x3E: 1.5}
    for b, v in cases.items():
        assert L.oracle_e5m2_to_f64(b) == v, hex(b)
    assert math.isinf(L.oracle_e5m2_to_f64(0x7C)) and math.isnan(L.oracle_e5m2_to_f64(0x7D))


@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_fp8_decoders_exhaustive_against_torch(dt):
    torch = pytest.importorskip("torch")
    allbits = np.arange(256, dtype=np.uint8)
    got = oracle.decode(dt, allbits)
    tt = torch.float8_e4m3fn if dt == "e4m3" else torch.float8_e5m2
    want = torch.from_numpy(allbits.copy()).view(tt).double().numpy()
    assert np.array_equal(got, want, equal_nan=True)


@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_fp8_small_int_exact(dt):
    M, N, K = 9, 13, 40
    A = inputs.make("small_int", dt, M, K, 0, 0)
    B = inputs.make("small_int", dt, K, N, 0, 1)
    assert np.array_equal(oracle.gemm(dt, A, B), _pins.small_int_exact(M, N, K))


@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_fp8_transposed_op_and_rounding_of_inputs(dt):
    # inputs rounded to 8 bits keep the generator's value to within half an ulp
    x = inputs.uniform_f32(3, 0, (64, 64))
    bits = inputs.to_bits(x, dt)
    v = oracle.decode(dt, bits)
    frac = 3 if dt == "e4m3" else 2
    sub_ulp = 2.0 ** (-9 if dt == "e4m3" else -16)     # spacing of subnormals
    # half an ulp: relative for normal values, absolute among subnormals
    bound = np.maximum(np.abs(x) * 2.0 ** -(frac + 1), sub_ulp / 2)
    assert np.all(np.abs(v - x) <= bound + 1e-15)


def test_tf32_bound_covers_truncated_inputs():
    # a product of inputs with their low 13 fraction bits dropped stays within the bound
    A = inputs.uniform_f32(4, 0, (16, 256))
    B = inputs.uniform_f32(4, 1, (256, 16))
    trunc = lambda x: (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    exact = oracle.gemm("f32", A, B)
    approx = oracle.gemm("f32", trunc(A), trunc(B))
    S = oracle.gemm("f32", np.abs(A), np.abs(B))
    assert np.all(np.abs(approx - exact) <= oracle.tf32_bound(S))


def test_tf32_bound_covers_nearest_rounded_inputs():
    # the other reading: the low 13 fraction bits rounded to nearest (ties to even)
    A = inputs.uniform_f32(5, 0, (16, 256))
    B = inputs.uniform_f32(5, 1, (256, 16))

    def rne(x):
        u = x.view(np.uint32).astype(np.uint64)
        lsb = (u >> 13) & 1
        return ((u + 0xFFF + lsb) & 0xFFFFE000).astype(np.uint32).view(np.float32)

    exact = oracle.gemm("f32", A, B)
    approx = oracle.gemm("f32", rne(A), rne(B))
    S = oracle.gemm("f32", np.abs(A), np.abs(B))
    assert np.all(np.abs(approx - exact) <= oracle.tf32_bound(S))
    assert not np.array_equal(approx, exact)
