"""The oracle against its pins (CPU only)."""
from __future__ import annotations

import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import _pins


def _gemm(dt, A, B, M, N, K, lda, ldb):
    return oracle.gemm(dt, A, B, M, N, K, lda, ldb, nthreads=3)


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    fails = check(_gemm)
    assert not fails, "\n".join(fails[:10])


# ---- decoders: textbook bit patterns, then every pattern against numpy ----

F16_CASES = {
    0x0000: 0.0, 0x3C00: 1.0, 0xC000: -2.0, 0x3800: 0.5, 0x7BFF: 65504.0,
    0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
    0x3555: 0.333251953125, 0x4248: 3.140625, 0xFBFF: -65504.0,
}
BF16_CASES = {
    0x0000: 0.0, 0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625,
    0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,
    0xC2F7: -123.5, 0x3EAB: 0.333984375,
}


def test_f16_decoder_textbook_values():
    L = oracle.lib()
    for bits, want in F16_CASES.items():
        assert L.oracle_f16_to_f64(bits) == want, hex(bits)
    assert math.isinf(L.oracle_f16_to_f64(0x7C00)) and L.oracle_f16_to_f64(0x7C00) > 0
    assert math.isnan(L.oracle_f16_to_f64(0x7E00))
    assert math.copysign(1.0, L.oracle_f16_to_f64(0x8000)) == -1.0


def test_bf16_decoder_textbook_values():
    L = oracle.lib()
    for bits, want in BF16_CASES.items():
        assert L.oracle_bf16_to_f64(bits) == want, hex(bits)
    assert math.isinf(L.oracle_bf16_to_f64(0xFF80)) and L.oracle_bf16_to_f64(0xFF80) < 0
    assert math.isnan(L.oracle_bf16_to_f64(0x7FC0))


def test_decoders_exhaustive_against_numpy():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("f16", allbits)
    want = allbits.view(np.float16).astype(np.float64)
    assert np.array_equal(got, want, equal_nan=True)
    got = oracle.decode("bf16", allbits)
    want = (allbits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    assert np.array_equal(got, want, equal_nan=True)


def test_f32_decoder_against_numpy():
    rng = np.random.default_rng(5)
    w = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 1, 0x7FFFFF, 0x800000, 0x3F800000, 0x7F7FFFFF,
                        0x80000001, 0x7F800000, 0xFF800000, 0x7FC00000], dtype=np.uint32)
    w = np.concatenate([w, special])
    got = oracle.decode("f32", w)
    want = w.view(np.float32).astype(np.float64)
    assert np.array_equal(got, want, equal_nan=True)


# ---- library cross-check and structural properties ----

@pytest.mark.parametrize("dt,dist", [("f16", "uniform"), ("bf16", "normal"), ("f32", "uniform")])
def test_against_torch_float64(dt, dist):
    torch = pytest.importorskip("torch")
    M, N, K = 37, 70, 129
    A = inputs.make(dist, dt, M, K, 11, 0)
    B = inputs.make(dist, dt, K, N, 11, 1)
    C = oracle.gemm(dt, A, B)
    At = torch.from_numpy(oracle.decode(dt, A))
    Bt = torch.from_numpy(oracle.decode(dt, B))
    ref = (At @ Bt).numpy()
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_thread_count_does_not_change_result():
    A = inputs.make("normal", "bf16", 67, 300, 2, 0)
    B = inputs.make("normal", "bf16", 300, 45, 2, 1)
    C1 = oracle.gemm("bf16", A, B, nthreads=1)
    C7 = oracle.gemm("bf16", A, B, nthreads=7)
    assert np.array_equal(C1, C7)


def test_rows_and_entries_agree_with_full_product():
    A = inputs.make("uniform", "f16", 40, 77, 9, 0)
    B = inputs.make("uniform", "f16", 77, 33, 9, 1)
    C = oracle.gemm("f16", A, B, nthreads=2)
    band = oracle.gemm_rows("f16", A, B, 5, 19, nthreads=3)
    assert np.array_equal(band, C[5:19])
    rows = np.array([0, 39, 17, 5])
    cols = np.array([32, 0, 16, 7])
    ent = oracle.gemm_entries("f16", A, B, rows, cols)
    assert np.array_equal(ent, C[rows, cols])


def test_degenerate_shapes():
    A = np.zeros((4, 0), dtype=np.uint16)
    B = np.zeros((0, 3), dtype=np.uint16)
    C = oracle.gemm("f16", A, B, 4, 3, 0, 0, 3)
    assert C.shape == (4, 3) and np.all(C == 0.0)          # empty sum
    C = oracle.gemm("f16", np.zeros((0, 5), np.uint16), np.zeros((5, 3), np.uint16))
    assert C.shape == (0, 3)


def test_bad_arguments_rejected():
    L = oracle.lib()
    A = np.zeros(4, dtype=np.uint16)
    out = np.zeros(4, dtype=np.float64)
    rc = L.oracle_gemm(0, A.ctypes.data_as(ctypes.c_void_p), A.ctypes.data_as(ctypes.c_void_p),
                       out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                       2, 2, 2, 1, 2, 2, 1)          # lda < K
    assert rc == -1
    with pytest.raises(ValueError):
        oracle.gemm_entries("f16", np.zeros((2, 2), np.uint16), np.zeros((2, 2), np.uint16),
                            [2], [0])


# ---- the checker itself ----

def test_compare_rule():
    R = np.array([[1.0, -2.0], [3.0, 0.5]])
    ok = oracle.compare(R.astype(np.float32), R, K=4, max_abs_a=1.0, max_abs_b=1.0)
    assert ok.ok and ok.exact and ok.max_abs == 0.0
    # abs bound = 1e-3 * 2 * 1 * 1 = 2e-3
    C = R.copy(); C[1, 0] += 3e-3
    bad = oracle.compare(C, R, K=4, max_abs_a=1.0, max_abs_b=1.0)
    assert not bad.ok and bad.first_bad[:2] == (1, 0)
    C = R.copy(); C[0, 0] = np.nan
    assert not oracle.compare(C, R, 4, 1.0, 1.0).ok
    Z = np.zeros((2, 2))
    assert oracle.compare(Z, Z, 0, 0.0, 0.0).ok
    assert not oracle.compare(Z + 1e-30, Z, 0, 0.0, 0.0).ok


# ---- the pins catch planted mistakes in a copy of the oracle ----

MUTATIONS = {
    "dropped_last_term": ("for (int64_t p = 0; p < j->k; ++p) {",
                          "for (int64_t p = 0; p < j->k - 1; ++p) {"),
    "sign_flip": ("crow[c] += av * brow[c];", "crow[c] -= av * brow[c];"),
    "b_rows_reversed": ("b[p * N + c] = decode_one(dtype, B, p * ldb + c);",
                        "b[p * N + c] = decode_one(dtype, B, (K - 1 - p) * ldb + c);"),
    "b_cols_reversed": ("b[p * N + c] = decode_one(dtype, B, p * ldb + c);",
                        "b[p * N + c] = decode_one(dtype, B, p * ldb + (N - 1 - c));"),
    "f16_bias_off_by_one": ("v = ldexp((double)(1024 + f), e - 25);",
                            "v = ldexp((double)(1024 + f), e - 24);"),
    "bf16_subnormal_scale": ("v = ldexp((double)f, -133);", "v = ldexp((double)f, -134);"),
    "a_row_stride": ("a[i * lda + p] = decode_one(dtype, A, (row0 + i) * lda + p);",
                     "a[i * lda + p] = decode_one(dtype, A, (row0 + i) * K + p);"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(path), "-lm", "-lpthread"], check=True)
    L = ctypes.CDLL(str(so))
    L.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.POINTER(ctypes.c_double)] + [ctypes.c_int64] * 6 + [ctypes.c_int]
    L.oracle_gemm.restype = ctypes.c_int
    codes = {"f16": 0, "bf16": 1, "f32": 2}

    def gemm(dt, A, B, M, N, K, lda, ldb):
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
        C = np.zeros((M, N), dtype=np.float64)
        L.oracle_gemm(codes[dt], A.ctypes.data_as(ctypes.c_void_p), B.ctypes.data_as(ctypes.c_void_p),
                      C.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), M, N, K, lda, ldb, N, 1)
        return C
    return gemm


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    gemm = _build_mutant(tmp_path, name, old, new)
    assert _pins.run_all(gemm), f"no pin caught mutation {name}"
