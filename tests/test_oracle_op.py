"""Pins for the oracle's transposed-operand form op(A) x op(B) (CPU only)."""
import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs


def _int_matrix(rows, cols, a, b, m):
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    return ((a * r + b * c) % m - m // 2).astype(np.float32)


def _exact(opA, opB):
    """Exact integer product by Python integers."""
    M, K = opA.shape
    N = opB.shape[1]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            out[i, j] = sum(int(opA[i, p]) * int(opB[p, j]) for p in range(K))
    return out


@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_small_int_exact_all_transposes(ta, tb, dt):
    M, N, K = 7, 9, 11
    opA = _int_matrix(M, K, 1, 2, 7)
    opB = _int_matrix(K, N, 3, 1, 5)
    As = opA.T.copy() if ta else opA          # storage
    Bs = opB.T.copy() if tb else opB
    C = oracle.gemm_op(dt, ta, tb, inputs.to_bits(As, dt), inputs.to_bits(Bs, dt), M, N, K)
    assert np.array_equal(C, _exact(opA, opB))


def test_transposed_identity():
    I = inputs.make("identity", "f16", 6, 6, 0, 0)
    X = inputs.make("uniform", "f16", 6, 6, 1, 1)
    C = oracle.gemm_op("f16", True, True, I, X, 6, 6, 6)     # I^T X^T = X^T
    assert np.array_equal(C, X.view(np.float16).astype(np.float64).T)


def test_transpose_of_product_identity():
    # (A B)^T = B^T A^T: op(A) = B^T read from B's storage with trans, etc.
    M, N, K = 5, 8, 6
    A = inputs.make("uniform", "bf16", M, K, 2, 0)
    B = inputs.make("uniform", "bf16", K, N, 2, 1)
    AB = oracle.gemm_op("bf16", False, False, A, B, M, N, K)
    BtAt = oracle.gemm_op("bf16", True, True, B, A, N, M, K)
    assert np.array_equal(AB.T, BtAt)


def test_padded_transposed_leading_dimensions():
    M, N, K = 4, 5, 3
    opA = _int_matrix(M, K, 1, 1, 5)
    opB = _int_matrix(K, N, 2, 1, 7)
    As = inputs.padded(inputs.to_bits(opA.T.copy(), "f16"), M + 6)   # K x M, lda = M + 6
    Bs = inputs.padded(inputs.to_bits(opB.T.copy(), "f16"), K + 2)   # N x K, ldb = K + 2
    C = oracle.gemm_op("f16", True, True, As, Bs, M, N, K, lda=M + 6, ldb=K + 2)
    assert np.array_equal(C, _exact(opA, opB))


def test_bad_leading_dimension_rejected():
    with pytest.raises(RuntimeError):
        oracle.gemm_op("f16", True, False, np.zeros((3, 4), np.uint16), np.zeros((3, 2), np.uint16),
                       5, 2, 3, lda=4)       # trans_a needs lda >= M = 5
