"""The largest shapes: C past 2^32 elements, and a K of two million.

Inputs are the small-integer pattern, so every element of C is an exact
integer (|C| <= 6K < 2^24 even at K = 2^21) and sampled rows are compared with
the oracle bit for bit.

* M = N = 65536: C holds 2^32 elements (16 GiB in FP32), so row offsets into C
  pass 2^31 elements and 2^34 bytes.  C starts as NaN; every sampled row must
  be written in full.  The rows sampled include both ends of every tile edge
  the planners may cut at and the last row.
* K = 2^21 + 37 with a ragged 300 x 264 C: long split-K slices and a K tail.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

C_NAMES = {0: "f32", 1: "f16", 2: "bf16"}


def _rows(M, extra, seed):
    fixed = [0, 1, 127, 128, 255, 256, M // 2 - 1, M // 2, M - 257, M - 256, M - 129, M - 128, M - 2, M - 1]
    rnd = np.random.default_rng(seed).integers(0, M, extra).tolist()
    return sorted(set(r for r in fixed + rnd if 0 <= r < M))


@pytest.mark.parametrize("dt,c_dtype", [("bf16", 0), ("f16", 2), ("f32", 0), ("e4m3", 1)])
def test_c_beyond_2_pow_32_elements(dt, c_dtype):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M = N = 65536
    K = 32
    A = inputs.make("small_int", dt, M, K, 11, 0)
    B = inputs.make("small_int", dt, K, N, 11, 1)
    tb = 1 if dt == "e4m3" else 0
    Bs = np.ascontiguousarray(B.T) if tb else B
    Ad, Bd = gu.to_device(A, dt), gu.to_device(Bs, dt)
    if c_dtype == 0:
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    else:
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")   # 0xFFFF: a NaN either way
    s = torch.cuda.current_stream().cuda_stream
    g.gemm_ex(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, Bs.shape[1], N,
              dtype=gu.CODE[dt], stream=s, trans_b=tb, c_dtype=c_dtype)
    g.gemm_device_error(s)
    rows = _rows(M, 8, 12)
    got = C[torch.tensor(rows, device="cuda")].cpu().numpy()
    R = oracle.gemm_op(dt, 0, tb, A[rows], Bs, len(rows), N, K)
    if c_dtype == 0:
        assert np.array_equal(got, R.astype(np.float32))
    else:
        zero = lambda b: np.where((b & 0x7FFF) == 0, 0, b)
        assert np.array_equal(zero(got.view(np.uint16)), zero(oracle.encode16(C_NAMES[c_dtype], R)))
    del C


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32", "e4m3"])
def test_k_two_million(dt):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 300, 264, (1 << 21) + 37
    A = inputs.make("small_int", dt, M, K, 13, 0)
    B = inputs.make("small_int", dt, K, N, 13, 1)
    tb = 1 if dt == "e4m3" else 0
    Bs = np.ascontiguousarray(B.T) if tb else B
    # K-contiguous rows padded to 16 elements, so every type takes its TMA (or
    # vectorised SGEMM) path
    lda = -(-K // 16) * 16
    ldb = lda if tb else N
    A = inputs.padded(A, lda)
    if tb:
        Bs = inputs.padded(Bs, ldb)
    Ad, Bd = gu.to_device(A, dt), gu.to_device(Bs, dt)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    g.gemm_ex(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, N,
              dtype=gu.CODE[dt], stream=s, trans_b=tb)
    g.gemm_device_error(s)
    # both sides of each tile edge and the last row / column (the oracle on
    # a sample: a full row of C is 264 sums of two million terms)
    rows = [0, 127, 128, 255, 256, M - 1]
    cols = [0, 1, 63, 64, 127, 128, 255, 256, N - 1]
    got = C.cpu().numpy()[np.ix_(rows, cols)]
    Bsub = np.ascontiguousarray(Bs[cols] if tb else Bs[:, cols])
    R = oracle.gemm_op(dt, 0, tb, A[rows], Bsub, len(rows), len(cols), K, lda=lda,
                       ldb=ldb if tb else len(cols))
    assert np.array_equal(got, R.astype(np.float32))
    assert not np.isnan(C.cpu().numpy()).any(), "an element of C was not written"
