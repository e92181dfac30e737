"""gemm_ex_host with transposed storage, every input type and 16-bit C.

The host entry copies A row panels and B column panels into device staging
buffers.  With trans_a an A panel is a column block of the stored K x M
matrix; with trans_b a B panel is a row block of the stored N x K matrix.
The staging copies round their row strides up to 16 elements, so host
leading dimensions that the device kernels could not take directly (odd, or
not a multiple of 16 for the 8-bit types) still run on the TMA kernels.
Shapes span several row and column panels with ragged last panels; inputs
are small integers, so every result is exact and is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

C_NAMES = {0: "f32", 1: "f16", 2: "bf16"}


def _pinned(bits, dt):
    import torch
    flat = np.ascontiguousarray(bits)
    if dt in ("f32", "tf32"):
        t = torch.from_numpy(flat.astype(np.float32, copy=False))
    elif dt in ("e4m3", "e5m2"):
        t = torch.from_numpy(flat.view(np.uint8))
    else:
        t = torch.from_numpy(flat.view(np.int16))
    return t.pin_memory()


def _host_case(dt, M, N, K, ta, tb, pad, c_dtype=0, alpha=None, beta=None, seed=0):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    A = inputs.make("small_int", dt, M, K, seed, 0)
    B = inputs.make("small_int", dt, K, N, seed, 1)
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    lda, ldb = As.shape[1] + pad, Bs.shape[1] + pad
    As, Bs = inputs.padded(As, lda), inputs.padded(Bs, ldb)
    ldc = N + pad
    cin = ((np.arange(M * ldc).reshape(M, ldc) % 7) - 3).astype(np.float64)
    if c_dtype == 0:
        Ct = torch.from_numpy(cin.astype(np.float32)).pin_memory()
    else:
        Ct = torch.from_numpy(oracle.encode16(C_NAMES[c_dtype], cin).view(np.int16)).pin_memory()
    At, Bt = _pinned(As, dt), _pinned(Bs, dt)
    opts = dict(trans_a=ta, trans_b=tb, c_dtype=c_dtype)
    if alpha is not None:
        opts.update(alpha=alpha, beta=beta)
    st = torch.cuda.current_stream()
    for _ in range(2):   # the second call reuses the staging buffers
        Ct_run = Ct.clone().pin_memory()
        g.gemm_ex_host(At.data_ptr(), Bt.data_ptr(), Ct_run.data_ptr(), M, N, K, lda, ldb, ldc,
                       dtype=gu.CODE[dt], stream=st.cuda_stream, **opts)
        st.synchronize()
        out = Ct_run.numpy()
        R = oracle.gemm_op(dt, ta, tb, As, Bs, M, N, K, lda=lda, ldb=ldb)
        if alpha is not None:
            R = alpha * R if beta == 0.0 else alpha * R + beta * cin[:, :N]
        if c_dtype == 0:
            assert np.array_equal(out[:, :N], R.astype(np.float32))
            assert np.array_equal(out[:, N:], cin[:, N:].astype(np.float32)), "padding columns changed"
        else:
            bits = out.view(np.uint16)
            zero = lambda b: np.where((b & 0x7FFF) == 0, 0, b)
            assert np.array_equal(zero(bits[:, :N]), zero(oracle.encode16(C_NAMES[c_dtype], R)))
            assert np.array_equal(bits[:, N:], oracle.encode16(C_NAMES[c_dtype], cin)[:, N:]), \
                "padding columns changed"


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("trans", [(1, 0), (0, 1), (1, 1)], ids=["tA", "tB", "tAtB"])
@pytest.mark.parametrize("shape", [(2600, 2100, 300), (700, 3000, 77)],
                         ids=lambda s: "x".join(map(str, s)))
def test_host_transposed(dt, trans, shape):
    M, N, K = shape
    _host_case(dt, M, N, K, *trans, pad=3)


@pytest.mark.parametrize("dt", ["tf32", "e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(2600, 2100, 300), (300, 1300, 129)],
                         ids=lambda s: "x".join(map(str, s)))
def test_host_lowprec(dt, shape):
    # B stored N x K (the only layout these types take); K and the host
    # leading dimensions are not multiples of 16
    M, N, K = shape
    _host_case(dt, M, N, K, 0, 1, pad=5)


@pytest.mark.parametrize("case", [("bf16", 1, 1, 2, 1.5, -0.75), ("f16", 1, 0, 1, -2.0, 1.0),
                                  ("e4m3", 0, 1, 2, 0.5, 0.0), ("f32", 0, 1, 1, 1.5, 1.0)],
                         ids=lambda c: "-".join(map(str, c)))
def test_host_epilogue_c16(case):
    dt, ta, tb, c_dtype, alpha, beta = case
    _host_case(dt, 1500, 1100, 200, ta, tb, pad=8, c_dtype=c_dtype, alpha=alpha, beta=beta, seed=3)


def test_matmul_host_views():
    # CPU tensors: column-major views (.t()) go to gemm_ex_host as transposed storage
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 1300, 1100, 96
    A = inputs.make("small_int", "f16", M, K, 5, 0)
    B = inputs.make("small_int", "f16", K, N, 5, 1)
    At = torch.from_numpy(np.ascontiguousarray(A.T).view(np.int16)).view(torch.float16)
    Bt = torch.from_numpy(np.ascontiguousarray(B.T).view(np.int16)).view(torch.float16)
    C = g.matmul(At.t(), Bt.t())
    assert np.array_equal(C.numpy(), oracle.gemm("f16", A, B).astype(np.float32))
    # FP8 from the host: B as the .t() view of a row-major N x K matrix
    A8 = inputs.make("small_int", "e4m3", M, K, 6, 0)
    B8 = inputs.make("small_int", "e4m3", K, N, 6, 1)
    a8 = torch.from_numpy(A8.view(np.uint8)).view(torch.float8_e4m3fn)
    b8 = torch.from_numpy(np.ascontiguousarray(B8.T).view(np.uint8)).view(torch.float8_e4m3fn)
    C8 = g.matmul(a8, b8.t(), out_dtype=torch.bfloat16)
    R8 = oracle.gemm_op("e4m3", 0, 1, A8, np.ascontiguousarray(B8.T), M, N, K)
    assert np.array_equal(C8.view(torch.int16).numpy().view(np.uint16), oracle.encode16("bf16", R8))


@pytest.mark.parametrize("case", [("f16", 0, 0, None, None), ("bf16", 1, 1, 1.5, -0.75),
                                  ("e4m3", 0, 1, 2.0, 0.5), ("f32", 1, 0, 0.5, 0.0)],
                         ids=lambda c: "-".join(map(str, c)))
def test_host_empty_k(case):
    # K = 0: nothing is copied in but C's old values (beta != 0); C = beta * C or 0
    dt, ta, tb, alpha, beta = case
    _host_case(dt, 1300, 1100, 0, ta, tb, pad=4, alpha=alpha, beta=beta, seed=7)
