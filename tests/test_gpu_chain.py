"""Dependent products back to back on one stream, with no host synchronisation.

The tensor-core kernels are launched with programmatic stream serialization:
a launch may begin while the previous kernel on the stream is still running,
and it waits for that kernel to finish before its first global memory
access.  These tests chain products through memory -- each result read as
the next product's A (read after write), a C read through beta and then
overwritten by the next product (write after read), torch kernels in
between -- over every plan kind, and compare every result with the oracle
bit for bit.  Permutation matrices keep the chained values small integers,
exact in FP16, so every step is exact.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

ONE16 = 0x3C00   # 1.0 in FP16

PLANS = [
    {},
    {"cta_pair": 2, "tile_n": 256},
    {"cta_pair": 1, "tile_n": 64, "split_k": 2},
    {"cta_pair": 2, "tile_n": 128},
    {"cta_pair": 1, "tile_n": 128, "stream_k": 2},
    {"cta_pair": 1, "tile_n": 256, "store_mode": 1},
    {"generic": 1},
    {"cta_pair": 2, "tile_n": 256, "stream_k": 2},
]


def _perm_bits(n, seed):
    P = np.zeros((n, n), dtype=np.uint16)
    P[np.arange(n), np.random.default_rng(seed).permutation(n)] = ONE16
    return P


def _f16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).cuda()


def test_chain_read_after_write():
    # X_{i+1} = X_i x P_i with a 16-bit C that the next product reads as A
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, K = 600, 320
    steps = 3 * len(PLANS)
    X0 = inputs.make("small_int", "f16", M, K, 21, 0)
    Ps = [_perm_bits(K, 100 + i) for i in range(steps)]
    Pd = [_f16(P) for P in Ps]
    bufs = [_f16(X0)] + [torch.empty((M, K), dtype=torch.float16, device="cuda") for _ in range(steps)]
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for i in range(steps):
        g.gemm_ex(bufs[i].data_ptr(), Pd[i].data_ptr(), bufs[i + 1].data_ptr(), M, K, K, K, K, K,
                  dtype=0, stream=s, c_dtype=1, **PLANS[i % len(PLANS)])
    g.gemm_device_error(s)
    X = X0
    for i in range(steps):
        X = oracle.encode16("f16", oracle.gemm("f16", X, Ps[i]))
        got = bufs[i + 1].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, X), f"step {i}, plan {PLANS[i % len(PLANS)]}"


def test_chain_through_torch_kernels():
    # FP32 results converted to FP16 by a torch kernel, then multiplied again;
    # an in-place torch update of an input between two products
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, K = 520, 256
    steps = 2 * len(PLANS)
    X0 = inputs.make("small_int", "f16", M, K, 22, 0)
    Ps = [_perm_bits(K, 200 + i) for i in range(steps)]
    Pd = [_f16(P) for P in Ps]
    x = _f16(X0)
    outs = []
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for i in range(steps):
        c = torch.empty((M, K), dtype=torch.float32, device="cuda")
        g.gemm_ex(x.data_ptr(), Pd[i].data_ptr(), c.data_ptr(), M, K, K, K, K, K, dtype=0, stream=s,
                  **PLANS[i % len(PLANS)])
        outs.append(c)
        x = c.to(torch.float16)
        x.add_(1.0)                      # torch writes the next product's A in place
    g.gemm_device_error(s)
    X = X0
    for i in range(steps):
        R = oracle.gemm("f16", X, Ps[i])
        assert np.array_equal(outs[i].cpu().numpy(), R.astype(np.float32)), f"step {i}"
        X = oracle.encode16("f16", R + 1.0)


def test_chain_write_after_read():
    # D_i = W x B + C0 reads W (and D's old values through beta); the next
    # product overwrites W with E_i x P_i as a 16-bit C
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 700, 512, 256
    rounds = len(PLANS)
    W0 = inputs.make("small_int", "f16", M, K, 23, 0)
    B = inputs.make("small_int", "f16", K, N, 23, 1)
    Es = [inputs.make("small_int", "f16", M, K, 300 + i, 0) for i in range(rounds)]
    Ps = [_perm_bits(K, 400 + i) for i in range(rounds)]
    Bd = _f16(B)
    Ed, Pd = [_f16(E) for E in Es], [_f16(P) for P in Ps]
    W = _f16(W0)
    C0 = ((np.arange(M * N).reshape(M, N) % 5) - 2).astype(np.float32)
    Cbase = torch.from_numpy(C0).cuda()
    Ds = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(rounds)]
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for i in range(rounds):
        Ds[i].copy_(Cbase)   # a torch kernel writes the C the product adds onto
        g.gemm_ex(W.data_ptr(), Bd.data_ptr(), Ds[i].data_ptr(), M, N, K, K, N, N, dtype=0,
                  stream=s, alpha=1.0, beta=1.0, **PLANS[i % len(PLANS)])
        g.gemm_ex(Ed[i].data_ptr(), Pd[i].data_ptr(), W.data_ptr(), M, K, K, K, K, K, dtype=0,
                  stream=s, c_dtype=1, **PLANS[(i + 3) % len(PLANS)])
    g.gemm_device_error(s)
    Wi = W0
    for i in range(rounds):
        want = oracle.gemm("f16", Wi, B) + C0.astype(np.float64)
        assert np.array_equal(Ds[i].cpu().numpy(), want.astype(np.float32)), f"round {i}"
        Wi = oracle.encode16("f16", oracle.gemm("f16", Es[i], Ps[i]))
    assert np.array_equal(W.view(torch.int16).cpu().numpy().view(np.uint16), Wi)



SG_PLANS = [{}, {"tile_n": 64, "stream_k": 2}, {"tile_n": 128, "stream_k": 2},
            {"tile_n": 32, "stream_k": 2}, {"tile_n": 64, "split_k": 3}, {"generic": 1},
            {"tile_n": 256}, {"tile_n": 256, "stream_k": 2}]


def test_sgemm_chain_read_after_write_and_write_after_read():
    # FP32: X_{i+1} = X_i x P_i (read after write), with the stream-K SGEMM
    # (programmatic dependent launch) among the plans.  A torch kernel copies
    # each result out (read after write), and another then zeroes the input
    # the product has just read (write after read).
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, K = 1000, 512
    steps = 3 * len(SG_PLANS)
    X0 = inputs.make("small_int", "f32", M, K, 31, 0)
    Ps = []
    for i in range(steps):
        P = np.zeros((K, K), dtype=np.float32)
        P[np.arange(K), np.random.default_rng(500 + i).permutation(K)] = 1.0
        Ps.append(P)
    Pd = [torch.from_numpy(P).cuda() for P in Ps]
    bufs = [torch.from_numpy(X0).cuda()] + [torch.empty((M, K), device="cuda") for _ in range(steps)]
    snaps = []
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for i in range(steps):
        g.gemm_ex(bufs[i].data_ptr(), Pd[i].data_ptr(), bufs[i + 1].data_ptr(), M, K, K, K, K, K,
                  dtype=2, stream=s, **SG_PLANS[i % len(SG_PLANS)])
        snaps.append(bufs[i + 1].clone())
        bufs[i].zero_()
    g.gemm_device_error(s)
    X = X0
    for i in range(steps):
        X = oracle.gemm("f32", X, Ps[i]).astype(np.float32)
        assert np.array_equal(snaps[i].cpu().numpy(), X), f"step {i}, plan {SG_PLANS[i % len(SG_PLANS)]}"
