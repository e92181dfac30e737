"""GPU parity for C = alpha * (A x B) + beta * C against the oracle's
general form, on every store path of the library."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PLANS = {
    "tc_tma_store": ("bf16", dict(cta_pair=1, tile_n=256)),
    "tc_plain_store": ("f16", dict(cta_pair=1, tile_n=128, store_mode=1)),
    "tc_swap": ("f16", dict(tile_n=32, swap_ab=1)),
    "tc_split_k": ("bf16", dict(cta_pair=1, tile_n=128, split_k=3)),
    "tc_swap_split_k": ("f16", dict(tile_n=16, swap_ab=1, split_k=4)),
    "tc_stream_k": ("bf16", dict(cta_pair=1, tile_n=64, stream_k=2)),
    "tc_pair": ("bf16", dict(cta_pair=2)),
    "tc_pair_stream_k": ("f16", dict(cta_pair=2, stream_k=2)),
    "sgemm_128x64": ("f32", dict(tile_n=64)),
    "sgemm_128x128": ("f32", dict(tile_n=128)),
    "sgemm_8x16": ("f32", dict(tile_n=256)),
    "sgemm_split": ("f32", dict(tile_n=64, split_k=3)),
    "generic_f16": ("f16", dict(generic=1)),
    "generic_f32": ("f32", dict(generic=1)),
}


def _check(dt, M, N, K, alpha, beta, opts, dist="uniform", ldc_pad=0, exact=False, seed=0):
    A, B = gu.make_inputs(dt, dist, M, N, K, seed)
    ldc = N + ldc_pad
    if dist == "small_int":
        Cin = ((np.arange(M * ldc).reshape(M, ldc) % 7) - 3).astype(np.float32)
    else:
        Cin = inputs.uniform_f32(seed + 7, 3, (M, ldc))
    if beta == 0.0:
        Cin[:] = np.nan     # beta == 0: C must not be read
    C = gu.run_gpu(dt, A, B, M, N, K, ldc=ldc, c_init=Cin, alpha=alpha, beta=beta, **opts)
    R = oracle.gemm_general(dt, A, B, Cin, np.float32(alpha), np.float32(beta), ldc_in=ldc)
    bound = oracle.general_bounds(K, inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt),
                                  alpha, beta, 0.0 if beta == 0 else float(np.abs(Cin[:, :N]).max()))
    err = np.abs(C.astype(np.float64) - R)
    assert np.all(np.isfinite(C)), "non-finite output"
    assert err.max() <= bound, f"max err {err.max():.3e} > {bound:.3e}"
    # the relative Frobenius half of the acceptance rule
    rel = np.linalg.norm(C.astype(np.float64) - R) / np.linalg.norm(R)
    assert rel <= oracle.REL_FROB, f"relative Frobenius error {rel:.3e}"
    if exact:
        assert np.array_equal(C, R.astype(np.float32))


@pytest.mark.parametrize("name", sorted(PLANS))
@pytest.mark.parametrize("alpha,beta", [(1.5, -0.75), (0.5, 0.0), (1.0, 1.0)],
                         ids=["ab", "alpha_only_nan_c", "accumulate"])
def test_general_epilogue_random(name, alpha, beta):
    dt, opts = PLANS[name]
    _check(dt, 300, 520, 700, alpha, beta, opts, ldc_pad=4)


@pytest.mark.parametrize("name", sorted(PLANS))
def test_general_epilogue_exact_integers(name):
    dt, opts = PLANS[name]
    _check(dt, 257, 264, 130, 2.0, -3.0, opts, dist="small_int", exact=True)


@pytest.mark.parametrize("name", ["tc_tma_store", "tc_pair", "sgemm_128x64"])
def test_general_epilogue_ragged_multi_tile(name):
    dt, opts = PLANS[name]
    _check(dt, 4000, 2248, 512, -1.25, 0.5, opts)


def test_k_zero_gives_beta_c():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    for dt in ("f16", "bf16", "f32"):
        C = torch.full((6, 9), 4.0, device="cuda")
        g.gemm_ex(0, 0, C.data_ptr(), 6, 9, 0, 0, 9, 9, dtype=gu.CODE[dt],
                  stream=torch.cuda.current_stream().cuda_stream, alpha=2.0, beta=-0.5)
        torch.cuda.synchronize()
        assert torch.all(C == -2.0).item(), dt


def test_host_pipeline_with_beta():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 2600, 2100, 300
    A, B = gu.make_inputs("bf16", "small_int", M, N, K, 0)
    Cin = ((np.arange(M * N).reshape(M, N) % 5) - 2).astype(np.float32)
    At = torch.from_numpy(A.view(np.int16)).pin_memory()
    Bt = torch.from_numpy(B.view(np.int16)).pin_memory()
    Ct = torch.from_numpy(Cin.copy()).pin_memory()
    s = torch.cuda.current_stream()
    g.gemm_ex_host(At.data_ptr(), Bt.data_ptr(), Ct.data_ptr(), M, N, K, K, N, N, dtype=1,
                   stream=s.cuda_stream, alpha=3.0, beta=2.0)
    s.synchronize()
    R = oracle.gemm_general("bf16", A, B, Cin, 3.0, 2.0)
    assert np.array_equal(Ct.numpy(), R.astype(np.float32))


def test_noalloc_with_beta():
    import ctypes
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 8, 4096, 8192
    A, B = gu.make_inputs("f16", "small_int", M, N, K, 0)
    Cin = ((np.arange(M * N).reshape(M, N) % 3) - 1).astype(np.float32)
    Ad, Bd = gu.to_device(A, "f16"), gu.to_device(B, "f16")
    C = torch.from_numpy(Cin.copy()).cuda()
    o = g._options(0, tile_n=16, swap_ab=1, split_k=4, alpha=-1.0, beta=4.0)
    st = g.lib().gemm_ex_noalloc(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                                 ctypes.byref(o), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    R = oracle.gemm_general("f16", A, B, Cin, -1.0, 4.0)
    assert np.array_equal(C.cpu().numpy(), R.astype(np.float32))


@pytest.mark.parametrize("alpha,beta", [(1.5, -0.75), (0.5, 0.0)], ids=["ab", "alpha_only_nan_c"])
def test_general_epilogue_pair_stream_k_cut_tiles(alpha, beta):
    # the scale and the old C are applied once, by the piece that sums a cut tile
    _check("bf16", 2560, 2600, 1024, alpha, beta, dict(cta_pair=2, stream_k=2), ldc_pad=4)
    _check("f16", 2560, 2600, 1024, alpha, beta, dict(cta_pair=2, stream_k=2), dist="small_int",
           exact=True, seed=2)
