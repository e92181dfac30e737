"""GPU parity for a 16-bit output C (FP16 or BF16) on every kernel path,
against the oracle.

The library forms each result in FP32 and rounds it once, to nearest with
ties to even.  So:
  * small-integer inputs (every FP32 partial sum exact) must give exactly
    the oracle's rounding of the exact result, bit for bit;
  * other inputs must lie within the FP32 bound of the exact result plus
    half a 16-bit ulp of it;
  * padding columns of C and the memory after it keep their sentinels.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CT = {"f16": 1, "bf16": 2}
NAN16 = {"f16": 0x7E00, "bf16": 0x7FC0}

PLANS = {
    "tc_128x256_tma": ("bf16", dict(cta_pair=1, tile_n=256)),
    "tc_128x128_tma": ("f16", dict(cta_pair=1, tile_n=128)),
    "tc_128x64_plain": ("f16", dict(cta_pair=1, tile_n=64, store_mode=1)),
    "tc_swap32": ("bf16", dict(tile_n=32, swap_ab=1)),
    "tc_split_k": ("f16", dict(cta_pair=1, tile_n=128, split_k=3)),
    "tc_stream_k": ("bf16", dict(cta_pair=1, tile_n=128, stream_k=2)),
    "tc_pair256": ("bf16", dict(cta_pair=2, tile_n=256)),
    "tc_pair128": ("f16", dict(cta_pair=2, tile_n=128)),
    "tc_pair_plain": ("bf16", dict(cta_pair=2, tile_n=256, store_mode=1)),
    "sgemm_128x64": ("f32", dict(tile_n=64)),
    "sgemm_128x128": ("f32", dict(tile_n=128)),
    "sgemm_8x16": ("f32", dict(tile_n=256)),
    "sgemm_split": ("f32", dict(tile_n=64, split_k=3)),
    "generic_f16": ("f16", dict(generic=1)),
    "generic_f32": ("f32", dict(generic=1)),
    "tf32": ("tf32", dict(trans_b=1)),
    "e4m3": ("e4m3", dict(trans_b=1)),
}


def run_gpu_c16(dt, A_bits, B_bits, M, N, K, lda, ldb, ldc, c_name, c_init=None, c_offset=0,
                **opts):
    """C bits (M x N uint16) from gemm_ex with a 16-bit C; checks that the
    padding columns and a guard zone after C keep their sentinels."""
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    Ad = gu.to_device(A_bits, dt)
    Bd = gu.to_device(B_bits, dt)
    guard = 4096
    rows = max(M, 1)
    nan = np.uint16(NAN16[c_name]).view(np.int16)
    cbuf = torch.full((c_offset + rows * ldc + guard,), int(nan), dtype=torch.int16, device="cuda")
    Cd = cbuf[c_offset:]
    if c_init is not None:
        Cd[: M * ldc].copy_(torch.from_numpy(np.ascontiguousarray(c_init).view(np.int16).ravel()))
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    g.gemm_ex(Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, lda, ldb, ldc,
              dtype=gu.CODE[dt], stream=s, c_dtype=CT[c_name], **opts)
    g.gemm_device_error(s)
    out = Cd.cpu().numpy().view(np.uint16)
    assert np.all(out[rows * ldc:] == NAN16[c_name]), "kernel wrote past the end of C"
    if c_offset:
        assert np.all(cbuf[:c_offset].cpu().numpy().view(np.uint16) == NAN16[c_name])
    C = out[: rows * ldc].reshape(rows, ldc)[:M]
    if ldc > N and M > 0:
        want_pad = NAN16[c_name] if c_init is None else c_init[:, N:]
        assert np.all(C[:, N:] == want_pad), "kernel wrote into C's padding columns"
    return C[:, :N]


def _operands(dt, dist, M, N, K, seed, trans_b, sigma=1.0):
    A = inputs.make(dist, dt, M, K, seed, 0, sigma)
    B = inputs.make(dist, dt, K, N, seed, 1, sigma)
    Bs = np.ascontiguousarray(B.T) if trans_b else B
    align = {"tf32": 4, "e4m3": 16, "e5m2": 16}.get(dt, 1)
    lda = -(-K // align) * align
    ldb = lda if trans_b else N
    As = inputs.padded(A, lda) if lda != K else A
    if trans_b and ldb != K:
        Bs = inputs.padded(Bs, ldb)
    return A, B, As, Bs, lda, ldb


def _bounds(dt, A, B, K, R):
    if dt == "tf32":
        S = oracle.gemm("f32", np.abs(A), np.abs(B))
        return oracle.tf32_bound(S)
    return oracle.ABS_COEF * math.sqrt(K) * inputs.bits_abs_max(A, dt) * inputs.bits_abs_max(B, dt)


def _check(name, c_name, M, N, K, dist, exact, ldc_pad=0, seed=0, c_offset=0):
    dt, opts = PLANS[name]
    tb = opts.get("trans_b", 0)
    A, B, As, Bs, lda, ldb = _operands(dt, dist, M, N, K, seed, tb)
    ldc = N + ldc_pad
    C = run_gpu_c16(dt, As, Bs, M, N, K, lda, ldb, ldc, c_name, c_offset=c_offset, **opts)
    R = oracle.gemm(dt, A, B)
    what = f"{name} c={c_name} {dist} {M}x{N}x{K} ldc={ldc}"
    if exact:
        want = oracle.encode16(c_name, R)
        bad = np.argwhere(C != want)
        assert bad.size == 0, f"{what}: {len(bad)} differ, first {bad[0].tolist()} " \
                              f"got {C[tuple(bad[0])]:#06x} want {want[tuple(bad[0])]:#06x}"
        return
    got = oracle.decode(c_name, C)
    e32 = _bounds(dt, A, B, K, R)
    bound = e32 + oracle.half_ulp16(c_name, np.abs(R) + e32)
    err = np.abs(got - R)
    assert np.all(err <= bound), f"{what}: max excess {np.max(err - bound):.3e}"


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
@pytest.mark.parametrize("name", sorted(PLANS))
def test_c16_exact_small_integers(name, c_name):
    # results up to 6K: beyond 2048 (FP16) and 256 (BF16) the rounding of
    # exact integers is exercised too
    _check(name, c_name, 300, 520, 700, "small_int", exact=True)


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
@pytest.mark.parametrize("name", sorted(PLANS))
def test_c16_random_ragged(name, c_name):
    # N = 130: not a multiple of 8, so the plain store path; ldc padded
    _check(name, c_name, 257, 130, 200, "uniform", exact=False, ldc_pad=6, seed=3)


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(1024, 1536, 512), (8, 1024, 2048), (2048, 64, 256),
                                   (4000, 2248, 512), (129, 17, 33)],
                         ids=lambda s: "x".join(map(str, s)))
def test_c16_default_plans(shape, c_name):
    M, N, K = shape
    for dt in ("bf16", "f16", "f32"):
        A, B, _, _, _, _ = _operands(dt, "small_int", M, N, K, 0, 0)
        C = run_gpu_c16(dt, A, B, M, N, K, K, N, N, c_name)
        assert np.array_equal(C, oracle.encode16(c_name, oracle.gemm(dt, A, B))), (dt, shape)


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
def test_c16_misaligned_c_and_odd_ldc(c_name):
    # C one element off a 16-byte boundary and ldc odd: no vector or tensor stores
    for name in ("tc_128x256_tma", "tc_pair256", "sgemm_128x64"):
        _check(name, c_name, 300, 264, 128, "small_int", exact=True, ldc_pad=3, c_offset=1)


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
@pytest.mark.parametrize("name", ["tc_128x256_tma", "tc_pair256", "tc_swap32", "tc_split_k",
                                  "sgemm_128x64", "generic_f16"])
def test_c16_alpha_beta(name, c_name):
    dt, opts = PLANS[name]
    M, N, K = 300, 264, 200
    A, B, As, Bs, lda, ldb = _operands(dt, "small_int", M, N, K, 1, 0)
    ldc = N + 8
    cin_vals = ((np.arange(M * ldc).reshape(M, ldc) % 9) - 4).astype(np.float64)
    c_init = oracle.encode16(c_name, cin_vals)
    alpha, beta = 1.5, -0.75
    C = run_gpu_c16(dt, As, Bs, M, N, K, lda, ldb, ldc, c_name, c_init=c_init, alpha=alpha,
                    beta=beta, **opts)
    want = alpha * oracle.gemm(dt, A, B) + beta * cin_vals[:, :N]
    # every value is a multiple of 1/4 far below 2^22: exact in FP32, rounded once
    assert np.array_equal(C, oracle.encode16(c_name, want))


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
def test_c16_pair_stream_k_cut_tiles(c_name):
    M, N, K = 2560, 2560, 1024
    A, B, _, _, _, _ = _operands("bf16", "small_int", M, N, K, 0, 0)
    C = run_gpu_c16("bf16", A, B, M, N, K, K, N, N, c_name, cta_pair=2, stream_k=2)
    assert np.array_equal(C, oracle.encode16(c_name, oracle.gemm("bf16", A, B)))


def test_c16_config_8192_sampled():
    M = N = K = 8192
    A, B = gu.make_inputs("bf16", "normal", M, N, K, 1238, sigma=1 / math.sqrt(K))
    C = oracle.decode("bf16", run_gpu_c16("bf16", A, B, M, N, K, K, N, N, "bf16"))
    assert np.isfinite(C).all()
    rows = np.concatenate([np.arange(16), np.random.default_rng(0).integers(0, M, 1024), [M - 1]])
    cols = np.concatenate([np.arange(16), np.random.default_rng(1).integers(0, N, 1024), [N - 1]])
    R = oracle.gemm_entries("bf16", A, B, rows, cols, M=M, N=N, K=K)
    e32 = _bounds("bf16", A, B, K, R)
    assert np.all(np.abs(C[rows, cols] - R) <= e32 + oracle.half_ulp16("bf16", np.abs(R) + e32))


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
def test_c16_k_zero(c_name):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    s = torch.cuda.current_stream().cuda_stream
    C = torch.full((5, 8), -1, dtype=torch.int16, device="cuda")
    g.gemm_ex(0, 0, C.data_ptr(), 5, 7, 0, 0, 7, 8, dtype=0, stream=s, c_dtype=CT[c_name])
    torch.cuda.synchronize()
    out = C.cpu().numpy().view(np.uint16)
    assert np.all(out[:, :7] == 0) and np.all(out[:, 7] == 0xFFFF)
    # K == 0 with beta: C = beta * C, rounded
    vals = np.arange(40, dtype=np.float64).reshape(5, 8)
    C = torch.from_numpy(oracle.encode16(c_name, vals).view(np.int16)).cuda()
    g.gemm_ex(0, 0, C.data_ptr(), 5, 8, 0, 0, 8, 8, dtype=1, stream=s, c_dtype=CT[c_name],
              alpha=2.0, beta=0.5)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.encode16(c_name, 0.5 * vals))


@pytest.mark.parametrize("c_name", ["f16", "bf16"])
def test_c16_host_pipeline_and_matmul(c_name):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[c_name]
    M, N, K = 2600, 2100, 300
    A, B, _, _, _, _ = _operands("bf16", "small_int", M, N, K, 4, 0)
    At = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16)
    Bt = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16)
    want = oracle.encode16(c_name, oracle.gemm("bf16", A, B))
    Ch = g.matmul(At.pin_memory(), Bt.pin_memory(), out_dtype=tdt)     # gemm_ex_host
    assert Ch.dtype == tdt and np.array_equal(Ch.view(torch.int16).numpy().view(np.uint16), want)
    Cd = g.matmul(At.cuda(), Bt.cuda(), out_dtype=tdt)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.view(torch.int16).cpu().numpy().view(np.uint16), want)
    assert "c=" + c_name in g.plan(At.cuda(), Bt.cuda(), out=Cd)


def test_c16_rejects_bad_type():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    C = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    A = torch.zeros((4, 4), dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_ex(A.data_ptr(), A.data_ptr(), C.data_ptr(), 4, 4, 4, 4, 4, 4, dtype=0, c_dtype=3)
