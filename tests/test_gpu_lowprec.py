"""GPU parity for the TF32 and 8-bit floating-point (E4M3, E5M2) tensor-core
products against the oracle.  A is M x K row-major and B is passed as its
N x K transpose (both operands K-contiguous), through the _bt entry points
and through gemm_ex on every tensor-core plan.

Tolerances: FP8 operands are decoded exactly by the oracle, so only FP32
accumulation separates the two and the standard acceptance rule applies.
TF32 drops input bits, so each element must lie within oracle.tf32_bound of
the exact product of the FP32 inputs; and the whole result must meet the
standard rule (absolute and relative-Frobenius) against the oracle's product
of the inputs cut to TF32 by one of the two readings of that cut
(oracle.tf32_cut: the low 13 fraction bits dropped, or rounded to nearest).
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TYPES = ["tf32", "e4m3", "e5m2"]
# leading-dimension granule (elements) that keeps rows on 16-byte boundaries
ALIGN = {"tf32": 4, "e4m3": 16, "e5m2": 16}

PLANS = {
    "default": {},
    "tc_128x256": dict(cta_pair=1, tile_n=256),
    "tc_128x128_plain": dict(cta_pair=1, tile_n=128, store_mode=1),
    "tc_128x64": dict(cta_pair=1, tile_n=64),
    "tc_swap16": dict(tile_n=16, swap_ab=1),
    "tc_swap64": dict(tile_n=64, swap_ab=1),
    "tc_split_k": dict(cta_pair=1, tile_n=128, split_k=3),
    "tc_stream_k": dict(cta_pair=1, tile_n=128, stream_k=2),
    "tc_pair256": dict(cta_pair=2, tile_n=256),
    "tc_pair128": dict(cta_pair=2, tile_n=128),
}


def _round_up(x, m):
    return (x + m - 1) // m * m


def _operands(dt, dist, M, N, K, seed, sigma=1.0, pad=0):
    """(A stored, Bt stored, lda, ldb, A logical, B logical K x N)."""
    A = inputs.make(dist, dt, M, K, seed, 0, sigma)
    B = inputs.make(dist, dt, K, N, seed, 1, sigma)
    Bt = np.ascontiguousarray(B.T)
    ld = _round_up(max(K, 1), ALIGN[dt]) + pad
    As = inputs.padded(A, ld) if ld != K else A
    Bs = inputs.padded(Bt, ld) if ld != K else Bt
    return As, Bs, ld, ld, A, B


def _tf32_check(C, R, S, what):
    C = np.asarray(C, dtype=np.float64)
    bound = oracle.tf32_bound(S)
    d = np.abs(C - R)
    bad = ~(d <= bound)           # NaN fails too
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside the TF32 bound; first "
                           f"{np.argwhere(bad)[0].tolist()} got {C[bad][0]} want {R[bad][0]}")


def _tf32_readings_check(C, As, Bs, M, N, K, lda, ldb, what):
    """C against the product of the inputs cut to TF32, under the standard
    acceptance rule, for at least one reading of the cut; returns it."""
    cmps = {}
    for mode in ("trunc", "rne"):
        Ac, Bc = oracle.tf32_cut(As, mode), oracle.tf32_cut(Bs, mode)
        R = oracle.gemm_op("f32", False, True, Ac, Bc, M, N, K, lda=lda, ldb=ldb)
        amax = float(np.abs(Ac.reshape(-1, lda)[:, :K]).max()) if K else 0.0
        bmax = float(np.abs(Bc.reshape(-1, ldb)[:, :K]).max()) if K else 0.0
        cmps[mode] = oracle.compare(C, R, K, amax, bmax)
    assert any(c.ok for c in cmps.values()), f"{what}: {cmps}"
    return [m for m, c in cmps.items() if c.ok][0]


def _check(dt, opts, M, N, K, dist, exact, pad=0, seed=0, sigma=1.0):
    As, Bs, lda, ldb, A, B = _operands(dt, dist, M, N, K, seed, sigma, pad)
    o = dict(opts, trans_b=1) if opts else {}
    C = gu.run_gpu(dt, As, Bs, M, N, K, lda=lda, ldb=ldb, **o)
    R = oracle.gemm_op(dt, False, True, As, Bs, M, N, K, lda=lda, ldb=ldb)
    what = f"{dt} {dist} {M}x{N}x{K} {opts}"
    if dt == "tf32":
        S = oracle.gemm_op("f32", False, True, np.abs(As), np.abs(Bs), M, N, K, lda=lda, ldb=ldb)
        _tf32_check(C, R, S, what)
        _tf32_readings_check(C, As, Bs, M, N, K, lda, ldb, what)
        if exact:
            assert np.array_equal(C, R.astype(np.float32)), what
        return
    cmp = oracle.compare(C, R, K, inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt))
    assert cmp.ok, f"{what}: {cmp}"
    if exact:
        assert cmp.exact, f"{what}: not bit-exact: {cmp}"


@pytest.mark.parametrize("dt", TYPES)
@pytest.mark.parametrize("name", sorted(PLANS))
def test_lowprec_plans_exact(dt, name):
    _check(dt, PLANS[name], 300, 520, 700, "small_int", exact=True, pad=ALIGN[dt])


@pytest.mark.parametrize("dt", TYPES)
@pytest.mark.parametrize("name", sorted(PLANS))
def test_lowprec_plans_random_ragged(dt, name):
    _check(dt, PLANS[name], 257, 130, 72, "uniform", exact=False, seed=3)


@pytest.mark.parametrize("dt", TYPES)
@pytest.mark.parametrize("shape", [(1024, 1536, 512), (8, 1024, 2048), (2048, 64, 256),
                                   (4000, 2248, 512), (129, 17, 33), (1, 1, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_lowprec_default_plan_shapes(dt, shape):
    M, N, K = shape
    _check(dt, {}, M, N, K, "small_int", exact=True)
    _check(dt, {}, M, N, K, "normal", exact=False, seed=11, sigma=1 / math.sqrt(K))


@pytest.mark.parametrize("dt", TYPES)
def test_lowprec_k_tail_of_one_element(dt):
    # K one past a k-block boundary: the last k-block holds a single element
    kb = {"tf32": 32, "e4m3": 128, "e5m2": 128}[dt]
    _check(dt, {}, 256, 256, 2 * kb + 1, "uniform", exact=False, seed=5)


@pytest.mark.parametrize("dt", TYPES)
def test_lowprec_alpha_beta(dt):
    M, N, K = 300, 260, 200
    As, Bs, lda, ldb, A, B = _operands(dt, "uniform", M, N, K, 7)
    Cin = inputs.uniform_f32(7, 2, (M, N))
    alpha, beta = 0.75, -1.5
    C = gu.run_gpu(dt, As, Bs, M, N, K, lda=lda, ldb=ldb, c_init=Cin, trans_b=1,
                   alpha=alpha, beta=beta)
    R = oracle.gemm_op(dt, False, True, As, Bs, M, N, K, lda=lda, ldb=ldb)
    want = alpha * R + beta * Cin.astype(np.float64)
    if dt == "tf32":
        S = oracle.gemm_op("f32", False, True, np.abs(As), np.abs(Bs), M, N, K, lda=lda, ldb=ldb)
        bound = abs(alpha) * oracle.tf32_bound(S) + 2.0 ** -21 * (abs(beta) + abs(alpha) * S)
        assert np.all(np.abs(C - want) <= bound)
        # the relative Frobenius half of the rule, against the TF32-cut product
        mode = _tf32_readings_check((C - beta * Cin.astype(np.float64)) / alpha, As, Bs, M, N, K,
                                    lda, ldb, "tf32 alpha/beta")
        Ac, Bc = oracle.tf32_cut(As, mode), oracle.tf32_cut(Bs, mode)
        want = alpha * oracle.gemm_op("f32", False, True, Ac, Bc, M, N, K, lda=lda, ldb=ldb) + \
            beta * Cin.astype(np.float64)
    else:
        tol = oracle.general_bounds(K, inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt),
                                    alpha, beta, 1.0)
        assert float(np.max(np.abs(C - want))) <= tol
    rel = np.linalg.norm(C - want) / np.linalg.norm(want)
    assert rel <= oracle.REL_FROB, rel


@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_fp8_saturated_and_subnormal_values(dt):
    # every finite code of the format, so the largest normals and the
    # subnormals reach the tensor cores; products stay exact in FP32 when
    # one operand is a power of two
    import torch
    M, N, K = 128, 128, 256
    tt = torch.float8_e4m3fn if dt == "e4m3" else torch.float8_e5m2
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(tt).float().numpy()
    finite = codes[np.isfinite(vals)]
    rng = np.random.default_rng(17)
    A = finite[rng.integers(0, finite.size, size=(M, K))].astype(np.uint8)
    pow2 = np.array([0x38 if dt == "e4m3" else 0x3C, 0x40 if dt == "e4m3" else 0x40],
                    dtype=np.uint8)   # 1.0, 2.0
    Bt = np.zeros((N, K), dtype=np.uint8)
    Bt[np.arange(N), np.arange(N) % K] = pow2[np.arange(N) % 2]
    C = gu.run_gpu(dt, A, Bt, M, N, K, lda=K, ldb=K)
    R = oracle.gemm_op(dt, False, True, A, Bt, M, N, K)
    assert np.array_equal(C, R.astype(np.float32))


@pytest.mark.parametrize("dt", TYPES)
def test_lowprec_config_4096_full(dt):
    M = N = K = 4096
    _check(dt, {}, M, N, K, "normal", exact=False, seed=1240, sigma=1 / math.sqrt(K))


def test_fp8_8192_full_in_bench_configuration():
    M = N = K = 8192
    _check("e4m3", {}, M, N, K, "normal", exact=False, seed=1241, sigma=1 / math.sqrt(K))


def test_tf32_is_not_fp32():
    # FP32 inputs whose low mantissa bits TF32 drops: the product differs
    # from the FP32 SGEMM's by far more than FP32 rounding, within the bound
    M = N = K = 128
    As, Bs, lda, ldb, A, B = _operands("tf32", "uniform", M, N, K, 9)
    C = gu.run_gpu("tf32", As, Bs, M, N, K, lda=lda, ldb=ldb)
    R = oracle.gemm_op("tf32", False, True, As, Bs, M, N, K, lda=lda, ldb=ldb)
    rel = np.linalg.norm(C - R) / np.linalg.norm(R)
    assert rel > 1e-5, rel      # FP32 alone would be near 1e-7


@pytest.mark.parametrize("dt", TYPES)
def test_lowprec_rejects_other_layouts_and_alignment(dt):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    code = gu.CODE[dt]
    eb = 4 if dt == "tf32" else 1
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    with pytest.raises(g.GemmError):   # B K x N (N-contiguous)
        g.gemm_ex(p, p, C.data_ptr(), 64, 64, 64, 64, 64, 64, dtype=code, stream=s)
    with pytest.raises(g.GemmError):   # A stored transposed
        g.gemm_ex(p, p, C.data_ptr(), 64, 64, 64, 64, 64, 64, dtype=code, stream=s,
                  trans_a=1, trans_b=1)
    bad_ld = 64 + ALIGN[dt] // 2 if ALIGN[dt] > 1 else 65
    with pytest.raises(g.GemmError):   # rows off 16-byte boundaries
        g.gemm_ex(p, p, C.data_ptr(), 64, 64, 64, bad_ld, 64, 64, dtype=code, stream=s,
                  trans_b=1)
    with pytest.raises(g.GemmError):   # misaligned base
        g.gemm_ex(p + eb, p, C.data_ptr(), 64, 64, 64, 64, 64, 64, dtype=code, stream=s,
                  trans_b=1)
    with pytest.raises(g.GemmError):   # no generic kernel for these types
        g.gemm_ex(p, p, C.data_ptr(), 64, 64, 64, 64, 64, 64, dtype=code, stream=s,
                  trans_b=1, generic=1)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dt", TYPES)
def test_lowprec_k_zero_and_empty(dt):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    fn = {"tf32": g.gemm_tf32f32_bt, "e4m3": g.gemm_e4m3f32_bt, "e5m2": g.gemm_e5m2f32_bt}[dt]
    C = torch.full((5, 7), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    fn(0, 0, C.data_ptr(), 5, 7, 0, 16, 16, 7, s)
    torch.cuda.synchronize()
    assert torch.all(C == 0).item()
    before = g.gemm_launch_count()
    fn(0, 0, 0, 0, 16, 16, 16, 16, 16, s)
    fn(0, 0, 0, 16, 0, 16, 16, 16, 0, s)
    torch.cuda.synchronize()
    assert g.gemm_launch_count() == before


def test_matmul_fp8_and_tf32():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 256, 192, 320
    for dt, tt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        As, Bs, lda, ldb, A, B = _operands(dt, "small_int", M, N, K, 2)
        Ad = torch.from_numpy(As).cuda().view(tt)
        Btd = torch.from_numpy(Bs).cuda().view(tt)
        C = g.matmul(Ad, Btd.t())
        torch.cuda.synchronize()
        R = oracle.gemm(dt, A, B)
        assert np.array_equal(C.cpu().numpy(), R.astype(np.float32)), dt
        assert "tcgen05" in g.plan(Ad, Btd.t())
    As, Bs, lda, ldb, A, B = _operands("tf32", "small_int", M, N, K, 2)
    C = g.matmul(torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda().t(), tf32=True)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.gemm("f32", A, B).astype(np.float32))
