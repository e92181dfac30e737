"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  Needs a GB300 and the built library."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    from dense_gemm_tensor_tcgen05_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    build.build()
    oracle.build()
    g.lib()
    yield


# ---- exact cases first: small integers are exact in every summation order ----

EXACT_SHAPES = [(1, 1, 1), (7, 9, 5), (128, 256, 64), (128, 64, 64), (100, 300, 70),
                (256, 512, 1024), (129, 257, 65), (8, 200, 130), (33, 1000, 129)]


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("shape", EXACT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_int_exact_default_plan(dt, shape):
    M, N, K = shape
    gu.check_full(dt, "small_int", M, N, K, exact=True)


TC_CONFIGS = [
    dict(tile_n=256, swap_ab=0, split_k=1), dict(tile_n=128, swap_ab=0, split_k=1),
    dict(tile_n=64, swap_ab=0, split_k=1), dict(tile_n=16, swap_ab=1, split_k=1),
    dict(tile_n=32, swap_ab=1, split_k=1), dict(tile_n=64, swap_ab=1, split_k=1),
    dict(tile_n=256, swap_ab=0, split_k=3), dict(tile_n=128, swap_ab=0, split_k=2),
    dict(tile_n=64, swap_ab=0, split_k=7), dict(tile_n=16, swap_ab=1, split_k=4),
    dict(tile_n=64, swap_ab=1, split_k=5), dict(tile_n=128, swap_ab=0, split_k=1, group_m=1),
    dict(tile_n=256, swap_ab=0, split_k=1, group_m=3),
    dict(cta_pair=2, tile_n=256), dict(cta_pair=2, tile_n=128),
    dict(cta_pair=2, tile_n=256, group_m=1), dict(cta_pair=1, tile_n=256),
    dict(cta_pair=1, stream_k=2, tile_n=256), dict(cta_pair=1, stream_k=2, tile_n=64),
    dict(stream_k=2, tile_n=16, swap_ab=1), dict(stream_k=2, tile_n=64, swap_ab=1),
    dict(cta_pair=1, stream_k=1, tile_n=128),
]


def _cfg_id(c):
    return "-".join(f"{k}{v}" for k, v in c.items())


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("cfg", TC_CONFIGS, ids=_cfg_id)
@pytest.mark.parametrize("shape", [(300, 520, 700), (1, 129, 1000), (640, 512, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tensor_core_configs_exact(dt, cfg, shape):
    M, N, K = shape
    gu.check_full(dt, "small_int", M, N, K, exact=True, **cfg)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("cfg", TC_CONFIGS, ids=_cfg_id)
def test_tensor_core_configs_random(dt, cfg):
    gu.check_full(dt, "uniform", 333, 450, 1111, seed=5, **cfg)


@pytest.mark.parametrize("cfg", [dict(tile_n=256), dict(tile_n=128), dict(tile_n=64), dict(tile_n=32),
                                 dict(tile_n=256, split_k=3)], ids=_cfg_id)
@pytest.mark.parametrize("shape", [(300, 520, 700), (9, 7, 3), (130, 200, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_sgemm_tiles_exact(cfg, shape):
    M, N, K = shape
    gu.check_full("f32", "small_int", M, N, K, exact=True, **cfg)


# ---- the workloads' configurations ------------------------------------------

def test_config_f16_1024_uniform_full():
    gu.check_full("f16", "uniform", 1024, 1024, 1024, seed=1234)


def test_config_sgemm_1024_uniform_full():
    gu.check_full("f32", "uniform", 1024, 1024, 1024, seed=1235)


# Every element of C is compared with the oracle at the workloads' full sizes,
# on the default plan of each fixed entry point (the plan the benchmark
# times).  The oracle threads over all host cores; 8192^3 takes about 20 s.

def test_config_sgemm_4096_uniform_full():
    gu.check_full("f32", "uniform", 4096, 4096, 4096, seed=1236)


def test_config_f16_2048_normal_full():
    gu.check_full("f16", "normal", 2048, 2048, 2048, seed=1237)


def _default_plan(dt, M, N, K):
    import dense_gemm_tensor_tcgen05_gb300 as g
    return g.gemm_plan_describe(gu.CODE[dt], 1 << 20, 1 << 34, 1 << 40, M, N, K, K, N, N)


def test_config_bf16_8192_normal_full():
    M = N = K = 8192
    assert "pair=1" in _default_plan("bf16", M, N, K)
    gu.check_full("bf16", "normal", M, N, K, seed=1238, sigma=1 / math.sqrt(K))


def test_config_bf16_8192_small_int_exact_default_plan():
    # every partial sum is an integer below 6K < 2^24: the CTA-pair kernel's
    # whole 32-wave schedule must reproduce the oracle bit for bit
    M = N = K = 8192
    gu.check_full("bf16", "small_int", M, N, K, exact=True)


@pytest.mark.parametrize("shape", [(4000, 3000, 1000), (16384, 128, 4096), (8, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_config_ragged_skinny_full(shape):
    M, N, K = shape
    gu.check_full("f16", "uniform", M, N, K, seed=1239)


@pytest.mark.parametrize("shape", [(4000, 3000, 1000), (16384, 128, 4096), (8, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_config_ragged_skinny_small_int_exact(shape):
    M, N, K = shape
    gu.check_full("f16", "small_int", M, N, K, exact=True)


# ---- edges and degenerate cases ----------------------------------------------

EDGE = [1, 2, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257]


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("aligned", [True, False], ids=["aligned_ld", "tight_ld"])
def test_edge_sweep_small_int(dt, aligned):
    rng = np.random.default_rng(7)
    align = (8 if dt != "f32" else 4) if aligned else 0
    for _ in range(40):
        M, N, K = (int(x) for x in rng.choice(EDGE, size=3))
        gu.check_full(dt, "small_int", M, N, K, exact=True, align_ld=align)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_tiny_shapes_tensor_core_path(dt):
    # every (M, N, K) in 1..9 through the TMA + tcgen05 kernels (padded rows),
    # with and without swap
    for M in range(1, 10):
        for N in range(1, 10, 2):
            for K in range(1, 10, 2):
                gu.check_full(dt, "small_int", M, N, K, exact=True, align_ld=8)
                gu.check_full(dt, "uniform", M, N, K, seed=K, align_ld=8, swap_ab=0)


@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_tiny_shapes_bruteforce(dt):
    for M in range(1, 10, 2):
        for N in range(1, 10, 3):
            for K in range(1, 10, 4):
                gu.check_full(dt, "uniform", M, N, K, seed=M * 100 + N * 10 + K)


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_padded_leading_dimensions(dt):
    # padding holds poison; a kernel that reads or writes past K or N fails
    gu.check_full(dt, "small_int", 200, 300, 150, exact=True, pad=(8, 16, 12))
    gu.check_full(dt, "uniform", 131, 77, 259, seed=3, pad=(24, 8, 5))


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_misaligned_pointers_and_leading_dims(dt):
    M, N, K = 70, 90, 50          # K, N not multiples of 8: no TMA, no float4
    A, B = gu.make_inputs(dt, "small_int", M, N, K, 0)
    C = gu.run_gpu(dt, A, B, M, N, K, offsets=(1, 3, 1))
    R = oracle.gemm(dt, A, B)
    assert np.array_equal(C, R.astype(np.float32))


def test_k_zero_gives_zeros():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    for dt, fn in (("f16", g.gemm_f16f32), ("bf16", g.gemm_bf16f32), ("f32", g.sgemm_f32)):
        C = torch.full((5, 7), float("nan"), device="cuda")
        fn(0, 0, C.data_ptr(), 5, 7, 0, 0, 7, 7, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert torch.all(C == 0).item(), dt


def test_m_or_n_zero_is_a_no_op():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    before = g.gemm_launch_count()
    g.gemm_f16f32(0, 0, 0, 0, 16, 16, 16, 16, 16)
    g.gemm_bf16f32(0, 0, 0, 16, 0, 16, 16, 0, 0)
    torch.cuda.synchronize()
    assert g.gemm_launch_count() == before


def test_golden_fixtures_on_gpu():
    import os
    gold = os.path.join(os.path.dirname(__file__), "golden")

    def load(name, M, N):
        v = [float(l) for l in open(os.path.join(gold, name)) if not l.startswith("#")]
        return np.array(v).reshape(M, N)

    A, B = gu.make_inputs("f16", "small_int", 12, 10, 9, 0)
    C = gu.run_gpu("f16", A, B, 12, 10, 9)
    assert np.array_equal(C, load("small_int_12x10x9.txt", 12, 10).astype(np.float32))
    A, B = gu.make_inputs("f16", "mod_pattern", 16, 16, 16, 0)
    C = gu.run_gpu("f16", A, B, 16, 16, 16)
    cmp = oracle.compare(C, load("mod_pattern_16.txt", 16, 16), 16, 0.5, 0.5)
    assert cmp.ok, str(cmp)


# ---- determinism, streams, host buffers --------------------------------------------

@pytest.mark.parametrize("cfg", [dict(), dict(tile_n=64, swap_ab=1, split_k=6),
                                 dict(tile_n=128, swap_ab=0, split_k=5),
                                 dict(cta_pair=1, tile_n=128, stream_k=2)], ids=_cfg_id)
def test_repeat_runs_bit_identical(cfg):
    A, B = gu.make_inputs("bf16", "normal", 96, 1000, 2048, 11)
    Cs = [gu.run_gpu("bf16", A, B, 96, 1000, 2048, **cfg) for _ in range(4)]
    for C in Cs[1:]:
        assert np.array_equal(C, Cs[0])


def test_concurrent_streams_split_k():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 8, 4096, 8192
    A, B = gu.make_inputs("f16", "small_int", M, N, K, 0)
    Ad, Bd = gu.to_device(A, "f16"), gu.to_device(B, "f16")
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = [torch.full((M, N), float("nan"), device="cuda") for _ in streams]
    torch.cuda.synchronize()
    for _ in range(3):
        for s, C in zip(streams, outs):
            g.gemm_f16f32(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                          s.cuda_stream)
    torch.cuda.synchronize()
    g.gemm_device_error()
    R = oracle.gemm("f16", A, B).astype(np.float32)
    for C in outs:
        assert np.array_equal(C.cpu().numpy(), R)


def test_matmul_with_host_buffers():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    A, B = gu.make_inputs("bf16", "uniform", 300, 200, 500, 21)
    At = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()
    Bt = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).pin_memory()
    C = g.matmul(At, Bt)
    assert not C.is_cuda
    R = oracle.gemm("bf16", A, B)
    cmp = oracle.compare(C.numpy(), R, 500, inputs.bits_abs_max(A, "bf16"), inputs.bits_abs_max(B, "bf16"))
    assert cmp.ok, str(cmp)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(256, 256, 64), (257, 255, 65), (1024, 1280, 2048),
                                   (130, 700, 300), (600, 260, 4100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cta_pair_kernel(dt, shape):
    M, N, K = shape
    gu.check_full(dt, "small_int", M, N, K, exact=True, cta_pair=2)
    gu.check_full(dt, "normal", M, N, K, seed=3, cta_pair=2)


MULTI_TILE_PLANS = [dict(cta_pair=1, tile_n=256), dict(cta_pair=1, tile_n=128),
                    dict(cta_pair=1, tile_n=64), dict(cta_pair=2, tile_n=256),
                    dict(cta_pair=2, tile_n=128), dict(cta_pair=1, tile_n=256, store_mode=1),
                    dict(cta_pair=2, tile_n=256, store_mode=1),
                    dict(cta_pair=1, tile_n=256, stream_k=2), dict(cta_pair=1, tile_n=128, stream_k=2),
                    dict(cta_pair=1, tile_n=256, stream_k=2, store_mode=1),
                    dict(cta_pair=2, tile_n=256, stream_k=2), dict(cta_pair=2, tile_n=128, stream_k=2),
                    dict(cta_pair=2, tile_n=256, stream_k=2, store_mode=1)]


@pytest.mark.parametrize("cfg", MULTI_TILE_PLANS, ids=_cfg_id)
@pytest.mark.parametrize("shape", [(4000, 3000, 1000), (4000, 2248, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_multi_tile_ragged_every_plan(cfg, shape):
    # several tiles per CTA with ragged M and N; (4000, 2248, 512) leaves a
    # single 32-column chunk of the last 256-wide tile wholly past N
    M, N, K = shape
    gu.check_full("f16", "small_int", M, N, K, exact=True, **cfg)
    gu.check_full("bf16", "uniform", M, N, K, seed=4, **cfg)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(2560, 2560, 1024), (2500, 2600, 1000), (1280, 4864, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cta_pair_stream_k_cut_tiles(dt, shape):
    # more 256 x 256 tiles than clusters with a partial last wave: tiles are
    # cut into pieces along K and summed by the last piece to finish
    M, N, K = shape
    import dense_gemm_tensor_tcgen05_gb300 as g
    A, B = gu.make_inputs(dt, "small_int", M, N, K, 0)
    desc = g.gemm_plan_describe(gu.CODE[dt], 1 << 20, 1 << 34, 1 << 40, M, N, K, K, N, N, cta_pair=2,
                                stream_k=2)
    assert "pair=1" in desc and "stream_k" in desc and "max_seg=1 " not in desc, desc
    C = gu.run_gpu(dt, A, B, M, N, K, cta_pair=2, stream_k=2)
    assert np.array_equal(C, oracle.gemm(dt, A, B).astype(np.float32))


def test_cta_pair_stream_k_on_request_only():
    import dense_gemm_tensor_tcgen05_gb300 as g
    args = (1 << 20, 1 << 34, 1 << 40, 8192, 8192, 8192, 8192, 8192, 8192)
    assert "stream_k" not in g.gemm_plan_describe(1, *args)
    assert "stream_k" in g.gemm_plan_describe(1, *args, stream_k=2)


def test_cta_pair_many_units_per_cluster():
    # more pair tiles than resident clusters: every cluster loops over several
    # tiles and both accumulators
    gu.check_full("bf16", "small_int", 4096, 4096, 256, exact=True, cta_pair=2)


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", [(2600, 384, 520), (2600, 2100, 300), (700, 3000, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_ex_host_pipeline(dt, pinned, shape):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = shape    # row panels and column panels, the last ones ragged
    lda, ldb, ldc = K + 8, N + 4, N + 4
    A, B = gu.make_inputs(dt, "small_int", M, N, K, 0)
    Ap, Bp = inputs.padded(A, lda), inputs.padded(B, ldb)
    Ch = np.full((M, ldc), np.nan, dtype=np.float32)
    if pinned:
        At = torch.from_numpy(Ap.view(np.int32 if dt == "f32" else np.int16)).pin_memory()
        Bt = torch.from_numpy(Bp.view(np.int32 if dt == "f32" else np.int16)).pin_memory()
        Ct = torch.from_numpy(Ch).pin_memory()
        ptrs = (At.data_ptr(), Bt.data_ptr(), Ct.data_ptr())
    else:
        Ct = None
        ptrs = (Ap.ctypes.data, Bp.ctypes.data, Ch.ctypes.data)
    stream = torch.cuda.current_stream()
    for _ in range(2):   # the second call reuses the library's staging buffers
        g.gemm_ex_host(*ptrs, M, N, K, lda, ldb, ldc, dtype=gu.CODE[dt], stream=stream.cuda_stream)
        stream.synchronize()
        C = Ct.numpy() if pinned else Ch
        R = oracle.gemm(dt, A, B)
        assert np.array_equal(C[:, :N], R.astype(np.float32))
        assert np.all(np.isnan(C[:, N:]))


def test_matmul_host_uses_pipeline():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    A, B = gu.make_inputs("f16", "uniform", 1500, 256, 300, 8)
    At = torch.from_numpy(A.view(np.int16)).view(torch.float16)
    Bt = torch.from_numpy(B.view(np.int16)).view(torch.float16)
    C = g.matmul(At, Bt)
    R = oracle.gemm("f16", A, B)
    cmp = oracle.compare(C.numpy(), R, 300, inputs.bits_abs_max(A, "f16"), inputs.bits_abs_max(B, "f16"))
    assert cmp.ok, str(cmp)


def test_watchdog_gives_up_and_context_stays_usable():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    s = torch.cuda.current_stream().cuda_stream
    g.gemm_device_error(s)                          # start from a clear error word
    g.gemm_watchdog_selftest(20, s)                 # a wait nothing satisfies, 20 ms limit
    with pytest.raises(g.GemmError) as e:
        g.gemm_device_error(s)
    assert e.value.name == "GEMM_ERR_DEVICE_TIMEOUT"
    g.gemm_device_error(s)                          # the word was cleared
    gu.check_full("bf16", "small_int", 300, 520, 700, exact=True)   # GEMMs still work


def test_plan_describe_routes():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g

    def plan(dt, M, N, K):
        A = torch.empty((M, K), dtype=gu.torch_dtype(dt), device="cuda")
        B = torch.empty((K, N), dtype=gu.torch_dtype(dt), device="cuda")
        return g.plan(A, B)
    assert plan("bf16", 8192, 8192, 8192).startswith("tcgen05")
    assert "pair=1" in plan("bf16", 8192, 8192, 8192)
    assert "swap=1" in plan("f16", 8, 8192, 8192)
    assert plan("f32", 4096, 4096, 4096).startswith("sgemm")
    assert plan("f16", 10, 10, 7).startswith("generic")   # lda = 7: no TMA


@pytest.mark.parametrize("cfg", [dict(tile_n=64, stream_k=2), dict(tile_n=128, stream_k=2),
                                 dict(tile_n=32, stream_k=2), dict(tile_n=256, stream_k=2)],
                         ids=_cfg_id)
@pytest.mark.parametrize("shape", [(300, 520, 700), (1024, 1024, 1024), (9, 7, 3), (130, 200, 1),
                                   (2000, 3000, 256), (64, 64, 16000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_sgemm_stream_k_exact(cfg, shape):
    # the SGEMM's persistent stream-K grid: whole tiles, then K steps shared
    # out evenly; cut tiles are summed by their last piece in piece order
    M, N, K = shape
    gu.check_full("f32", "small_int", M, N, K, exact=True, **cfg)
    gu.check_full("f32", "uniform", M, N, K, seed=M + N + K, **cfg)


def test_sgemm_stream_k_repeat_bit_identical():
    A, B = gu.make_inputs("f32", "uniform", 1024, 1024, 1024, 3)
    Cs = [gu.run_gpu("f32", A, B, 1024, 1024, 1024, tile_n=64, stream_k=2) for _ in range(3)]
    for C in Cs[1:]:
        assert np.array_equal(C, Cs[0])


@pytest.mark.parametrize("shape", [(6144, 6144, 256), (5000, 5004, 300)],
                         ids=lambda s: "x".join(map(str, s)))
def test_sgemm_default_wide_micro_tile_exact(shape):
    # from four waves of 128 x 128 tiles on, the default SGEMM plan runs
    # whole waves of tiles with 8 x 16 outputs per thread (ragged edges in
    # the second shape)
    M, N, K = shape
    assert "thread=8x16" in _default_plan("f32", M, N, K), _default_plan("f32", M, N, K)
    gu.check_full("f32", "small_int", M, N, K, exact=True)
    gu.check_full("f32", "uniform", M, N, K, seed=M + K)



@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", [((2560, 2600, 1024), dict(cta_pair=2, stream_k=3)),
                                  ((2560, 2048, 512), dict(cta_pair=1, tile_n=256, stream_k=3)),
                                  ((3000, 2100, 700), dict(cta_pair=1, tile_n=128, stream_k=3)),
                                  ((4000, 3000, 1000), dict(cta_pair=2, stream_k=3))],
                         ids=lambda c: "x".join(map(str, c[0])) + "-" + _cfg_id(c[1]))
def test_tail_split_exact_and_random(dt, case):
    # whole waves of whole tiles, then the leftover tiles each cut into equal
    # K pieces over more CTAs (or clusters), summed in piece order
    (M, N, K), cfg = case
    gu.check_full(dt, "small_int", M, N, K, exact=True, **cfg)
    gu.check_full(dt, "uniform", M, N, K, seed=9, **cfg)


def test_tail_split_plan_text():
    import dense_gemm_tensor_tcgen05_gb300 as g
    args = (1 << 20, 1 << 34, 1 << 40, 2560, 2600, 1024, 1024, 2600, 2600)
    assert "tail_split" in g.gemm_plan_describe(1, *args, cta_pair=2, stream_k=3)
    # fewer leftover tiles than half a wave's worth is what tail split needs;
    # a whole number of waves leaves nothing to cut
    assert "tail_split" not in g.gemm_plan_describe(1, 1 << 20, 1 << 34, 1 << 40, 256 * 76, 256, 1024,
                                                    1024, 256, 256, cta_pair=2, stream_k=3)


def test_tail_split_is_the_default_from_eight_waves():
    import dense_gemm_tensor_tcgen05_gb300 as g
    plan = lambda n: g.gemm_plan_describe(1, 1 << 20, 1 << 34, 1 << 40, n, n, n, n, n, n)
    assert "tail_split" in plan(8192) and "pair=1" in plan(8192)     # 13 waves + 36 tiles
    assert "tail_split" not in plan(4096)                             # 3 waves + 28 tiles
    assert "tail_split" not in plan(16384)                            # 53 waves + 68 tiles: S = 1
    assert "tail_split" not in g.gemm_plan_describe(1, 1 << 20, 1 << 34, 1 << 40, 8192, 8192, 8192,
                                                    8192, 8192, 8192, stream_k=1)
