"""The tensor-core kernels' own failure path, exercised without any fault.

gemm_ex_stall_selftest runs an ordinary plan with every pipeline wait limited
to a few tens of milliseconds and one CTA's (or CTA pair's) TMA producer
withholding the copies of one pipeline stage.  The MMA thread's wait for that
stage runs out, the CTA records the timeout in the device error word, leaves
its loops, waits (bounded) for its own copies and MMAs, frees its tensor
memory and exits; every other CTA finishes normally.  Each test checks that

  * the call returns promptly and gemm_device_error reports
    GEMM_ERR_DEVICE_TIMEOUT (then a clear word);
  * the next ordinary product on the same stream -- the same plan, so the
    same kernel, workspace and split-K counters -- is bit-exact against the
    oracle, which shows the aborted CTA freed its tensor memory (an
    allocation would otherwise wait forever) and that the counters it left
    part-way were cleared;
  * a stall index past the CTA's last stage fill changes nothing.
"""
from __future__ import annotations

import time

import numpy as np
import pytest

import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

LIMIT_MS = 20

# (dtype, M, N, K, plan options): every kernel form with a pipeline.  Each
# plan gives CTA 0 at least three stage fills (the stall is at fill 2).
PLANS = {
    "one_cta_whole_tiles": ("bf16", 512, 512, 4096, dict(cta_pair=1, tile_n=128, split_k=1)),
    "one_cta_tma_store_256": ("f16", 384, 768, 2048, dict(cta_pair=1, tile_n=256, split_k=1)),
    "one_cta_split_k": ("bf16", 300, 520, 2000, dict(cta_pair=1, tile_n=128, split_k=3)),
    "swap_split_k": ("f16", 8, 4096, 8192, dict(tile_n=16, swap_ab=1, split_k=4)),
    "one_cta_stream_k": ("bf16", 1000, 1104, 1536, dict(cta_pair=1, tile_n=64, stream_k=2)),
    "pair_whole_tiles": ("bf16", 1024, 1024, 4096, dict(cta_pair=2, tile_n=256)),
    "pair_128": ("f16", 768, 512, 2048, dict(cta_pair=2, tile_n=128)),
    "pair_stream_k": ("bf16", 2560, 2600, 1024, dict(cta_pair=2, stream_k=2)),
    "e4m3_one_cta": ("e4m3", 512, 384, 4096, dict(cta_pair=1, tile_n=128, split_k=1, trans_b=1)),
}


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


def _operands(dt, M, N, K, opts):
    A, B = gu.make_inputs(dt, "small_int", M, N, K, 0)
    if opts.get("trans_b"):
        Bs = np.ascontiguousarray(B.T)           # stored N x K
        return A, B, gu.to_device(A, dt), gu.to_device(Bs, dt), K
    return A, B, gu.to_device(A, dt), gu.to_device(B, dt), N


def _run(fn_name, dt, Ad, Bd, M, N, K, ldb, opts, stream, **extra):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    args = (Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, ldb, N)
    getattr(g, fn_name)(*args, dtype=gu.CODE[dt], stream=stream.cuda_stream, **extra, **opts)
    return C


@pytest.mark.parametrize("name", sorted(PLANS))
def test_stalled_stage_times_out_and_next_call_is_exact(name):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    dt, M, N, K, opts = PLANS[name]
    A, B, Ad, Bd, ldb = _operands(dt, M, N, K, opts)
    want = oracle.gemm(dt, A, B).astype(np.float32)
    desc = g.gemm_plan_describe(gu.CODE[dt], Ad.data_ptr(), Bd.data_ptr(), 1 << 20, M, N, K, K,
                                ldb, N, **opts)
    assert desc.startswith("tcgen05"), desc
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    # warm the plan (workspace allocated, kernels loaded) and start from a
    # clear error word
    C0 = _run("gemm_ex", dt, Ad, Bd, M, N, K, ldb, opts, stream)
    g.gemm_device_error(sh)
    assert np.array_equal(C0.cpu().numpy(), want)

    t0 = time.perf_counter()
    _run("gemm_ex_stall_selftest", dt, Ad, Bd, M, N, K, ldb, opts, stream,
         limit_ms=LIMIT_MS, stall_cta=0, stall_fill=2)
    with pytest.raises(g.GemmError) as e:
        g.gemm_device_error(sh)
    elapsed = time.perf_counter() - t0
    assert e.value.name == "GEMM_ERR_DEVICE_TIMEOUT", str(e.value)
    # the limit, the bounded drains and a cluster's final wait, far below the
    # 2 s a production wait would take
    assert elapsed < 1.5, f"abort took {elapsed:.3f} s"
    g.gemm_device_error(sh)                      # the word was cleared

    # the same plan again on the same stream and workspace: exact
    for _ in range(2):
        C = _run("gemm_ex", dt, Ad, Bd, M, N, K, ldb, opts, stream)
        g.gemm_device_error(sh)
        assert np.array_equal(C.cpu().numpy(), want), name


@pytest.mark.parametrize("name", ["one_cta_whole_tiles", "pair_whole_tiles", "one_cta_split_k"])
def test_stall_past_the_last_fill_changes_nothing(name):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    dt, M, N, K, opts = PLANS[name]
    A, B, Ad, Bd, ldb = _operands(dt, M, N, K, opts)
    stream = torch.cuda.Stream()
    C = _run("gemm_ex_stall_selftest", dt, Ad, Bd, M, N, K, ldb, opts, stream,
             limit_ms=LIMIT_MS, stall_cta=0, stall_fill=1 << 30)
    g.gemm_device_error(stream.cuda_stream)      # no timeout
    assert np.array_equal(C.cpu().numpy(), oracle.gemm(dt, A, B).astype(np.float32))


def test_stall_in_the_last_cta_of_a_multi_wave_grid():
    # more tiles than CTAs: the stalled CTA aborts in its second work item,
    # after it has already stored a whole tile, and the others keep going
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    dt, M, N, K = "bf16", 4096, 4096, 512
    opts = dict(cta_pair=1, tile_n=64)
    A, B, Ad, Bd, ldb = _operands(dt, M, N, K, opts)
    desc = g.gemm_plan_describe(gu.CODE[dt], Ad.data_ptr(), Bd.data_ptr(), 1 << 20, M, N, K, K, N,
                                N, **opts)
    grid = int(desc.split("grid=")[1].split()[0])
    stream = torch.cuda.Stream()
    kb = K // 64
    _run("gemm_ex_stall_selftest", dt, Ad, Bd, M, N, K, ldb, opts, stream,
         limit_ms=LIMIT_MS, stall_cta=grid - 1, stall_fill=kb + 3)
    with pytest.raises(g.GemmError) as e:
        g.gemm_device_error(stream.cuda_stream)
    assert e.value.name == "GEMM_ERR_DEVICE_TIMEOUT"
    C = _run("gemm_ex", dt, Ad, Bd, M, N, K, ldb, opts, stream)
    g.gemm_device_error(stream.cuda_stream)
    assert np.array_equal(C.cpu().numpy(), oracle.gemm(dt, A, B).astype(np.float32))


def test_stall_selftest_rejects_plans_without_a_pipeline():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    A = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    for dt, extra in ((2, {}), (0, dict(generic=1))):
        with pytest.raises(g.GemmError) as e:
            g.gemm_ex_stall_selftest(A.data_ptr(), A.data_ptr() + 0, C.data_ptr(), 32, 32, 32, 64,
                                     64, 64, dtype=dt, limit_ms=20, stall_cta=0, stall_fill=0,
                                     stream=torch.cuda.current_stream().cuda_stream, **extra)
        assert e.value.name == "GEMM_ERR_INVALID_VALUE"
    # a CTA index beyond the plan's grid is refused too
    Ah = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_ex_stall_selftest(Ah.data_ptr(), Ah.data_ptr(), C.data_ptr(), 64, 64, 256, 256, 256,
                                 64, dtype=1, limit_ms=20, stall_cta=100000, stall_fill=0,
                                 stream=torch.cuda.current_stream().cuda_stream)
