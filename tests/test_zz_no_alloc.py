"""gemm_ex_noalloc: the entry point for callers that cannot allocate device
memory (applications that own all GPU memory through their own pool, or
latency-critical loops where a cudaMalloc/cudaFree, which can synchronise the
device, is not acceptable).  Its split-K scratch lives in a fixed array inside
the library, so here it is compared with gemm_ex, which allocates its
workspace, on the same inputs and plans, twice in a row -- the second call
reuses the array the first one left behind.  Both run the same plan, whose
split-K sums are taken in a fixed order, so the results must be identical
bit for bit; both are also checked against the oracle.

Collected last on purpose (file name), so a run that stops at the first
failure has run every other test first; it also passes alone in a fresh
process."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [
    # dtype, M, N, K, options (split-K so that the scratch is used)
    ("f16", 8, 4096, 8192, dict(tile_n=16, swap_ab=1, split_k=4)),
    ("bf16", 300, 520, 2000, dict(tile_n=128, swap_ab=0, split_k=3)),
    ("bf16", 64, 1000, 4096, dict(tile_n=64, swap_ab=1, split_k=7)),
    ("f16", 256, 768, 640, dict()),     # the planner's own choice
]


@pytest.fixture(scope="module")
def L():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    from dense_gemm_tensor_tcgen05_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    build.build()
    oracle.build()
    return g.lib()


def _opts(dtype, **kw):
    import dense_gemm_tensor_tcgen05_gb300 as g
    o = g.GemmOptions()
    o.dtype = gu.CODE[dtype]
    o.swap_ab = -1
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def _call(L, fn, dt, Ad, Bd, M, N, K, opts):
    import torch
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    o = _opts(dt, **opts)
    st = getattr(L, fn)(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                        ctypes.byref(o), stream)
    assert st == 0, (fn, st, L.gemm_last_cuda_error())
    assert L.gemm_device_error(stream) == 0
    return C.cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_noalloc_matches_gemm_ex_twice(L, case):
    dt, M, N, K, opts = case
    A, B = gu.make_inputs(dt, "uniform", M, N, K, 77)
    Ad, Bd = gu.to_device(A, dt), gu.to_device(B, dt)
    ref = _call(L, "gemm_ex", dt, Ad, Bd, M, N, K, opts)
    amax, bmax = inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt)
    R = oracle.gemm(dt, A, B)
    assert oracle.compare(ref, R, K, amax, bmax).ok
    for _ in range(2):
        got = _call(L, "gemm_ex_noalloc", dt, Ad, Bd, M, N, K, opts)
        assert np.array_equal(got, ref), "gemm_ex_noalloc differs from gemm_ex on the same plan"
        cmp = oracle.compare(got, R, K, amax, bmax)
        assert cmp.ok, str(cmp)


def test_noalloc_small_integers_exact_twice(L):
    # exact inputs: every summation order gives the oracle's value
    dt, M, N, K, opts = CASES[1]
    A, B = gu.make_inputs(dt, "small_int", M, N, K, 0)
    Ad, Bd = gu.to_device(A, dt), gu.to_device(B, dt)
    want = oracle.gemm(dt, A, B).astype(np.float32)
    for _ in range(2):
        assert np.array_equal(_call(L, "gemm_ex_noalloc", dt, Ad, Bd, M, N, K, opts), want)


def test_noalloc_repeat_calls_allocate_nothing(L):
    # The library counts every device allocation it makes (gemm_alloc_count);
    # other processes or torch's caching allocator do not touch this count.
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    dt, M, N, K, opts = CASES[0]
    A, B = gu.make_inputs(dt, "uniform", M, N, K, 78)
    Ad, Bd = gu.to_device(A, dt), gu.to_device(B, dt)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fresh = torch.cuda.Stream()                   # a stream no call has used yet
    o = _opts(dt, **opts)
    args = (Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N, ctypes.byref(o))
    before = g.gemm_alloc_count()
    for _ in range(3):
        assert L.gemm_ex_noalloc(*args, fresh.cuda_stream) == 0
    torch.cuda.synchronize()
    assert g.gemm_alloc_count() == before
    # the same split-K plan through gemm_ex on that stream allocates its
    # workspace, so the counter does see allocations
    assert L.gemm_ex(*args, fresh.cuda_stream) == 0
    torch.cuda.synchronize()
    assert g.gemm_alloc_count() > before


def test_noalloc_plans_without_pieces_that_do_not_fit(L):
    # At 8192^3 the planner's own plan cuts the 36 tiles after 13 whole waves
    # into two K pieces each (19 MB of pieces); the scratch holds 8 MiB, so
    # this entry point runs whole tiles instead -- the plan gemm_ex runs with
    # stream_k = 1, bit for bit -- and the result still meets the oracle.
    import torch
    M = N = K = 8192
    A, B = gu.make_inputs("bf16", "normal", M, N, K, 1238, sigma=1 / np.sqrt(K))
    Ad, Bd = gu.to_device(A, "bf16"), gu.to_device(B, "bf16")
    got = _call(L, "gemm_ex_noalloc", "bf16", Ad, Bd, M, N, K, dict())
    whole = _call(L, "gemm_ex", "bf16", Ad, Bd, M, N, K, dict(stream_k=1))
    assert np.array_equal(got, whole)
    rows = list(range(0, 16)) + list(range(M - 16, M))
    R = np.concatenate([oracle.gemm_rows("bf16", A, B, 0, 16), oracle.gemm_rows("bf16", A, B, M - 16, M)])
    cmp = oracle.compare(got[rows], R, K, inputs.bits_abs_max(A, "bf16"), inputs.bits_abs_max(B, "bf16"))
    assert cmp.ok, str(cmp)


def test_noalloc_rejects_scratch_beyond_maximum(L):
    import torch
    M = N = K = 2048                               # 128 tiles x 8 slices x 128 KiB >> 8 MiB
    Ad = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    o = _opts("f16", tile_n=256, swap_ab=0, split_k=8)
    st = L.gemm_ex_noalloc(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                           ctypes.byref(o), torch.cuda.current_stream().cuda_stream)
    assert st == 1
    assert b"exceeds the no-alloc maximum" in L.gemm_last_cuda_error()
