"""Library calls captured in a CUDA graph and replayed.

Every launch goes through the stream it is given and the host-side plan is
fixed at capture time, so a captured call replays the same kernels.  A plan
that needs a split-K or stream-K workspace allocates it on its first call,
so each plan runs once before capture (allocation is not allowed while a
stream is being captured); the workspace then stays put and is reused."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PLANS = [
    ("bf16", 512, 768, 640, dict(cta_pair=2)),
    ("f16", 8, 2048, 4096, dict(tile_n=16, swap_ab=1, split_k=4)),
    ("bf16", 300, 520, 700, dict(cta_pair=1, tile_n=128, stream_k=2)),
    ("f32", 200, 136, 72, dict()),
    ("bf16", 256, 512, 384, dict(c_dtype=2)),
]


def test_graph_capture_and_replay():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    st = torch.cuda.Stream()
    calls, expect = [], []
    for n, (dt, M, N, K, o) in enumerate(PLANS):
        A = inputs.make("small_int", dt, M, K, n, 0)
        B = inputs.make("small_int", dt, K, N, n, 1)
        Ad, Bd = gu.to_device(A, dt), gu.to_device(B, dt)
        c16 = o.get("c_dtype", 0)
        C = torch.zeros((M, N), dtype=torch.int16 if c16 else torch.float32, device="cuda")
        args = (Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K, K, N, N)
        calls.append((args, dt, o, (Ad, Bd, C)))
        R = oracle.gemm(dt, A, B)
        expect.append(oracle.encode16("bf16", R) if c16 else R.astype(np.float32))
    # one call of each plan outside capture: any workspace is allocated here
    with torch.cuda.stream(st):
        for args, dt, o, _ in calls:
            g.gemm_ex(*args, dtype=gu.CODE[dt], stream=st.cuda_stream, **o)
    st.synchronize()
    for _, _, _, (_, _, C) in calls:
        C.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    before = g.gemm_launch_count()
    with torch.cuda.graph(graph, stream=st):
        for args, dt, o, _ in calls:
            g.gemm_ex(*args, dtype=gu.CODE[dt], stream=st.cuda_stream, **o)
    launched = g.gemm_launch_count() - before
    assert launched >= len(PLANS)
    for rep in range(3):
        for _, _, _, (_, _, C) in calls:
            C.zero_()
        graph.replay()
        torch.cuda.synchronize()
        g.gemm_device_error(st.cuda_stream)
        for (args, dt, o, (_, _, C)), want in zip(calls, expect):
            got = C.cpu().numpy()
            if o.get("c_dtype"):
                got = got.view(np.uint16)
            assert np.array_equal(got, want), (dt, args[3:6], o, rep)
