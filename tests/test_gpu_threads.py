"""Several host threads calling the library at once, each on its own stream.

The header promises that calls from several threads are safe and that each
stream has its own split-K / stream-K workspace.  Four threads each issue a
mixed sequence of plans (split-K, stream-K, swap-AB, CTA pairs, SGEMM, 16-bit
C) on shared inputs and their own outputs; every result is compared with the
oracle afterwards (small-integer inputs: bit-exact)."""
from __future__ import annotations

import threading

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PLANS = [
    ("f16", 8, 2048, 4096, dict(tile_n=16, swap_ab=1, split_k=4)),
    ("bf16", 300, 520, 700, dict(cta_pair=1, tile_n=128, split_k=3)),
    ("bf16", 600, 1040, 640, dict(cta_pair=1, tile_n=128, stream_k=2)),
    ("bf16", 512, 768, 640, dict(cta_pair=2)),
    ("f32", 257, 130, 200, dict(tile_n=64, split_k=3)),
    ("f16", 300, 520, 700, dict(c_dtype=2)),
]
THREADS = 4
ROUNDS = 6


def test_threads_on_their_own_streams():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    data = []
    for n, (dt, M, N, K, o) in enumerate(PLANS):
        A = inputs.make("small_int", dt, M, K, n, 0)
        B = inputs.make("small_int", dt, K, N, n, 1)
        R = oracle.gemm(dt, A, B)
        want = oracle.encode16("bf16", R) if o.get("c_dtype") else R.astype(np.float32)
        data.append((gu.to_device(A, dt), gu.to_device(B, dt), want))
    outs = [[None] * len(PLANS) for _ in range(THREADS)]
    errors = []

    def worker(t):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                Cs = []
                for (dt, M, N, K, o) in PLANS:
                    dtype = torch.int16 if o.get("c_dtype") else torch.float32
                    Cs.append(torch.zeros((M, N), dtype=dtype, device="cuda"))
                for r in range(ROUNDS):
                    # a different order per thread and round
                    order = [(t + r + i) % len(PLANS) for i in range(len(PLANS))]
                    for i in order:
                        dt, M, N, K, o = PLANS[i]
                        Ad, Bd, _ = data[i]
                        g.gemm_ex(Ad.data_ptr(), Bd.data_ptr(), Cs[i].data_ptr(), M, N, K, K, N, N,
                                  dtype=gu.CODE[dt], stream=st.cuda_stream, **o)
                g.gemm_device_error(st.cuda_stream)
                outs[t] = [C.cpu().numpy() for C in Cs]
        except Exception as e:  # reported in the main thread
            errors.append((t, repr(e)))

    torch.cuda.synchronize()
    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(THREADS):
        for i, (dt, M, N, K, o) in enumerate(PLANS):
            got = outs[t][i]
            if o.get("c_dtype"):
                got = got.view(np.uint16)
            assert np.array_equal(got, data[i][2]), (t, dt, M, N, K, o)
