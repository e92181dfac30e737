"""Split tiles with every piece count the summing code distinguishes.

The last piece of a split tile sums the pieces in piece order, loading two
pieces (four for 16-column swapped chunks) before adding them.  Piece counts
from 2 to 9 put every remainder of those batches through the sum, for the
1-CTA kernel (128- and 64-column tiles) and the swapped kernel (16, 32 and
64 columns), by split-K and by stream-K on fewer tiles than SMs (CTA pairs
cut a tile into at most two pieces; other tests cover them).  Small-integer
inputs: exact.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PLANS = [dict(cta_pair=1, tile_n=128), dict(cta_pair=1, tile_n=64), dict(swap_ab=1, tile_n=16),
         dict(swap_ab=1, tile_n=32), dict(swap_ab=1, tile_n=64)]


@pytest.mark.parametrize("splits", [2, 3, 4, 5, 6, 7, 9])
@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_split_piece_counts(plan, splits):
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 200, 704, 64 * 18 + 8    # 19 k-blocks: splits of 2..9 give 2..7 pieces
    A, B = gu.make_inputs("f16", "small_int", M, N, K, splits)
    desc = g.gemm_plan_describe(0, 1 << 20, 1 << 34, 1 << 40, M, N, K, K, N, N, split_k=splits, **plan)
    assert "split_k=" in desc and "split_k=1 " not in desc, desc
    C = gu.run_gpu("f16", A, B, M, N, K, split_k=splits, **plan)
    assert np.array_equal(C, oracle.gemm("f16", A, B).astype(np.float32)), desc


@pytest.mark.parametrize("plan", [dict(cta_pair=1, tile_n=256), dict(cta_pair=1, tile_n=128),
                                  dict(swap_ab=1, tile_n=16), dict(swap_ab=1, tile_n=64)],
                         ids=lambda p: "-".join(f"{k}{v}" for k, v in p.items()))
def test_stream_k_many_pieces(plan):
    # fewer tiles than SMs, so stream-K cuts every tile into three or more
    # pieces (a dozen for the swapped plans)
    import dense_gemm_tensor_tcgen05_gb300 as g
    M = 40 if plan.get("swap_ab") else 1280
    N, K = 1536, 64 * 40 + 8
    A, B = gu.make_inputs("bf16", "small_int", M, N, K, 1)
    desc = g.gemm_plan_describe(1, 1 << 20, 1 << 34, 1 << 40, M, N, K, K, N, N, stream_k=2, **plan)
    assert "stream_k" in desc and "max_seg=1 " not in desc and "max_seg=2 " not in desc, desc
    C = gu.run_gpu("bf16", A, B, M, N, K, stream_k=2, **plan)
    assert np.array_equal(C, oracle.gemm("bf16", A, B).astype(np.float32)), desc
