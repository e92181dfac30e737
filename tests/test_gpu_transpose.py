"""GPU parity for C = op(A) x op(B) with A and/or B stored transposed,
against the oracle's op form, on every kernel path."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PLANS = {
    "tc_128x256": ("bf16", dict(cta_pair=1, tile_n=256)),
    "tc_128x128_plain": ("f16", dict(cta_pair=1, tile_n=128, store_mode=1)),
    "tc_128x64": ("f16", dict(cta_pair=1, tile_n=64)),
    "tc_swap64": ("bf16", dict(tile_n=64, swap_ab=1)),
    "tc_split_k": ("f16", dict(cta_pair=1, tile_n=128, split_k=3)),
    "tc_stream_k": ("bf16", dict(cta_pair=1, tile_n=128, stream_k=2)),
    "tc_pair256": ("bf16", dict(cta_pair=2, tile_n=256)),
    "tc_pair128": ("f16", dict(cta_pair=2, tile_n=128)),
    "generic_f16": ("f16", dict(generic=1)),
    "f32": ("f32", dict()),
}
TRANS = [(0, 0), (0, 1), (1, 0), (1, 1)]


def _storage(bits, trans, pad):
    """Stored form of an operand: itself, or its transpose; rows padded."""
    st = np.ascontiguousarray(bits.T) if trans else bits
    ld = st.shape[1] + pad
    return (inputs.padded(st, ld) if pad else st), ld


def _check(dt, opts, ta, tb, M, N, K, dist, exact, pad=8, seed=0):
    opA = inputs.make(dist, dt, M, K, seed, 0)
    opB = inputs.make(dist, dt, K, N, seed, 1)
    As, lda = _storage(opA, ta, pad)
    Bs, ldb = _storage(opB, tb, pad)
    C = gu.run_gpu(dt, As, Bs, M, N, K, lda=lda, ldb=ldb, trans_a=ta, trans_b=tb, **opts)
    R = oracle.gemm_op(dt, ta, tb, As, Bs, M, N, K, lda=lda, ldb=ldb)
    cmp = oracle.compare(C, R, K, inputs.bits_abs_max(opA, dt), inputs.bits_abs_max(opB, dt))
    assert cmp.ok, f"{dt} ta={ta} tb={tb} {M}x{N}x{K} {opts}: {cmp}"
    if exact:
        assert cmp.exact, str(cmp)


@pytest.mark.parametrize("name", sorted(PLANS))
@pytest.mark.parametrize("ta,tb", TRANS, ids=lambda t: str(t))
def test_transposed_operands_exact(name, ta, tb):
    dt, opts = PLANS[name]
    _check(dt, opts, ta, tb, 300, 520, 700, "small_int", exact=True)


@pytest.mark.parametrize("name", sorted(PLANS))
@pytest.mark.parametrize("ta,tb", TRANS, ids=lambda t: str(t))
def test_transposed_operands_random_ragged(name, ta, tb):
    dt, opts = PLANS[name]
    _check(dt, opts, ta, tb, 257, 130, 72, "uniform", exact=False, seed=3)


@pytest.mark.parametrize("ta,tb", TRANS, ids=lambda t: str(t))
def test_transposed_default_plans(ta, tb):
    for dt, (M, N, K) in (("bf16", (1024, 1536, 512)), ("f16", (8, 1024, 2048)),
                          ("f16", (2048, 64, 256))):
        _check(dt, {}, ta, tb, M, N, K, "small_int", exact=True, pad=0)


def test_matmul_takes_transposed_views():
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    M, N, K = 300, 200, 260
    opA = inputs.make("uniform", "bf16", M, K, 5, 0)
    opB = inputs.make("uniform", "bf16", K, N, 5, 1)
    At = torch.from_numpy(np.ascontiguousarray(opA.T).view(np.int16)).view(torch.bfloat16).cuda()
    Bt = torch.from_numpy(np.ascontiguousarray(opB.T).view(np.int16)).view(torch.bfloat16).cuda()
    C = g.matmul(At.t(), Bt.t())            # column-major views of op(A), op(B)
    R = oracle.gemm_op("bf16", True, True, np.ascontiguousarray(opA.T), np.ascontiguousarray(opB.T),
                       M, N, K)
    cmp = oracle.compare(C.cpu().numpy(), R, K, inputs.bits_abs_max(opA, "bf16"),
                         inputs.bits_abs_max(opB, "bf16"))
    assert cmp.ok, str(cmp)
