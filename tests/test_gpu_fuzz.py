"""Seeded random combinations of the library's options against the oracle.

Every case draws an input type, a ragged shape (several tiles at most), a plan (tile width, CTA
pairs, split-K, stream-K, swap-AB, store mode, generic kernel), transposed
storage, the alpha/beta epilogue, C's type and padded leading dimensions,
keeping to the combinations include/gb300gemm.h documents as valid.  Inputs
are small integers and alpha, beta are small dyadic numbers, so every FP32
result is exact and the library must reproduce the oracle bit for bit (for a
16-bit C: the oracle's own rounding of the exact value).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

N_CASES = 400
C_NAMES = {0: "f32", 1: "f16", 2: "bf16"}
NAN16 = {1: 0x7E00, 2: 0x7FC0}


def _draw(rng):
    dt = rng.choice(["f16", "bf16", "f16", "bf16", "f32", "tf32", "e4m3", "e5m2"])
    M = int(rng.choice([1, 7, 64, 129, 200, 257, 300, 513, 1100]))
    N = int(rng.choice([8, 16, 63, 128, 130, 256, 264, 520, 1040]))
    K = int(rng.choice([1, 16, 64, 65, 127, 200, 320, 700]))
    o = {}
    lowp = dt in ("tf32", "e4m3", "e5m2")
    if lowp:
        o["trans_b"] = 1
    elif dt != "f32" or rng.random() < 0.3:
        o["trans_a"] = int(rng.random() < 0.3)
        o["trans_b"] = int(rng.random() < 0.3)
    if dt in ("f16", "bf16") and rng.random() < 0.1:
        o["generic"] = 1
    elif dt != "f32":
        kind = rng.choice(["plain", "swap", "pair", "auto"])
        if kind == "pair":
            o["cta_pair"] = 2
            o["tile_n"] = int(rng.choice([128, 256]))
            r = rng.random()
            if r < 0.3:
                o["stream_k"] = 2
            elif r < 0.5:
                o["stream_k"] = 3      # tail split
        elif kind == "swap":
            o["swap_ab"] = 1
            o["tile_n"] = 64 if o.get("trans_a") else int(rng.choice([16, 32, 64]))
            if rng.random() < 0.4:
                o["split_k"] = int(rng.choice([2, 3]))
        elif kind == "plain":
            o["cta_pair"] = 1
            o["swap_ab"] = 0
            o["tile_n"] = int(rng.choice([64, 128, 256]))
            r = rng.random()
            if r < 0.3:
                o["split_k"] = int(rng.choice([2, 3, 5]))
            elif r < 0.45:
                o["stream_k"] = 2
            elif r < 0.55:
                o["stream_k"] = 3      # tail split
        if rng.random() < 0.3:
            o["store_mode"] = 1
    else:
        if not (o.get("trans_a") or o.get("trans_b")):
            o["tile_n"] = int(rng.choice([0, 32, 64, 128, 256]))
            r = rng.random()
            if r < 0.3:
                o["split_k"] = int(rng.choice([2, 3]))
            elif r < 0.55:
                o["stream_k"] = int(rng.choice([1, 2]))   # split waves, or the persistent stream-K grid
    if rng.random() < 0.4:
        o["alpha"], o["beta"] = float(rng.choice([0.5, 1.5, -2.0])), float(rng.choice([0.0, 1.0, -0.75]))
    c_dtype = int(rng.choice([0, 0, 1, 2]))
    pad = int(rng.choice([0, 0, 8, 3]))
    return dt, M, N, K, o, c_dtype, pad


def _run(dt, M, N, K, o, c_dtype, pad, seed, entry="ex"):
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    ta, tb = o.get("trans_a", 0), o.get("trans_b", 0)
    A = inputs.make("small_int", dt, M, K, seed, 0)
    B = inputs.make("small_int", dt, K, N, seed, 1)
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    align = {"tf32": 4, "e4m3": 16, "e5m2": 16}.get(dt, 8)
    lda = -(-As.shape[1] // align) * align + (align if pad else 0)
    ldb = -(-Bs.shape[1] // align) * align + (align if pad else 0)
    As, Bs = inputs.padded(As, lda), inputs.padded(Bs, ldb)
    ldc = N + pad
    host = entry == "host"
    if host:   # page-locked host buffers: the library stages them itself
        Ad, Bd = gu.to_device(As, dt).cpu().pin_memory(), gu.to_device(Bs, dt).cpu().pin_memory()
    else:
        Ad, Bd = gu.to_device(As, dt), gu.to_device(Bs, dt)
    dev = "cpu" if host else "cuda"
    guard = 4096
    cin = ((np.arange(M * ldc).reshape(M, ldc) % 7) - 3).astype(np.float64)
    if c_dtype == 0:
        cbuf = torch.full((M * ldc + guard,), float("nan"), dtype=torch.float32, device=dev)
        cbuf[: M * ldc] = torch.from_numpy(cin.astype(np.float32).ravel())
    else:
        cbuf = torch.full((M * ldc + guard,), int(np.uint16(NAN16[c_dtype]).view(np.int16)),
                          dtype=torch.int16, device=dev)
        cbits = oracle.encode16(C_NAMES[c_dtype], cin)
        cbuf[: M * ldc] = torch.from_numpy(cbits.view(np.int16).ravel())
    if host:
        cbuf = cbuf.pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    call = {"ex": g.gemm_ex, "noalloc": g.gemm_ex_noalloc, "host": g.gemm_ex_host}[entry]
    try:
        call(Ad.data_ptr(), Bd.data_ptr(), cbuf.data_ptr(), M, N, K, lda, ldb, ldc,
             dtype=gu.CODE[dt], stream=s, c_dtype=c_dtype, **o)
    except g.GemmError as e:
        # the documented refusal of an explicitly requested plan whose split
        # pieces do not fit the no-alloc scratch; any other error fails
        if entry == "noalloc" and e.name == "GEMM_ERR_INVALID_VALUE" and \
                "exceeds the no-alloc maximum" in str(e):
            return
        raise
    torch.cuda.current_stream().synchronize()
    g.gemm_device_error(s)
    out = cbuf.cpu().numpy()
    if c_dtype:
        out = out.view(np.uint16)
        assert np.all(out[M * ldc:] == NAN16[c_dtype]), "write past the end of C"
    else:
        assert np.all(np.isnan(out[M * ldc:])), "write past the end of C"
    C = out[: M * ldc].reshape(M, ldc)
    R = oracle.gemm_op(dt, ta, tb, As, Bs, M, N, K, lda=lda, ldb=ldb)
    if "alpha" in o:
        # with beta == 0 the library does not read C, so no beta * C term
        # (0 * a negative C would turn a -0 result into +0)
        R = o["alpha"] * R if o["beta"] == 0.0 else o["alpha"] * R + o["beta"] * cin[:, :N]
    if c_dtype == 0:
        assert np.array_equal(C[:, :N], R.astype(np.float32))
        if pad:
            assert np.array_equal(C[:, N:], cin[:, N:].astype(np.float32)), "padding columns changed"
    else:
        # the sign of an exact zero is not part of the contract: compare -0 as +0
        zero = lambda b: np.where((b & 0x7FFF) == 0, 0, b)
        assert np.array_equal(zero(C[:, :N]), zero(oracle.encode16(C_NAMES[c_dtype], R)))
        if pad:
            assert np.array_equal(C[:, N:], cbits[:, N:]), "padding columns changed"


CASES = [_draw(np.random.default_rng(1000 + i)) for i in range(N_CASES)]


@pytest.mark.parametrize("case", range(N_CASES))
def test_fuzz_case(case):
    dt, M, N, K, o, c_dtype, pad = CASES[case]
    _run(dt, M, N, K, o, c_dtype, pad, seed=case)


@pytest.mark.parametrize("case", range(0, N_CASES, 4))
def test_fuzz_case_noalloc(case):
    # the same cases through the entry point that never allocates (its fixed
    # scratch holds every split-K / stream-K workspace these shapes need)
    dt, M, N, K, o, c_dtype, pad = CASES[case]
    _run(dt, M, N, K, o, c_dtype, pad, seed=case, entry="noalloc")


@pytest.mark.parametrize("case", range(1, N_CASES, 4))
def test_fuzz_case_host(case):
    # other cases through the host-buffer entry point (page-locked A, B, C);
    # its staging copies pad the leading dimensions, so the plan options act
    # on panels of the same shapes with other strides
    dt, M, N, K, o, c_dtype, pad = CASES[case]
    _run(dt, M, N, K, o, c_dtype, pad, seed=case, entry="host")
