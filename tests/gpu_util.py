"""Helpers for the GPU parity tests: run the CUDA library through its C ABI on
seeded inputs and compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from dense_gemm_tensor_tcgen05_gb300 import inputs

CODE = {"f16": 0, "bf16": 1, "f32": 2, "tf32": 3, "e4m3": 4, "e5m2": 5}


def torch_dtype(dt):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "tf32": torch.float32, "e4m3": torch.uint8, "e5m2": torch.uint8}[dt]


def to_device(bits: np.ndarray, dt: str, offset_elems: int = 0):
    """Element bits -> a CUDA tensor of the element type.  offset_elems > 0
    returns a view that starts that many elements into a larger buffer (to
    make misaligned pointers)."""
    import torch
    flat = np.ascontiguousarray(bits).reshape(-1)
    if dt in ("f32", "tf32"):
        host = torch.from_numpy(flat.astype(np.float32, copy=False).view(np.float32))
    elif dt in ("e4m3", "e5m2"):
        host = torch.from_numpy(flat.view(np.uint8))
    else:
        host = torch.from_numpy(flat.view(np.int16)).view(torch_dtype(dt))
    if offset_elems:
        buf = torch.zeros(host.numel() + offset_elems, dtype=host.dtype, device="cuda")
        buf[offset_elems:] = host.cuda()
        return buf[offset_elems:]
    return host.cuda()


def run_gpu(dt, A_bits, B_bits, M, N, K, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
            stream=None, c_init=None, **opts):
    """C (M x N float32 numpy) from the library.  C starts as NaN everywhere,
    so an unwritten element fails any comparison, and padding columns of C
    (ldc > N) must still be NaN afterwards."""
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    lda = A_bits.shape[1] if lda is None else lda
    ldb = B_bits.shape[1] if ldb is None else ldb
    ldc = N if ldc is None else ldc
    Ad = to_device(A_bits, dt, offsets[0])
    Bd = to_device(B_bits, dt, offsets[1])
    rows = max(M, 1)
    guard = 4096   # NaN floats after C: a write past C's last row shows up here
    cbuf = torch.full((rows * ldc + offsets[2] + guard,), float("nan"), dtype=torch.float32,
                      device="cuda")
    Cd = cbuf[offsets[2]:]
    if c_init is not None:   # C's old values (M x ldc), for C = alpha AB + beta C
        Cd[: M * ldc].copy_(torch.from_numpy(np.ascontiguousarray(c_init, dtype=np.float32).ravel()))
    st = stream if stream is not None else torch.cuda.current_stream()
    sh = st.cuda_stream
    args = (Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, lda, ldb, ldc)
    torch.cuda.synchronize()
    if opts:
        g.gemm_ex(*args, dtype=CODE[dt], stream=sh, **opts)
    else:
        # tf32/e4m3/e5m2: the _bt entry points (B passed as its N x K transpose)
        {"f16": g.gemm_f16f32, "bf16": g.gemm_bf16f32, "f32": g.sgemm_f32,
         "tf32": g.gemm_tf32f32_bt, "e4m3": g.gemm_e4m3f32_bt,
         "e5m2": g.gemm_e5m2f32_bt}[dt](*args, stream=sh)
    g.gemm_device_error(sh)
    tail = Cd[rows * ldc:].cpu().numpy()
    assert np.all(np.isnan(tail)), "kernel wrote past the end of C"
    if offsets[2]:
        assert torch.isnan(cbuf[:offsets[2]]).all().item(), "kernel wrote before the start of C"
    C = Cd[: rows * ldc].reshape(rows, ldc).cpu().numpy()[:M]
    if ldc > N and M > 0:
        if c_init is None:
            assert np.all(np.isnan(C[:, N:])), "kernel wrote into C's padding columns"
        else:
            assert np.array_equal(C[:, N:], c_init[:, N:], equal_nan=True), \
                "kernel wrote into C's padding columns"
    return C[:, :N]


def make_inputs(dt, dist, M, N, K, seed, sigma=1.0):
    A = inputs.make(dist, dt, M, K, seed, 0, sigma)
    B = inputs.make(dist, dt, K, N, seed, 1, sigma)
    return A, B


def round_up(x, a):
    return (x + a - 1) // a * a


def check_full(dt, dist, M, N, K, seed=0, sigma=1.0, exact=False, pad=(0, 0, 0), align_ld=0,
               **opts):
    """Whole-matrix parity with the oracle.  align_ld > 0 rounds lda and ldb up
    to that many elements (and ldc to 4), poisoning the padding, so that odd
    shapes still take the TMA / vectorised paths."""
    A, B = make_inputs(dt, dist, M, N, K, seed, sigma)
    if align_ld:
        pad = (round_up(K, align_ld) - K, round_up(N, align_ld) - N, round_up(N, 4) - N)
    lda, ldb, ldc = K + pad[0], N + pad[1], N + pad[2]
    Ap = inputs.padded(A, lda) if pad[0] else A
    Bp = inputs.padded(B, ldb) if pad[1] else B
    C = run_gpu(dt, Ap, Bp, M, N, K, lda, ldb, ldc, **opts)
    R = oracle.gemm(dt, A, B)
    cmp = oracle.compare(C, R, K, inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt))
    assert cmp.ok, f"{dt} {dist} {M}x{N}x{K} {opts}: {cmp}"
    if exact:
        assert cmp.exact, f"{dt} {dist} {M}x{N}x{K} {opts}: not bit-exact: {cmp}"
    return cmp


def sample_rows(M, band=16, seed=0):
    """A few row bands: the first, one in the middle, the last (ragged tail)."""
    bands = [(0, min(band, M))]
    mid = (M // 2) // 8 * 8
    if mid + band < M:
        bands.append((mid, mid + band))
    if M > band:
        bands.append((M - band, M))
    return bands


def check_sampled(dt, A, B, C, M, N, K, n_entries=4096, seed=0, band=16):
    """Parity on samples the oracle can afford at full size: whole row bands
    (first, middle, last) and random single entries, including the last
    columns."""
    rng = np.random.default_rng(seed)
    got, want = [], []
    for (r0, r1) in sample_rows(M, band):
        R = oracle.gemm_rows(dt, A, B, r0, r1, M=M, N=N, K=K)
        got.append(C[r0:r1].ravel())
        want.append(R.ravel())
    rows = rng.integers(0, M, size=n_entries)
    cols = rng.integers(0, N, size=n_entries)
    cols[: min(256, n_entries)] = N - 1 - (np.arange(min(256, n_entries)) % min(N, 64))
    ent = oracle.gemm_entries(dt, A, B, rows, cols, M=M, N=N, K=K)
    got.append(C[rows, cols])
    want.append(ent)
    cmp = oracle.compare(np.concatenate(got), np.concatenate(want), K,
                         inputs.bits_abs_max(A, dt), inputs.bits_abs_max(B, dt))
    return cmp
