"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each check takes the oracle's product routine as ``gemm(dtype, A_bits,
B_bits, M, N, K, lda, ldb) -> float64 C`` and returns a list of failure
strings (empty when it holds), so the same checks run against the real
oracle and against deliberately broken copies of it (the mutation test).

What pins the oracle, and why each would catch a plausible mistake:
  * a worked 2x3 by 3x4 integer product, hand-computed from the definition
    (catches transposed operands, swapped loop bounds, wrong strides);
  * all-ones inputs give C = K exactly (catches a dropped or extra term);
  * identity on either side returns the other operand exactly (catches index
    mix-ups that keep sums but move them);
  * a rank-one integer product gives C = K u_i v_j (catches row/column swaps
    on rectangles);
  * the small-integer pattern of "matmul_registers.cu" against an exact
    integer brute force in Python (catches sign errors and index errors that
    happen to preserve the other pins);
  * random rationals against exact Fraction arithmetic (catches wrong
    decoding of fractional values, subnormals included);
  * padded leading dimensions with poison in the padding (catches reading
    past K or N).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from dense_gemm_tensor_tcgen05_gb300 import inputs


def _bits(dist, dtype, rows, cols, seed=0, mid=0, sigma=1.0):
    return inputs.make(dist, dtype, rows, cols, seed, mid, sigma)


def _exact_value(bits: np.ndarray, dtype: str):
    """Exact rational value of each element, via numpy's own IEEE types
    (float16 / float32 views), which are independent of the oracle's
    decoders.  BF16 is the upper half of a float32."""
    if dtype == "f16":
        vals = bits.view(np.float16).astype(np.float64)
    elif dtype == "bf16":
        vals = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    else:
        vals = bits.astype(np.float64)
    return [[Fraction(float(v)) for v in row] for row in vals]


def check_worked_example(gemm) -> list[str]:
    A = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float32)
    B = np.array([[7, 8, 9, 10], [11, 12, 13, 14], [15, 16, 17, 18]], dtype=np.float32)
    want = np.array([[74, 80, 86, 92], [173, 188, 203, 218]], dtype=np.float64)
    fails = []
    for dt in ("f16", "bf16", "f32"):
        C = gemm(dt, inputs.to_bits(A, dt), inputs.to_bits(B, dt), 2, 4, 3, 3, 4)
        if not np.array_equal(C, want):
            fails.append(f"worked example {dt}: got {C.tolist()}")
    return fails


def check_ones(gemm) -> list[str]:
    fails = []
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (17, 9, 300), (4, 4, 4096)]:
        for dt in ("f16", "bf16", "f32"):
            A = _bits("ones", dt, M, K)
            B = _bits("ones", dt, K, N)
            C = gemm(dt, A, B, M, N, K, K, N)
            if not np.all(C == K):
                fails.append(f"ones {dt} {M}x{N}x{K}")
    return fails


def check_identity(gemm) -> list[str]:
    fails = []
    for dt in ("f16", "bf16", "f32"):
        for (M, N) in [(5, 7), (16, 3), (33, 64)]:
            X = _bits("uniform", dt, M, N, seed=3, mid=1)
            Xv = _exact_value(X, dt)
            want = np.array([[float(v) for v in row] for row in Xv])
            # I (M x M) @ X (M x N) == X
            I = _bits("identity", dt, M, M)
            C = gemm(dt, I, X, M, N, M, M, N)
            if not np.array_equal(C, want):
                fails.append(f"I@X {dt} {M}x{N}")
            # X (M x N) @ I (N x N) == X
            I = _bits("identity", dt, N, N)
            C = gemm(dt, X, I, M, N, N, N, N)
            if not np.array_equal(C, want):
                fails.append(f"X@I {dt} {M}x{N}")
    return fails


def check_rank1(gemm) -> list[str]:
    fails = []
    for dt in ("f16", "bf16", "f32"):
        for (M, N, K) in [(7, 11, 13), (40, 3, 129), (2, 65, 64)]:
            A = _bits("rank1", dt, M, K, mid=0)
            B = _bits("rank1", dt, K, N, mid=1)
            u = (np.arange(M) % 5 - 2).astype(np.float64)
            v = (np.arange(N) % 3 - 1).astype(np.float64)
            want = K * np.outer(u, v)
            C = gemm(dt, A, B, M, N, K, K, N)
            if not np.array_equal(C, want):
                fails.append(f"rank1 {dt} {M}x{N}x{K}")
    return fails


def small_int_exact(M: int, N: int, K: int) -> np.ndarray:
    """Exact integer product of the small-integer pattern, by plain Python
    integers (no floating point anywhere)."""
    a = [[((r + 2 * c) % 7) - 3 for c in range(K)] for r in range(M)]
    b = [[((3 * r + c) % 5) - 2 for c in range(N)] for r in range(K)]
    out = np.zeros((M, N), dtype=np.float64)
    for i in range(M):
        for j in range(N):
            s = 0
            for p in range(K):
                s += a[i][p] * b[p][j]
            out[i, j] = s
    return out


def check_small_int(gemm) -> list[str]:
    fails = []
    for (M, N, K) in [(1, 1, 1), (6, 10, 7), (13, 5, 35), (9, 31, 70)]:
        want = small_int_exact(M, N, K)
        for dt in ("f16", "bf16", "f32"):
            A = _bits("small_int", dt, M, K, mid=0)
            B = _bits("small_int", dt, K, N, mid=1)
            C = gemm(dt, A, B, M, N, K, K, N)
            if not np.array_equal(C, want):
                fails.append(f"small_int {dt} {M}x{N}x{K}")
    return fails


def check_fraction_bruteforce(gemm) -> list[str]:
    """Random inputs against exact rational sums.  The oracle's double sum
    must sit within K * 2^-52 * sum|a_k b_k| of the exact value (the
    standard bound for recursive summation in double, products exact)."""
    fails = []
    rng_shapes = [(1, 1, 1), (2, 3, 4), (5, 1, 9), (3, 7, 2), (4, 4, 16)]
    for si, (M, N, K) in enumerate(rng_shapes):
        for dt, dist in (("f16", "uniform"), ("bf16", "normal"), ("f32", "uniform")):
            A = _bits(dist, dt, M, K, seed=100 + si, mid=0)
            B = _bits(dist, dt, K, N, seed=100 + si, mid=1)
            Av, Bv = _exact_value(A, dt), _exact_value(B, dt)
            C = gemm(dt, A, B, M, N, K, K, N)
            if not np.all(np.isfinite(C)):
                fails.append(f"fraction {dt} {M}x{N}x{K}: non-finite output")
                continue
            for i in range(M):
                for j in range(N):
                    terms = [Av[i][p] * Bv[p][j] for p in range(K)]
                    exact = sum(terms, Fraction(0))
                    scale = sum((abs(t) for t in terms), Fraction(0))
                    err = abs(Fraction(float(C[i, j])) - exact)
                    if err > Fraction(K, 2 ** 52) * scale:
                        fails.append(f"fraction {dt} {M}x{N}x{K} at ({i},{j}): "
                                     f"{float(C[i, j])!r} vs {float(exact)!r}")
    return fails


def check_subnormals(gemm) -> list[str]:
    """FP16 subnormal inputs (below 2^-14) decode exactly: 1 x 2^-24 summed
    K times is K x 2^-24 exactly."""
    fails = []
    K = 10
    A = np.full((1, K), 0x0001, dtype=np.uint16)   # 2^-24, smallest FP16 subnormal
    B = np.full((K, 1), 0x3C00, dtype=np.uint16)   # 1.0
    C = gemm("f16", A, B, 1, 1, K, K, 1)
    if C[0, 0] != K * 2.0 ** -24:
        fails.append(f"f16 subnormal: {C[0, 0]!r}")
    A = np.full((1, K), 0x0001, dtype=np.uint16)   # 2^-133, smallest BF16 subnormal
    B = np.full((K, 1), 0x3F80, dtype=np.uint16)   # 1.0
    C = gemm("bf16", A, B, 1, 1, K, K, 1)
    if C[0, 0] != K * 2.0 ** -133:
        fails.append(f"bf16 subnormal: {C[0, 0]!r}")
    return fails


def check_leading_dims(gemm) -> list[str]:
    fails = []
    for dt in ("f16", "bf16", "f32"):
        M, N, K = 6, 5, 9
        A = _bits("small_int", dt, M, K, mid=0)
        B = _bits("small_int", dt, K, N, mid=1)
        want = small_int_exact(M, N, K)
        Ap = inputs.padded(A, K + 7)
        Bp = inputs.padded(B, N + 3)
        C = gemm(dt, Ap, Bp, M, N, K, K + 7, N + 3)
        if not np.array_equal(C, want):
            fails.append(f"leading dims {dt}")
    return fails


ALL_CHECKS = [check_worked_example, check_ones, check_identity, check_rank1,
              check_small_int, check_fraction_bruteforce, check_subnormals,
              check_leading_dims]


def run_all(gemm) -> list[str]:
    fails = []
    for chk in ALL_CHECKS:
        fails += chk(gemm)
    return fails
