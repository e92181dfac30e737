"""CPU oracle for the dense GEMM C = A x B (row-major).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``dense_gemm_tensor_tcgen05_gb300``) never imports it and it never imports
the product library; the two share no code.  The only module both sides take
inputs from is the seeded input generator, which holds none of the method's
arithmetic.

The arithmetic lives in ``gemm_oracle.c`` (plain C, double accumulation, own
FP16 / BF16 / FP32 bit decoders), built with gcc by :func:`build`.  This file
wraps it with ctypes and adds the tolerance check.

Definition followed: C[i][j] = sum_k A[i][k] B[k][j] for A of M x K, B of
K x N ("Tensor cores and matrix operations", section "Traditional Approach:
Element-by-Element"), on the same rounded 16-bit values the GPU reads
("04-wmma-matmul" code example, its CPU reference), summed in double
("matmul_registers.cu", its CPU reference).

Tolerance (the acceptance rule for floating-point results; the pages print
only informal error measures, a max relative error with a 1e-3 floor in
"04-wmma-matmul" and a 1e-5 relative gate in "matmul_registers.cu", which are
replaced by this rule):

    max |C - C_ref| <= 1e-3 * sqrt(K) * max|A| * max|B|
    ||C - C_ref||_F / ||C_ref||_F <= 1e-4

Inputs whose products and partial sums are small integers are exact in every
summation order, so for them the check is bit-exact equality with the oracle
rounded to FP32 ("matmul_registers.cu", the argument next to its tolerance).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

__all__ = [
    "F16", "BF16", "F32", "build", "lib", "decode", "gemm", "gemm_rows", "gemm_general", "gemm_op",
    "general_bounds", "tf32_bound", "tf32_cut", "E4M3", "E5M2", "encode16", "round16",
    "half_ulp16",
    "gemm_entries", "compare", "Comparison", "ABS_COEF", "REL_FROB",
]

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
_DTYPE_NAMES = {"f16": F16, "fp16": F16, "float16": F16,
                "bf16": BF16, "bfloat16": BF16,
                "f32": F32, "fp32": F32, "float32": F32, "tf32": F32,
                "e4m3": E4M3, "e5m2": E5M2}

ABS_COEF = 1e-3
REL_FROB = 1e-4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgemm_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c with gcc into oracle/_build/. Returns the path.

    ``-ffp-contract=off`` keeps every product rounded to double before it is
    added, so the result does not depend on whether the host has fused
    multiply-add (x86 and Arm then agree bit for bit)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
            L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_f32_to_f64.argtypes = [ctypes.c_uint32]
            L.oracle_f32_to_f64.restype = ctypes.c_double
            L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_f64.restype = ctypes.c_double
            L.oracle_e5m2_to_f64.argtypes = [ctypes.c_uint8]
            L.oracle_e5m2_to_f64.restype = ctypes.c_double
            L.oracle_decode.argtypes = [ctypes.c_int, vp, dp, i64]
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_encode16.argtypes = [ctypes.c_int, dp, vp, i64]
            L.oracle_encode16.restype = ctypes.c_int
            L.oracle_gemm_rows.argtypes = [ctypes.c_int, vp, vp, dp, i64, i64, i64,
                                           i64, i64, i64, i64, i64, ctypes.c_int]
            L.oracle_gemm_rows.restype = ctypes.c_int
            L.oracle_gemm.argtypes = [ctypes.c_int, vp, vp, dp, i64, i64, i64,
                                      i64, i64, i64, ctypes.c_int]
            L.oracle_gemm.restype = ctypes.c_int
            L.oracle_gemm_entries.argtypes = [ctypes.c_int, vp, vp, i64, i64, i64, i64, i64,
                                              i64, ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int64), dp]
            L.oracle_gemm_entries.restype = ctypes.c_int
            L.oracle_gemm_general.argtypes = [ctypes.c_int, vp, vp, ctypes.POINTER(ctypes.c_float),
                                              ctypes.c_double, ctypes.c_double, dp, i64, i64, i64,
                                              i64, i64, i64, ctypes.c_int]
            L.oracle_gemm_general.restype = ctypes.c_int
            L.oracle_gemm_op.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, dp,
                                         i64, i64, i64, i64, i64, i64, ctypes.c_int]
            L.oracle_gemm_op.restype = ctypes.c_int
            _lib = L
    return _lib


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        if dtype not in (F16, BF16, F32, E4M3, E5M2):
            raise ValueError(f"bad dtype code {dtype}")
        return dtype
    try:
        return _DTYPE_NAMES[str(dtype).lower()]
    except KeyError:
        raise ValueError(f"unknown dtype {dtype!r}") from None


def _bits(x: np.ndarray, code: int) -> np.ndarray:
    """Raw element bits as a C-contiguous array (uint8 for 8-bit types,
    uint16 for 16-bit types, uint32 for FP32).  FP32 may be given as float32
    and is reinterpreted."""
    x = np.asarray(x)
    want = np.uint8 if code in (E4M3, E5M2) else np.uint16 if code in (F16, BF16) else np.uint32
    if x.dtype.itemsize != np.dtype(want).itemsize:
        raise TypeError(f"expected {np.dtype(want).itemsize}-byte elements, got {x.dtype}")
    return np.ascontiguousarray(x).view(want)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def decode(dtype, bits) -> np.ndarray:
    """Values (float64) of raw FP16 / BF16 / FP32 element bits, by the oracle's
    own decoders.  Keeps the input's shape."""
    code = _dtype_code(dtype)
    b = _bits(bits, code)
    out = np.empty(b.shape, dtype=np.float64)
    if lib().oracle_decode(code, _ptr(b), _dptr(out), b.size) != 0:
        raise ValueError("oracle_decode failed")
    return out


def encode16(dtype, values) -> np.ndarray:
    """FP16 or BF16 bits (uint16) of float64 values, rounded to nearest, ties
    to even, by the oracle's own encoder.  Keeps the input's shape."""
    code = _dtype_code(dtype)
    if code not in (F16, BF16):
        raise ValueError("encode16 takes f16 or bf16")
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    if lib().oracle_encode16(code, _dptr(v), _ptr(out), v.size) != 0:
        raise ValueError("oracle_encode16 failed")
    return out


def round16(dtype, values) -> np.ndarray:
    """float64 values rounded to FP16 or BF16 (nearest, ties to even) and
    decoded back: what a 16-bit C holds for an exactly known result."""
    return decode(dtype, encode16(dtype, values))


def half_ulp16(dtype, values) -> np.ndarray:
    """Half the spacing of FP16 / BF16 numbers at |values|: the largest error
    of rounding a value of that magnitude to the format (subnormal spacing
    below the smallest normal)."""
    code = _dtype_code(dtype)
    p, emin = (10, -14) if code == F16 else (7, -126)
    a = np.abs(np.asarray(values, dtype=np.float64))
    _, E = np.frexp(a)                   # a = m * 2^E, m in [0.5, 1): exponent E - 1
    e = np.where(a > 0, E - 1, emin)
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - p - 1).astype(np.int64))


def _shape_args(A, B, M, N, K, lda, ldb):
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("A and B must be 2-D arrays of element bits")
    M = A.shape[0] if M is None else M
    lda = A.shape[1] if lda is None else lda
    K = lda if K is None else K
    ldb = B.shape[1] if ldb is None else ldb
    N = ldb if N is None else N
    if A.size < (M - 1) * lda + K if M > 0 else False:
        raise ValueError("A too small for M, K, lda")
    if B.size < (K - 1) * ldb + N if K > 0 else False:
        raise ValueError("B too small for K, N, ldb")
    return M, N, K, lda, ldb


def gemm(dtype, A, B, M=None, N=None, K=None, lda=None, ldb=None,
         nthreads: int | None = None) -> np.ndarray:
    """The full product C (M x N, float64) of raw-bit inputs A (M rows of
    stride lda) and B (K rows of stride ldb).  Shapes default to the arrays'
    own: A is (M, lda), B is (K, ldb), with K = lda and N = ldb unless given."""
    code = _dtype_code(dtype)
    A, B = _bits(A, code), _bits(B, code)
    M, N, K, lda, ldb = _shape_args(A, B, M, N, K, lda, ldb)
    C = np.empty((M, N), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().oracle_gemm(code, _ptr(A), _ptr(B), _dptr(C), M, N, K, lda, ldb, N, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    return C


def gemm_general(dtype, A, B, C_in, alpha: float, beta: float, M=None, N=None, K=None,
                 lda=None, ldb=None, ldc_in=None, nthreads: int | None = None) -> np.ndarray:
    """alpha * (A x B) + beta * C_in (float64, M x N).  C_in is a float32
    array of M rows with row stride ldc_in (its own width by default); it is
    not read when beta == 0.  alpha and beta should be the FP32 values the
    kernels use (they are widened to double here)."""
    code = _dtype_code(dtype)
    A, B = _bits(A, code), _bits(B, code)
    M, N, K, lda, ldb = _shape_args(A, B, M, N, K, lda, ldb)
    Ci = np.ascontiguousarray(C_in, dtype=np.float32)
    ldc_in = Ci.shape[1] if ldc_in is None else ldc_in
    out = np.empty((M, N), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().oracle_gemm_general(code, _ptr(A), _ptr(B),
                                   Ci.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                   float(alpha), float(beta), _dptr(out), M, N, K, lda, ldb,
                                   ldc_in, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_general failed ({rc})")
    return out


def gemm_op(dtype, trans_a: bool, trans_b: bool, A, B, M: int, N: int, K: int,
            lda: int | None = None, ldb: int | None = None,
            nthreads: int | None = None) -> np.ndarray:
    """op(A) x op(B) (float64, M x N).  A holds op(A) row-major (M x K) when
    trans_a is false and its transpose row-major (K x M) when true; B
    likewise (K x N, or N x K when trans_b).  Leading dimensions default to
    the arrays' widths."""
    code = _dtype_code(dtype)
    A, B = _bits(A, code), _bits(B, code)
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    C = np.empty((M, N), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().oracle_gemm_op(code, int(bool(trans_a)), int(bool(trans_b)), _ptr(A), _ptr(B),
                              _dptr(C), M, N, K, lda, ldb, N, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_op failed ({rc})")
    return C


def tf32_bound(abs_sums: np.ndarray) -> np.ndarray:
    """Per-element tolerance for TF32 tensor-core products of FP32 inputs:
    TF32 keeps 10 fraction bits, so each input carries a relative error below
    2^-10 and each product below 2^-9 (whether the hardware rounds or drops
    the low 13 bits); FP32 accumulation adds about 2^-20 of the sum of
    magnitudes.  abs_sums[i, j] = sum_k |A[i][k]| |B[k][j]| (the oracle's
    product of the absolute values)."""
    return (2.0 ** -9 + 2.0 ** -20) * np.asarray(abs_sums, dtype=np.float64)


def tf32_cut(x, mode: str) -> np.ndarray:
    """FP32 values cut to TF32 (a float32 array of the same shape).

    TF32 keeps FP32's sign and 8-bit exponent and 10 of its 23 fraction bits.
    The pages only say that the TF32 mode changes results ("matmul_registers.cu",
    the note on CUBLAS_COMPUTE_32F), not how the 13 low fraction bits go, so
    both readings are offered: mode "trunc" drops them; mode "rne" rounds
    them to nearest, ties to even (a carry may raise the exponent).  For
    finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    if mode == "trunc":
        out = u & 0xFFFFE000
    elif mode == "rne":
        keep_lsb = (u >> 13) & 1            # the lowest kept fraction bit
        out = (u + 0xFFF + keep_lsb) & 0xFFFFE000
    else:
        raise ValueError("mode is 'trunc' or 'rne'")
    return out.astype(np.uint32).view(np.float32)


def general_bounds(K: int, max_abs_a: float, max_abs_b: float, alpha: float, beta: float,
                   max_abs_c: float) -> float:
    """Absolute tolerance for alpha * AB + beta * C: the product's bound scaled
    by |alpha|, plus a few FP32 rounding steps of |beta * C| and of the sum."""
    prod = ABS_COEF * math.sqrt(K) * max_abs_a * max_abs_b
    return abs(alpha) * prod + (abs(beta) * max_abs_c + abs(alpha) * K * max_abs_a * max_abs_b) * 2.0 ** -21


def gemm_rows(dtype, A, B, row0: int, row1: int, M=None, N=None, K=None,
              lda=None, ldb=None, nthreads: int | None = None) -> np.ndarray:
    """Rows [row0, row1) of the product, as a (row1-row0) x N float64 array."""
    code = _dtype_code(dtype)
    A, B = _bits(A, code), _bits(B, code)
    M, N, K, lda, ldb = _shape_args(A, B, M, N, K, lda, ldb)
    band = np.empty((max(row1 - row0, 0), N), dtype=np.float64)
    # The C routine indexes C by absolute row; hand it a pointer shifted back
    # by row0 rows so that row row0 lands at band[0].
    base = band.ctypes.data - row0 * N * 8
    nt = nthreads or os.cpu_count() or 1
    rc = lib().oracle_gemm_rows(code, _ptr(A), _ptr(B),
                                ctypes.cast(ctypes.c_void_p(base), ctypes.POINTER(ctypes.c_double)),
                                M, N, K, lda, ldb, N, row0, row1, nt)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed ({rc})")
    return band


def gemm_entries(dtype, A, B, rows, cols, M=None, N=None, K=None,
                 lda=None, ldb=None) -> np.ndarray:
    """Selected entries C[rows[t], cols[t]] (float64), one dot product each."""
    code = _dtype_code(dtype)
    A, B = _bits(A, code), _bits(B, code)
    M, N, K, lda, ldb = _shape_args(A, B, M, N, K, lda, ldb)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in shape")
    out = np.empty(r.shape, dtype=np.float64)
    rc = lib().oracle_gemm_entries(code, _ptr(A), _ptr(B), M, N, K, lda, ldb, r.size,
                                   r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   _dptr(out))
    if rc != 0:
        raise ValueError("oracle_gemm_entries: bad arguments")
    return out


@dataclass
class Comparison:
    """Result of checking a computed C against the oracle's C_ref."""
    max_abs: float
    abs_bound: float
    rel_frob: float
    rel_bound: float
    exact: bool          # every element equals C_ref rounded to FP32
    first_bad: tuple | None   # (row, col, got, want) of the first element over the abs bound

    @property
    def ok(self) -> bool:
        return self.max_abs <= self.abs_bound and self.rel_frob <= self.rel_bound

    def __str__(self) -> str:
        return (f"max|dC|={self.max_abs:.3e} (bound {self.abs_bound:.3e}), "
                f"relF={self.rel_frob:.3e} (bound {self.rel_bound:.1e}), exact={self.exact}, "
                f"first_bad={self.first_bad}")


def compare(C, C_ref, K: int, max_abs_a: float, max_abs_b: float) -> Comparison:
    """Check C (any float array) against the oracle's C_ref (float64) with the
    acceptance rule in this module's docstring.  The element check runs over
    every element given: pass full matrices, or matching 1-D samples.

    A non-finite element in C fails the check (it makes max|dC| infinite).
    When C_ref is all zero the relative Frobenius error is 0 if C is all zero
    too and infinite otherwise."""
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(C_ref, dtype=np.float64)
    if C.shape != R.shape:
        raise ValueError(f"shape mismatch {C.shape} vs {R.shape}")
    d = np.abs(C - R)
    d = np.where(np.isnan(d), np.inf, d)
    max_abs = float(d.max()) if d.size else 0.0
    abs_bound = ABS_COEF * math.sqrt(K) * max_abs_a * max_abs_b
    num = float(np.sqrt(np.sum(np.square(np.where(np.isinf(d), 0.0, d))))) if d.size else 0.0
    if np.isinf(max_abs):
        num = math.inf
    den = float(np.sqrt(np.sum(np.square(R)))) if R.size else 0.0
    if den == 0.0:
        rel = 0.0 if num == 0.0 else math.inf
    else:
        rel = num / den
    exact = bool(np.array_equal(C.astype(np.float32), R.astype(np.float32)))
    first_bad = None
    bad = np.argwhere(d > abs_bound)
    if bad.size:
        idx = tuple(int(v) for v in bad[0])
        first_bad = (*idx, float(C[idx]), float(R[idx]))
    return Comparison(max_abs, abs_bound, rel, REL_FROB, exact, first_bad)
