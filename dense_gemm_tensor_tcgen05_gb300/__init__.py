"""GB300-native dense GEMM: Python binding of libgb300gemm.so.

The library computes row-major C = A x B on one GB300 (sm_103a):

  * ``gemm_f16f32`` / ``gemm_bf16f32``: FP16 / BF16 inputs, FP32 accumulate
    and output, on the tensor cores (TMA + tcgen05.mma, accumulators in tensor
    memory);
  * ``sgemm_f32``: FP32 in and out on the CUDA cores.

The functions here carry the C ABI's names and arguments (device pointers as
ints, sizes, leading dimensions, a stream handle) and only marshal them:
every step of the product runs in the library's CUDA kernels.  ``matmul`` is
a convenience wrapper for torch tensors (device memory and streams come from
torch; nothing else does).  There is no CPU fallback: when the library is
missing or the GPU is not an sm_103 part, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "GemmError", "lib", "library_path", "gemm_f16f32", "gemm_bf16f32", "sgemm_f32", "gemm_ex",
    "gemm_ex_noalloc", "gemm_ex_host", "gemm_plan_describe", "gemm_device_error",
    "gemm_watchdog_selftest", "gemm_ex_stall_selftest", "gemm_tf32f32_bt", "gemm_e4m3f32_bt",
    "gemm_e5m2f32_bt", "gemm_release_workspace", "gemm_version", "gemm_launch_count",
    "gemm_alloc_count", "matmul", "gemm", "plan",
    "GemmOptions", "STATUS", "EXPORTED_SYMBOLS", "C_DTYPE",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libgb300gemm.so")

STATUS = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_VALUE",
    2: "GEMM_ERR_OVERLAP",
    3: "GEMM_ERR_UNSUPPORTED_DEVICE",
    4: "GEMM_ERR_LAUNCH",
    5: "GEMM_ERR_DEVICE_TIMEOUT",
    6: "GEMM_ERR_CUDA",
    7: "GEMM_ERR_OUT_OF_MEMORY",
}

# Every function include/gb300gemm.h declares.
EXPORTED_SYMBOLS = (
    "gemm_f16f32", "gemm_bf16f32", "sgemm_f32", "gemm_ex", "gemm_plan_describe",
    "gemm_device_error", "gemm_release_workspace", "gemm_status_string",
    "gemm_last_cuda_error", "gemm_version", "gemm_launch_count", "gemm_ex_noalloc",
    "gemm_ex_host", "gemm_watchdog_selftest", "gemm_tf32f32_bt", "gemm_e4m3f32_bt",
    "gemm_e5m2f32_bt", "gemm_ex_stall_selftest", "gemm_alloc_count",
)


class GemmError(RuntimeError):
    """A non-OK gemm_status_t."""

    def __init__(self, status: int, detail: str = ""):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}{': ' + detail if detail else ''}")


class GemmOptions(ctypes.Structure):
    """gemm_options_t (see include/gb300gemm.h)."""
    _fields_ = [("dtype", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("swap_ab", ctypes.c_int32),
                ("generic", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("store_mode", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float), ("epilogue", ctypes.c_int32),
                ("trans_a", ctypes.c_int32), ("trans_b", ctypes.c_int32),
                ("c_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libgb300gemm.so (built in-tree by ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"{library_path} is missing: build it with "
                    "`python -m dense_gemm_tensor_tcgen05_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(library_path)
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            sig = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
            for name in ("gemm_f16f32", "gemm_bf16f32", "sgemm_f32", "gemm_tf32f32_bt",
                         "gemm_e4m3f32_bt", "gemm_e5m2f32_bt"):
                f = getattr(L, name)
                f.argtypes = sig
                f.restype = ctypes.c_int
            L.gemm_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                  ctypes.POINTER(GemmOptions), vp]
            L.gemm_ex.restype = ctypes.c_int
            L.gemm_ex_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                          ctypes.POINTER(GemmOptions), vp]
            L.gemm_ex_noalloc.restype = ctypes.c_int
            L.gemm_ex_host.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                       ctypes.POINTER(GemmOptions), vp]
            L.gemm_ex_host.restype = ctypes.c_int
            L.gemm_plan_describe.argtypes = [ctypes.c_int32, vp, vp, vp, i64, i64, i64, i64, i64,
                                             i64, ctypes.POINTER(GemmOptions), ctypes.c_char_p, i64]
            L.gemm_plan_describe.restype = ctypes.c_int
            L.gemm_device_error.argtypes = [vp]
            L.gemm_device_error.restype = ctypes.c_int
            L.gemm_watchdog_selftest.argtypes = [ctypes.c_int32, vp]
            L.gemm_watchdog_selftest.restype = ctypes.c_int
            L.gemm_ex_stall_selftest.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                                 ctypes.POINTER(GemmOptions), ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32, vp]
            L.gemm_ex_stall_selftest.restype = ctypes.c_int
            L.gemm_release_workspace.argtypes = []
            L.gemm_release_workspace.restype = ctypes.c_int
            L.gemm_status_string.argtypes = [ctypes.c_int]
            L.gemm_status_string.restype = ctypes.c_char_p
            L.gemm_last_cuda_error.argtypes = []
            L.gemm_last_cuda_error.restype = ctypes.c_char_p
            L.gemm_version.argtypes = []
            L.gemm_version.restype = ctypes.c_int32
            L.gemm_launch_count.argtypes = []
            L.gemm_launch_count.restype = ctypes.c_int64
            L.gemm_alloc_count.argtypes = []
            L.gemm_alloc_count.restype = ctypes.c_int64
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        detail = lib().gemm_last_cuda_error().decode(errors="replace")
        raise GemmError(status, detail)


# ---- the C ABI, one Python function per entry point (marshalling only) ----

def gemm_f16f32(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                stream: int = 0) -> None:
    _check(lib().gemm_f16f32(A, B, C, M, N, K, lda, ldb, ldc, stream or None))


def gemm_bf16f32(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 stream: int = 0) -> None:
    _check(lib().gemm_bf16f32(A, B, C, M, N, K, lda, ldb, ldc, stream or None))


def sgemm_f32(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
              stream: int = 0) -> None:
    _check(lib().sgemm_f32(A, B, C, M, N, K, lda, ldb, ldc, stream or None))


def gemm_tf32f32_bt(A: int, Bt: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                    ldc: int, stream: int = 0) -> None:
    _check(lib().gemm_tf32f32_bt(A, Bt, C, M, N, K, lda, ldb, ldc, stream or None))


def gemm_e4m3f32_bt(A: int, Bt: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                    ldc: int, stream: int = 0) -> None:
    _check(lib().gemm_e4m3f32_bt(A, Bt, C, M, N, K, lda, ldb, ldc, stream or None))


def gemm_e5m2f32_bt(A: int, Bt: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                    ldc: int, stream: int = 0) -> None:
    _check(lib().gemm_e5m2f32_bt(A, Bt, C, M, N, K, lda, ldb, ldc, stream or None))


# gemm_options_t.c_dtype codes
C_DTYPE = {"float32": 0, "float16": 1, "bfloat16": 2}


def _options(dtype: int, tile_n=0, split_k=0, swap_ab=-1, generic=0, group_m=0,
             cta_pair=0, store_mode=0, stream_k=0, alpha=None, beta=None, trans_a=0,
             trans_b=0, c_dtype=0) -> GemmOptions:
    o = GemmOptions()
    o.c_dtype = c_dtype
    o.dtype, o.tile_n, o.split_k, o.swap_ab, o.generic, o.group_m = (
        dtype, tile_n, split_k, swap_ab, generic, group_m)
    o.cta_pair, o.store_mode, o.stream_k = cta_pair, store_mode, stream_k
    o.trans_a, o.trans_b = int(bool(trans_a)), int(bool(trans_b))
    if alpha is not None or beta is not None:
        # C = alpha * (A x B) + beta * C
        o.epilogue = 1
        o.alpha = 1.0 if alpha is None else float(alpha)
        o.beta = 0.0 if beta is None else float(beta)
    return o


def gemm_ex(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
            dtype: int, stream: int = 0, **opts) -> None:
    o = _options(dtype, **opts)
    _check(lib().gemm_ex(A, B, C, M, N, K, lda, ldb, ldc, ctypes.byref(o), stream or None))


def gemm_ex_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                    ldc: int, dtype: int, stream: int = 0, **opts) -> None:
    """gemm_ex without device allocations: split-K scratch lives in a fixed
    8 MiB array inside the library (see include/gb300gemm.h)."""
    o = _options(dtype, **opts)
    _check(lib().gemm_ex_noalloc(A, B, C, M, N, K, lda, ldb, ldc, ctypes.byref(o), stream or None))


def gemm_ex_host(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 dtype: int, stream: int = 0, **opts) -> None:
    """The product with A, B and C in (page-locked) host memory; copies and
    kernels are pipelined over row panels inside the library."""
    o = _options(dtype, **opts)
    _check(lib().gemm_ex_host(A, B, C, M, N, K, lda, ldb, ldc, ctypes.byref(o), stream or None))


def gemm_plan_describe(dtype: int, A: int, B: int, C: int, M: int, N: int, K: int, lda: int,
                       ldb: int, ldc: int, **opts) -> str:
    o = _options(dtype, **opts)
    buf = ctypes.create_string_buffer(512)
    _check(lib().gemm_plan_describe(dtype, A, B, C, M, N, K, lda, ldb, ldc, ctypes.byref(o),
                                    buf, len(buf)))
    return buf.value.decode()


def gemm_device_error(stream: int = 0) -> None:
    _check(lib().gemm_device_error(stream or None))


def gemm_watchdog_selftest(limit_ms: int = 20, stream: int = 0) -> None:
    """Enqueue the watchdog self-test kernel (see include/gb300gemm.h)."""
    _check(lib().gemm_watchdog_selftest(limit_ms, stream or None))


def gemm_ex_stall_selftest(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                           ldc: int, dtype: int, limit_ms: int, stall_cta: int, stall_fill: int,
                           stream: int = 0, **opts) -> None:
    """Run a tensor-core plan whose pipeline waits give up after limit_ms,
    with one CTA's producer withholding one stage (see include/gb300gemm.h).
    The timeout is then reported by gemm_device_error()."""
    o = _options(dtype, **opts)
    _check(lib().gemm_ex_stall_selftest(A, B, C, M, N, K, lda, ldb, ldc, ctypes.byref(o),
                                        limit_ms, stall_cta, stall_fill, stream or None))


def gemm_release_workspace() -> None:
    _check(lib().gemm_release_workspace())


def gemm_version() -> int:
    return int(lib().gemm_version())


def gemm_launch_count() -> int:
    return int(lib().gemm_launch_count())


def gemm_alloc_count() -> int:
    return int(lib().gemm_alloc_count())


# ---- torch convenience -------------------------------------------------------

_DTYPE_CODE = {"float16": 0, "bfloat16": 1, "float32": 2, "float8_e4m3fn": 4,
               "float8_e5m2": 5}


def _code(t) -> int:
    name = str(t.dtype).replace("torch.", "")
    if name not in _DTYPE_CODE:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPE_CODE[name]


def _row_major_ld(t, name: str) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.stride(1) != 1 and t.size(1) > 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    return max(t.stride(0), t.size(1)) if t.size(0) > 1 else max(t.size(1), 1)


def _operand_layout(t, name: str):
    """(transposed, ld) of a 2-D operand: row-major (unit column stride) is
    stored as itself; column-major (unit row stride, e.g. a .t() view) is the
    row-major storage of its transpose."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = t.shape
    if t.stride(1) == 1 or cols <= 1:
        return 0, _row_major_ld(t, name)
    if t.stride(0) == 1 or rows <= 1:
        return 1, max(t.stride(1), rows, 1)
    raise ValueError(f"{name} must be row-major or column-major")


def matmul(A, B, out=None, stream=None, tf32=False, out_dtype=None, **opts):
    """C = A @ B for 2-D tensors (row-major, any row stride).

    A and B: both float16, both bfloat16, both float32, both float8_e4m3fn
    or both float8_e5m2.  C is float32, or float16 / bfloat16 when ``out``
    has that dtype or ``out_dtype`` names it (the FP32 result rounded once to
    nearest even).  ``tf32=True`` runs float32 inputs on
    the tensor cores as TF32.  FP8 and TF32 products need A row-major and B
    column-major (B = Bt.t() for a row-major N x K Bt).  A and B may each
    be row-major or column-major (a .t() view), on the GPU or the host.
    CUDA tensors run gemm_f16f32 / gemm_bf16f32 / sgemm_f32 (or gemm_ex when
    plan options are given) on the current (or given) stream and return at
    once.  CPU tensors go through gemm_ex_host -- the library copies them in,
    multiplies and copies C back, pipelined over row panels -- and the call
    returns the CPU result after synchronising the stream (pass page-locked
    tensors for overlapped copies).  ``opts`` are gemm_options_t fields
    (tile_n, split_k, swap_ab, generic, group_m, cta_pair, store_mode,
    stream_k); alpha= and beta= give C = alpha * (A x B) + beta * out, with
    ``out`` supplying the old C.
    """
    import torch

    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    code = _code(A)
    if tf32:
        if code != 2:
            raise TypeError("tf32=True needs float32 operands")
        code = 3
    if A.is_cuda != B.is_cuda:
        raise ValueError("A and B must both be on the GPU or both on the host")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    st = stream if stream is not None else torch.cuda.current_stream()
    c_dt = out.dtype if out is not None else (out_dtype or torch.float32)
    c_name = str(c_dt).replace("torch.", "")
    if c_name not in C_DTYPE:
        raise TypeError(f"C must be float32, float16 or bfloat16, not {c_dt}")
    if out is not None and out_dtype is not None and out.dtype != out_dtype:
        raise TypeError("out and out_dtype disagree")
    if C_DTYPE[c_name]:
        opts = dict(opts, c_dtype=C_DTYPE[c_name])
    ta, lda = _operand_layout(A, "A")
    tb, ldb = _operand_layout(B, "B")
    if code >= 3 and (ta, tb) != (0, 1):
        raise ValueError("TF32 and FP8 products need A row-major and B column-major")
    if ta or tb:
        opts = dict(opts, trans_a=ta, trans_b=tb)
    if not A.is_cuda:
        if out is None:
            out = torch.empty((M, N), dtype=c_dt, pin_memory=True)
        elif out.is_cuda or tuple(out.shape) != (M, N):
            raise ValueError("out must be a CPU tensor of shape (M, N)")
        ldc = _row_major_ld(out, "C")
        gemm_ex_host(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc,
                     dtype=code, stream=st.cuda_stream, **opts)
        st.synchronize()
        return out
    if out is None:
        with torch.cuda.stream(st):
            out = torch.empty((M, N), dtype=c_dt, device=A.device)
    elif tuple(out.shape) != (M, N) or not out.is_cuda:
        raise ValueError("out must be a CUDA tensor of shape (M, N)")
    ldc = _row_major_ld(out, "C")
    args = (A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc)
    sh = st.cuda_stream
    if opts:
        gemm_ex(*args, dtype=code, stream=sh, **opts)
    elif code == 0:
        gemm_f16f32(*args, stream=sh)
    elif code == 1:
        gemm_bf16f32(*args, stream=sh)
    else:
        sgemm_f32(*args, stream=sh)
    return out


def gemm(A, B, out=None, **opts):
    """The same as matmul(A, B, out=out, ...): C = A @ B through the library."""
    return matmul(A, B, out=out, **opts)


def plan(A, B, out=None, tf32=False, **opts) -> str:
    """The plan text gemm_plan_describe gives for torch tensors A @ B."""
    code = _code(A)
    if out is not None and str(out.dtype).replace("torch.", "") in ("float16", "bfloat16"):
        opts = dict(opts, c_dtype=C_DTYPE[str(out.dtype).replace("torch.", "")])
    if tf32 and code == 2:
        code = 3
    M, K = A.shape
    _, N = B.shape
    # Only C's alignment is read; without `out`, describe a 256-byte aligned C.
    cptr = out.data_ptr() if out is not None else 256
    ldc = _row_major_ld(out, "C") if out is not None else N
    ta, lda = _operand_layout(A, "A")
    tb, ldb = _operand_layout(B, "B")
    if ta or tb:
        opts = dict(opts, trans_a=ta, trans_b=tb)
    return gemm_plan_describe(code, A.data_ptr(), B.data_ptr(), cptr, M, N, K,
                              lda, ldb, ldc, **opts)
