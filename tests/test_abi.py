"""The C-ABI library on the host: it builds, loads and exports every symbol
include/gb300gemm.h declares, and rejects bad arguments with status codes
before touching CUDA (no compute calls: no GPU here)."""
import ctypes
import os
import re

import pytest

import dense_gemm_tensor_tcgen05_gb300 as g
from dense_gemm_tensor_tcgen05_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gb300gemm.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return g.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_\w+|sgemm_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert header_functions() == sorted(g.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_exported_names_are_unmangled():
    syms = os.popen(f"nm -D --defined-only {g.library_path}").read()
    for name in header_functions():
        assert re.search(rf"\bT {name}$", syms, re.M), name


def test_status_strings_and_version(L):
    for code, name in g.STATUS.items():
        assert L.gemm_status_string(code).decode().startswith(name)
    assert L.gemm_status_string(99).decode() == "unknown gemm_status_t"
    assert g.gemm_version() == 200


# Argument errors are reported before any CUDA call, so these run without a GPU.
P = 1 << 20   # an aligned, never dereferenced address


@pytest.mark.parametrize("fn", ["gemm_f16f32", "gemm_bf16f32", "sgemm_f32"])
@pytest.mark.parametrize("args,status", [
    ((P, 2 * P, 3 * P, -1, 4, 4, 4, 4, 4), 1),        # negative M
    ((P, 2 * P, 3 * P, 4, -2, 4, 4, 4, 4), 1),        # negative N
    ((P, 2 * P, 3 * P, 4, 4, -3, 4, 4, 4), 1),        # negative K
    ((P, 2 * P, 3 * P, 4, 4, 8, 7, 4, 4), 1),         # lda < K
    ((P, 2 * P, 3 * P, 4, 8, 4, 4, 7, 8), 1),         # ldb < N
    ((P, 2 * P, 3 * P, 4, 8, 4, 4, 8, 7), 1),         # ldc < N
    ((0, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4), 1),         # null A
    ((P, 0, 3 * P, 4, 4, 4, 4, 4, 4), 1),             # null B
    ((P, 2 * P, 0, 4, 4, 4, 4, 4, 4), 1),             # null C
    ((P, 2 * P, 3 * P, 1 << 31, 4, 4, 4, 4, 4), 1),   # M beyond int32
    ((P, 2 * P, P + 8, 4, 4, 4, 4, 4, 4), 2),         # C overlaps A
    ((P, 2 * P, 2 * P, 4, 4, 4, 4, 4, 4), 2),         # C is B
])
def test_bad_arguments_rejected_on_host(L, fn, args, status):
    assert getattr(L, fn)(*args, None) == status


@pytest.mark.parametrize("fn", ["gemm_f16f32", "gemm_bf16f32", "sgemm_f32"])
def test_empty_output_is_a_no_op(L, fn):
    # M == 0 or N == 0: nothing to do, nothing enqueued, null pointers allowed
    assert getattr(L, fn)(0, 0, 0, 0, 5, 5, 5, 5, 5, None) == 0
    assert getattr(L, fn)(0, 0, 0, 5, 0, 5, 5, 0, 0, None) == 0


def test_k_zero_allows_null_inputs_in_argument_check(L):
    # K == 0 never reads A or B; only C must be given.  Without a GPU the call
    # then stops at the device query, which is not an argument error.
    st = L.gemm_f16f32(0, 0, P, 3, 3, 0, 0, 3, 3, None)
    assert st != 1


def test_gemm_ex_rejects_bad_options(L):
    o = g.GemmOptions()
    o.dtype = 7
    assert L.gemm_ex(P, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1
    assert L.gemm_ex(P, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4, None, None) == 1


def test_python_binding_raises_gemm_error(L):
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16f32(P, 2 * P, 3 * P, -1, 4, 4, 4, 4, 4)
    assert e.value.status == 1 and e.value.name == "GEMM_ERR_INVALID_VALUE"


def test_transposed_leading_dimensions_checked_on_host(L):
    o = g.GemmOptions()
    o.dtype, o.swap_ab, o.trans_a = 0, -1, 1
    # trans_a: A is K x M, so lda must be >= M = 8
    assert L.gemm_ex(P, 2 * P, 3 * P, 8, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1
    o.trans_a, o.trans_b = 0, 1
    # trans_b: B is N x K, so ldb must be >= K = 6
    assert L.gemm_ex(P, 2 * P, 3 * P, 4, 4, 6, 6, 4, 4, ctypes.byref(o), None) == 1
    o.trans_b = 2
    assert L.gemm_ex(P, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1


def test_host_entry_checks_transposed_storage_on_host(L):
    # gemm_ex_host takes the same transposed layouts as gemm_ex; the leading
    # dimensions are those of the host arrays and are checked before any
    # device work (host pointers here are never dereferenced)
    o = g.GemmOptions()
    o.dtype, o.swap_ab, o.trans_a = 1, -1, 1
    assert L.gemm_ex_host(P, 2 * P, 3 * P, 8, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1   # lda < M
    o.trans_a, o.trans_b = 0, 1
    assert L.gemm_ex_host(P, 2 * P, 3 * P, 4, 4, 6, 6, 4, 4, ctypes.byref(o), None) == 1   # ldb < K
    o.trans_b = 2
    assert L.gemm_ex_host(P, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1
    o.trans_b, o.c_dtype = 0, 3
    assert L.gemm_ex_host(P, 2 * P, 3 * P, 4, 4, 4, 4, 4, 4, ctypes.byref(o), None) == 1   # bad C type
    # valid arguments get past the checks; without a GPU the call then stops
    # at the device query, which is not an argument error
    o.c_dtype, o.trans_a, o.trans_b = 0, 1, 1
    assert L.gemm_ex_host(P, 2 * P, 3 * P, 4, 4, 6, 4, 6, 4, ctypes.byref(o), None) != 1


def test_stall_selftest_checks_its_arguments_on_host(L):
    # the wait limit is checked before anything else; options are required
    o = g.GemmOptions()
    o.dtype, o.swap_ab = 1, -1
    args = (P, 2 * P, 3 * P, 256, 256, 256, 256, 256, 256)
    assert L.gemm_ex_stall_selftest(*args, ctypes.byref(o), 0, 0, 0, None) == 1
    assert L.gemm_ex_stall_selftest(*args, ctypes.byref(o), 2001, 0, 0, None) == 1
    assert L.gemm_ex_stall_selftest(*args, None, 20, 0, 0, None) == 1
    # a valid request gets past the checks and stops at the device query here
    assert L.gemm_ex_stall_selftest(*args, ctypes.byref(o), 20, 0, 0, None) not in (0, 1)


def test_alloc_count_starts_at_zero_without_a_gpu(L):
    # nothing above allocated device memory (every call stopped on the host)
    assert g.gemm_alloc_count() == 0
