"""Seeded synthetic inputs for the GEMM workloads.

This module is the one thing the product path and the CPU oracle both take
inputs from, so it holds none of the GEMM's arithmetic: it only draws numbers
and rounds them to the element type.  It imports neither the CUDA library nor
the oracle.

Generator (counter-based, so any element can be drawn without the ones
before it): SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as published by
S. Vigna).  The i-th draw of stream ``key`` is

    mix(key + (i + 1) * 0x9E3779B97F4A7C15)

with mix(z) = z1 ^ (z1 >> 31), z1 = (z0 ^ (z0 >> 27)) * 0x94D049BB133111EB,
z0 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9, all mod 2^64.  ``key`` =
mix(seed * 4 + matrix_id) keeps A (id 0) and B (id 1) of one seed apart.

Distributions:
  uniform[-1, 1): the top 24 bits u of a draw give 2 * u / 2^24 - 1, which is
      exact in FP32; the closed endpoint 1 has probability zero and is taken
      as excluded.
  normal(0, sigma): Box-Muller in float64 on draws 2i and 2i+1
      (sqrt(-2 ln u1) cos(2 pi u2), u1 in (0, 1]), times sigma, then to FP32.
      sigma is a standard deviation: normal(0, 1/sqrt(K)) means sigma =
      1/sqrt(K).

The FP32 samples are rounded to nearest-even into FP16 (numpy's float16
cast) or BF16 (rounding the FP32 bit pattern to its upper half).  Arrays of
element bits (uint16 for 16-bit types, float32 for FP32) are returned; both
sides read those same bits.

Deterministic patterns used as exact pins:
  small_int: a[r][c] = ((r + 2c) mod 7) - 3, b[r][c] = ((3r + c) mod 5) - 2
      (the integer pattern of "matmul_registers.cu", fillInputs, extended to
      rectangles).  Every product is an integer of magnitude <= 6 and every
      partial sum of K <= 2^21 terms stays below 2^24, so FP16, BF16 and FP32
      hold the inputs and all partial sums exactly.
  mod_pattern: a_i = ((7i + 1) mod 13) / 13 - 1/2 and b_i = ((5i + 3) mod 11) / 11
      - 1/2 over the flat row-major index i, evaluated in FP32 (the input fill
      of the "04-wmma-matmul" code example), then rounded to the element type.
  ones, identity, rank-one integer patterns.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

DTYPES = ("f16", "bf16", "f32", "e4m3", "e5m2")


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, matrix_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(seed * 4 + matrix_id) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(z)[0]


def splitmix64(key: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of stream ``key`` (uint64)."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(np.uint64(key) + i * _GAMMA)


def _draws(seed: int, matrix_id: int, count: int, chunk: int = 1 << 24):
    key = int(_key(seed, matrix_id))
    out = np.empty(count, dtype=np.uint64)
    for s in range(0, count, chunk):
        n = min(chunk, count - s)
        out[s:s + n] = splitmix64(key, s, n)
    return out


def uniform_f32(seed: int, matrix_id: int, shape) -> np.ndarray:
    """uniform[-1, 1) samples in FP32 (each exact, on a 2^-23 grid)."""
    n = int(np.prod(shape))
    u = (_draws(seed, matrix_id, n) >> np.uint64(40)).astype(np.float64)
    return (u * (2.0 / 16777216.0) - 1.0).astype(np.float32).reshape(shape)


def normal_f32(seed: int, matrix_id: int, shape, sigma: float = 1.0) -> np.ndarray:
    """normal(0, sigma) samples in FP32 via Box-Muller on pairs of draws."""
    n = int(np.prod(shape))
    d = _draws(seed, matrix_id, 2 * n)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (z * sigma).astype(np.float32).reshape(shape)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bits, round to nearest, ties to even (finite inputs)."""
    w = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (w >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (w + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def round_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> FP16 bits, round to nearest, ties to even (numpy's cast)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def round_to_fp8_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """FP32 -> E4M3 / E5M2 bits (torch's round-to-nearest-even conversion;
    inputs are expected within range: |x| <= 448 for E4M3)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    tt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    return t.to(tt).view(torch.uint8).numpy().copy()


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round FP32 values to ``dtype`` and return the element bits
    (uint8 for e4m3/e5m2; uint16 for f16/bf16; float32 itself for f32)."""
    if dtype == "f16":
        return round_to_f16_bits(x)
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    if dtype in ("e4m3", "e5m2"):
        return round_to_fp8_bits(x, dtype)
    if dtype in ("f32", "tf32"):
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def bits_abs_max(bits: np.ndarray, dtype: str) -> float:
    """max |x| over element bits (a plain read of the values, for the error
    bound's scale)."""
    if bits.size == 0:
        return 0.0
    if dtype == "f16":
        return float(np.abs(bits.view(np.float16).astype(np.float32)).max())
    if dtype == "bf16":
        v = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        return float(np.abs(v).max())
    if dtype in ("e4m3", "e5m2"):
        import torch
        tt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        v = torch.from_numpy(np.ascontiguousarray(bits)).view(tt).float()
        return float(v.abs().max())
    return float(np.abs(bits.astype(np.float32)).max())


def padded(x: np.ndarray, ld: int) -> np.ndarray:
    """Copy a (rows, cols) array into a (rows, ld) array, ld >= cols, filling
    the padding with a recognisable non-zero bit pattern so that a kernel that
    reads past the logical columns is caught."""
    rows, cols = x.shape
    if ld < cols:
        raise ValueError("ld < cols")
    out = np.empty((rows, ld), dtype=x.dtype)
    if x.dtype == np.float32:
        out[...] = np.float32(1e30)
    elif x.dtype == np.uint8:
        out[...] = 0x7E     # 448 in E4M3, a NaN in E5M2: either spoils a sum it enters
    else:
        out[...] = 0x7BFF   # large finite in FP16; ~1.1e36 in BF16
    out[:, :cols] = x
    return out


def make(dist: str, dtype: str, rows: int, cols: int, seed: int, matrix_id: int,
         sigma: float = 1.0) -> np.ndarray:
    """One input matrix (rows x cols) as element bits.

    dist: 'uniform'  uniform[-1, 1)
          'normal'   normal(0, sigma)
          'small_int' the integer pattern (matrix_id 0 -> A form, 1 -> B form)
          'mod_pattern' the deterministic fractional pattern (same convention)
          'ones'     all ones
          'identity' ones on the diagonal
          'rank1'    A[i][k] = u_i (matrix_id 0) or B[k][j] = v_j (matrix_id 1),
                     small integers, so C = K u_i v_j exactly
    """
    if dist == "uniform":
        x = uniform_f32(seed, matrix_id, (rows, cols))
    elif dist == "normal":
        x = normal_f32(seed, matrix_id, (rows, cols), sigma)
    elif dist == "small_int":
        # (r + 2c) mod 7 and (3r + c) mod 5 depend on c only through c mod 7
        # (mod 5): round one period per row to the element type, then repeat
        # its bits along the row (the same bits as rounding every element)
        r = np.arange(rows, dtype=np.int64)[:, None]
        p = 7 if matrix_id == 0 else 5
        c = np.arange(p, dtype=np.int64)[None, :]
        if matrix_id == 0:
            period = ((r + 2 * c) % 7 - 3).astype(np.float32)
        else:
            period = ((3 * r + c) % 5 - 2).astype(np.float32)
        bits = to_bits(period, dtype)
        return np.ascontiguousarray(np.take(bits, np.arange(cols, dtype=np.int64) % p, axis=1))
    elif dist == "mod_pattern":
        i = np.arange(rows * cols, dtype=np.int64)
        if matrix_id == 0:
            num = ((i * 7 + 1) % 13).astype(np.float32)
            x = num / np.float32(13.0) - np.float32(0.5)
        else:
            num = ((i * 5 + 3) % 11).astype(np.float32)
            x = num / np.float32(11.0) - np.float32(0.5)
        x = x.astype(np.float32).reshape(rows, cols)
    elif dist == "ones":
        x = np.ones((rows, cols), dtype=np.float32)
    elif dist == "identity":
        x = np.eye(rows, cols, dtype=np.float32)
    elif dist == "rank1":
        if matrix_id == 0:
            u = (np.arange(rows, dtype=np.int64) % 5 - 2).astype(np.float32)
            x = np.repeat(u[:, None], cols, axis=1)
        else:
            v = (np.arange(cols, dtype=np.int64) % 3 - 1).astype(np.float32)
            x = np.repeat(v[None, :], rows, axis=0)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return to_bits(x, dtype)
