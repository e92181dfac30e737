"""Pins for the oracle's double -> FP16 / BF16 encoders (round to nearest,
ties to even), which state what a 16-bit output C must hold.

Anchors independent of the encoder: numpy's float64 -> float16 conversion
(IEEE round to nearest even), torch's float32 -> bfloat16 conversion on
values that are exact in float32, exhaustive round trips through the
oracle's separately pinned decoders, a nearest-neighbour check over the bit
patterns on either side, and hand-worked ties and overflow thresholds."""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def _random_doubles(rng, n, lo_exp, hi_exp):
    mant = rng.random(n) + 0.5
    exps = rng.integers(lo_exp, hi_exp, n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return sign * np.ldexp(mant, exps)


def test_f16_matches_numpy_rne():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _random_doubles(rng, 200000, -30, 18),                   # subnormal .. overflow
        np.ldexp(np.arange(1, 4096) + 0.5, -24 - 1),           # ties in the subnormal range
        np.ldexp(2048 + np.arange(0, 2048) + 0.5, -11),        # ties in [1, 2)
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300,
                  2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -26, 2.0 ** -14 * (1 - 2.0 ** -11)])])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = oracle.encode16("f16", x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_bf16_matches_torch_rne_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 32, 300000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    f = np.concatenate([bits, ties]).view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.encode16("bf16", f.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (f[bad[:5]], got[bad[:5]], want[bad[:5]])


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_round_trip_every_finite_pattern(dt):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode(dt, codes)
    fin = np.isfinite(vals)
    got = oracle.encode16(dt, vals[fin])
    want = codes[fin]
    # -0 and +0 keep their signs
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_result_is_the_nearest_representable(dt):
    rng = np.random.default_rng(3)
    lo, hi = (-26, 16) if dt == "f16" else (-134, 127)
    x = _random_doubles(rng, 50000, lo, hi)
    r = oracle.round16(dt, x)
    codes = oracle.encode16(dt, x)
    # the magnitude's neighbours: one pattern down and one up
    mag = codes & 0x7FFF
    sign = codes & 0x8000
    down = oracle.decode(dt, (sign | np.maximum(mag, 1) - 1).astype(np.uint16))
    up = oracle.decode(dt, (sign | (mag + 1)).astype(np.uint16))
    d = np.abs(r - x)
    fin = np.isfinite(r)
    assert np.all(d[fin] <= np.abs(down - x)[fin])
    up_ok = np.isfinite(up)
    assert np.all(d[fin & up_ok] <= np.abs(up - x)[fin & up_ok])
    assert np.all(d[fin] <= oracle.half_ulp16(dt, x)[fin])


def test_hand_worked_ties_and_thresholds():
    e = lambda dt, v: int(oracle.encode16(dt, [v])[0])
    assert e("f16", 1 + 2 ** -11) == 0x3C00          # tie, even neighbour is 1.0
    assert e("f16", 1 + 3 * 2 ** -11) == 0x3C02      # tie, even neighbour is 1 + 2^-9
    assert e("f16", 2 ** -25) == 0x0000              # half the smallest subnormal -> +0
    assert e("f16", 3 * 2 ** -25) == 0x0002          # tie between subnormals 1 and 2 -> 2
    assert e("f16", 2 ** -14 * (1 - 2 ** -11)) == 0x0400   # rounds up into the normals
    assert e("f16", 65504.0) == 0x7BFF
    assert e("f16", 65519.99) == 0x7BFF
    assert e("f16", 65520.0) == 0x7C00               # tie at the top rounds to infinity
    assert e("f16", -2.5) == 0xC100
    assert e("bf16", 1 + 2 ** -8) == 0x3F80
    assert e("bf16", 1 + 3 * 2 ** -8) == 0x3F82
    assert e("bf16", 3.0) == 0x4040
    assert e("bf16", 2.0 ** 127 * (2 - 2 ** -8)) == 0x7F80   # tie above the largest finite
    assert e("bf16", 2.0 ** 127 * (2 - 2 ** -7)) == 0x7F7F
    assert e("f16", float("nan")) & 0x7C00 == 0x7C00 and e("f16", float("nan")) & 0x3FF
    assert e("bf16", float("-inf")) == 0xFF80


def test_half_ulp16_values():
    assert oracle.half_ulp16("f16", [1.0])[0] == 2.0 ** -11
    assert oracle.half_ulp16("f16", [1.999])[0] == 2.0 ** -11
    assert oracle.half_ulp16("f16", [2.0])[0] == 2.0 ** -10
    assert oracle.half_ulp16("f16", [1e-7])[0] == 2.0 ** -25
    assert oracle.half_ulp16("bf16", [1.0])[0] == 2.0 ** -8
    assert oracle.half_ulp16("bf16", [0.0])[0] == 2.0 ** -134
