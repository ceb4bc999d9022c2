"""Pins for oracle.formats: decode and round-to-nearest-even of binary16 / bfloat16.

The oracle writes both formats from their field definitions.  Here they are tied to
things other than themselves: numpy's binary16 type, the definition of bfloat16 as the
upper half of binary32, torch's binary32 -> bfloat16 rounding, exhaustive round trips
and constructed tie cases.
"""

import numpy as np
import pytest
import torch

from oracle import formats

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def test_decode_f16_matches_numpy_half_for_every_pattern():
    ours = formats.decode(ALL, "f16")
    ref = ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_is_upper_half_of_binary32_for_every_pattern():
    ours = formats.decode(ALL, "bf16")
    ref = (ALL.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_round_trip_every_non_nan_pattern(fmt):
    vals = formats.decode(ALL, fmt)
    keep = ~np.isnan(vals)
    back = formats.round_rne(vals[keep], fmt)
    assert np.array_equal(back, ALL[keep])


def _random_doubles(n, lo_exp, hi_exp, seed):
    rng = np.random.default_rng(seed)
    mant = rng.random(n) + 1.0                      # [1, 2)
    exps = rng.integers(lo_exp, hi_exp, n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return sign * np.ldexp(mant, exps)


def test_round_f16_matches_numpy_on_random_doubles():
    # binade exponents from deep underflow (-30) through overflow (20 > emax=15)
    x = _random_doubles(2_000_000, -30, 20, seed=11)
    x = np.concatenate([x, [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.99, 65520.0,
                            2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14]])
    ours = formats.round_rne(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_bf16_matches_torch_on_binary32_values():
    # values representable in binary32 are rounded once by torch's fp32 -> bf16 cast
    rng = np.random.default_rng(12)
    raw = rng.integers(0, 1 << 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    f32 = raw.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    ours = formats.round_rne(f32.astype(np.float64), "bf16")
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_exact_midpoints_round_to_even(fmt):
    # every pair of adjacent positive finite values: the midpoint goes to the even pattern,
    # a hair above goes up, a hair below goes down
    ebits, mbits = formats.FIELDS[fmt]
    top = ((1 << ebits) - 1) << mbits          # +inf pattern
    lo = np.arange(0, top - 1, dtype=np.int64).astype(np.uint16)
    hi = (lo.astype(np.int64) + 1).astype(np.uint16)
    vlo = formats.decode(lo, fmt)
    vhi = formats.decode(hi, fmt)
    mid = (vlo + vhi) / 2.0                     # exact in binary64
    got = formats.round_rne(mid, fmt)
    even = np.where(lo % 2 == 0, lo, hi)
    assert np.array_equal(got, even)
    gap = vhi - vlo
    assert np.array_equal(formats.round_rne(mid + gap * 2.0 ** -20, fmt), hi)
    assert np.array_equal(formats.round_rne(mid - gap * 2.0 ** -20, fmt), lo)


@pytest.mark.parametrize("fmt,maxbits", [("f16", 0x7BFF), ("bf16", 0x7F7F)])
def test_overflow_threshold(fmt, maxbits):
    vmax = float(formats.decode(np.array([maxbits], np.uint16), fmt)[0])
    half_ulp = float(formats.ulp(np.array([maxbits], np.uint16), fmt)[0]) / 2
    inf_bits = maxbits + 1
    # below the midpoint to 2^(emax+1): stays finite; at the midpoint: ties to even = inf
    assert formats.round_rne(np.array([vmax + half_ulp * 0.999]), fmt)[0] == maxbits
    assert formats.round_rne(np.array([vmax + half_ulp]), fmt)[0] == inf_bits
    assert formats.round_rne(np.array([-(vmax + half_ulp)]), fmt)[0] == inf_bits | 0x8000


def test_nan_maps_to_nan():
    for fmt in ("f16", "bf16"):
        b = formats.round_rne(np.array([np.nan]), fmt)
        assert np.isnan(formats.decode(b, fmt)[0])
