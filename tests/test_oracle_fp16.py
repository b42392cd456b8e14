"""Pins for the oracle's FP16 decode / RNE encode (CPU only).

Pinned against numpy's float16 conversions (library routines), an exhaustive
round trip over all 65536 codes, and the closed-form rounding boundaries of
IEEE binary16 (midpoints round to even, overflow threshold 65520).
"""

import numpy as np

from oracle.fp16 import f64_to_fp16_bits, fp16_bits_to_f64

ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_decode_matches_numpy_all_codes():
    ours = fp16_bits_to_f64(ALL)
    ref = ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0x0000])


def test_round_trip_all_codes():
    vals = fp16_bits_to_f64(ALL)
    back = f64_to_fp16_bits(vals)
    nan = np.isnan(vals)
    assert np.array_equal(back[~nan], ALL[~nan])
    assert np.all(np.isnan(fp16_bits_to_f64(back[nan])))


def test_midpoints_round_to_even():
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    hi = lo + 1
    a = fp16_bits_to_f64(lo)
    b = fp16_bits_to_f64(hi)
    mid = (a + b) / 2.0                      # exact in float64
    even = np.where((lo & 1) == 0, lo, hi)
    assert np.array_equal(f64_to_fp16_bits(mid), even)
    assert np.array_equal(f64_to_fp16_bits(np.nextafter(mid, np.inf)), hi)
    assert np.array_equal(f64_to_fp16_bits(np.nextafter(mid, -np.inf)), lo)


def test_overflow_and_underflow_boundaries():
    cases = {
        65504.0: 0x7BFF,
        65519.99: 0x7BFF,
        65520.0: 0x7C00,         # halfway to 2^16 rounds to even -> overflow
        1e9: 0x7C00,
        -65520.0: 0xFC00,
        2.0 ** -24: 0x0001,
        2.0 ** -25: 0x0000,      # tie between 0 and the smallest subnormal -> even (0)
        2.0 ** -25 * 1.0000001: 0x0001,
        3 * 2.0 ** -25: 0x0002,  # tie between 1 and 2 subnormal steps -> 2
        2.0 ** -14: 0x0400,
        np.inf: 0x7C00,
        -np.inf: 0xFC00,
        -0.0: 0x8000,
    }
    for x, bits in cases.items():
        assert int(f64_to_fp16_bits(np.array([x]))[0]) == bits, x
    assert int(f64_to_fp16_bits(np.array([np.nan]))[0]) & 0x7C00 == 0x7C00


def test_encode_matches_numpy_random():
    # numpy's float64 -> float16 cast is a correctly rounded library routine.
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 4.5, 200000),
        rng.uniform(-65000, 65000, 50000),
    ])
    assert np.array_equal(f64_to_fp16_bits(x), x.astype(np.float16).view(np.uint16))
