"""Pins for the oracle's E4M3 decode and the paged E4M3 -> FP16 bridge (CPU only).

* The positive finite codes are checked against the exact bit construction
  printed on the FastVideo compare view (minimax_h3_swiglu_quant.cuh,
  ``scale_float``): FP32 bits ((e + 120) << 23) | (m << 20), or m * 2^-9 when
  e == 0.  The test builds those FP32 bit patterns itself (a different
  formulation from the oracle's arithmetic decode).
* The page-printed points in tests/golden/e4m3_points.txt.
* PyTorch's float8_e4m3fn -> float64 conversion (the library type the pages
  name) for all 256 codes.
* The bridge with non-power-of-two scales against exact rational arithmetic
  (fractions.Fraction) and a nearest-FP16 search over every FP16 value.
"""

import bisect
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle.e4m3 import e4m3_scaled_to_fp16_bits, e4m3fn_decode, paged_e4m3_to_fp16
from oracle.fp16 import fp16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")
CODES = np.arange(256, dtype=np.uint8)


def _page_bit_construction(code):
    """The page's positive-finite E4M3 construction, via FP32 bit patterns."""
    e = (code >> 3) & 15
    m = code & 7
    if e == 0:
        return float(np.float32(m) * np.float32(0.001953125))
    bits = ((e + 120) << 23) | (m << 20)
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_positive_finite_codes_match_page_construction():
    dec = e4m3fn_decode(CODES)
    for c in range(0x7F):             # 0x00 .. 0x7E
        assert dec[c] == _page_bit_construction(c), hex(c)


def test_sign_symmetry_zero_and_nan():
    dec = e4m3fn_decode(CODES)
    for c in range(0x7F):
        assert dec[c | 0x80] == -dec[c]
    assert dec[0x00] == 0.0 and not np.signbit(dec[0x00])
    assert dec[0x80] == 0.0 and np.signbit(dec[0x80])
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert np.sum(np.isnan(dec)) == 2
    assert np.nanmax(np.abs(dec)) == 448.0


def test_golden_points():
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, value = line.split()[:2]
            assert e4m3fn_decode(np.array([int(code, 16)], dtype=np.uint8))[0] == float(value)
            n += 1
    assert n >= 4


def test_decode_matches_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = e4m3fn_decode(CODES)
    nan = np.isnan(t)
    assert np.array_equal(nan, np.isnan(dec))
    assert np.array_equal(t[~nan], dec[~nan])


# Every non-negative finite FP16 value in code order, plus 2^16 standing for the
# overflow to infinity (code 0x7C00, which is even, so ties at 65520 go to inf).
_FP16_POS = [float(x) for x in fp16_bits_to_f64(np.arange(0x7C00, dtype=np.uint16))] + [65536.0]


def _nearest_fp16_bits_exact(value: Fraction):
    """The FP16 code nearest to an exact rational, ties to the even code."""
    sign = 0x8000 if value < 0 else 0
    a = abs(value)
    i = bisect.bisect_left(_FP16_POS, a)
    best = None
    for j in (i - 1, i):
        if 0 <= j < len(_FP16_POS):
            d = abs(Fraction(_FP16_POS[j]) - a)
            if best is None or d < best[0] or (d == best[0] and j % 2 == 0):
                best = (d, j)
    return sign | best[1]


@pytest.mark.parametrize("scale", [1.0, 0.0625, 0.125, 1.0 / 3.0, 0.3, 1.7e-3, 300.0, 7.123e-5])
def test_scaled_decode_is_single_rounding(scale):
    s32 = float(np.float32(scale))
    got = e4m3_scaled_to_fp16_bits(CODES, scale)
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        exact = Fraction(float(e4m3fn_decode(np.array([c], dtype=np.uint8))[0])) * Fraction(s32)
        want = _nearest_fp16_bits_exact(exact)
        if c & 0x80:
            want |= 0x8000           # keeps the sign of zero results too
        assert int(got[c]) == want, (hex(c), scale)


def test_power_of_two_scale_is_exact():
    torch = pytest.importorskip("torch")
    for s in (1.0, 0.0625, 0.125):
        t = (torch.from_numpy(CODES.copy()).view(torch.float8_e4m3fn).to(torch.float16) * s)
        ref = t.numpy().view(np.uint16)
        got = e4m3_scaled_to_fp16_bits(CODES, s)
        finite = (CODES & 0x7F) != 0x7F
        assert np.array_equal(got[finite], ref[finite])


def test_bridge_identity_table_equals_contiguous_decode():
    rng = np.random.default_rng(1)
    P, ps, Hkv, D = 8, 32, 2, 64
    kp = rng.integers(0, 256, (P, ps, Hkv, D)).astype(np.uint8)
    vp = rng.integers(0, 256, (P, ps, Hkv, D)).astype(np.uint8)
    kv_len = P * ps - 5                                   # live length inside the last page
    k, v = paged_e4m3_to_fp16(kp, vp, np.arange(P), kv_len, 1.0, 0.5)
    assert k.shape == (Hkv, kv_len, D)
    flat_k = kp.reshape(P * ps, Hkv, D)[:kv_len].transpose(1, 0, 2)
    flat_v = vp.reshape(P * ps, Hkv, D)[:kv_len].transpose(1, 0, 2)
    assert np.array_equal(k, e4m3_scaled_to_fp16_bits(flat_k, 1.0))
    assert np.array_equal(v, e4m3_scaled_to_fp16_bits(flat_v, 0.5))


def test_bridge_permuted_table_round_trip():
    rng = np.random.default_rng(2)
    P, ps, Hkv, D = 16, 32, 1, 32
    kp = rng.integers(0, 256, (P, ps, Hkv, D)).astype(np.uint8)
    perm = rng.permutation(P)
    phys = np.empty_like(kp)
    phys[perm] = kp                 # physical page perm[i] holds logical page i
    k1, _ = paged_e4m3_to_fp16(phys, phys, perm, P * ps, 0.25, 0.25)
    k0, _ = paged_e4m3_to_fp16(kp, kp, np.arange(P), P * ps, 0.25, 0.25)
    assert np.array_equal(k0, k1)
    t = 77                          # token t reads logical page t // ps, slot t % ps
    assert np.array_equal(k1[0, t], e4m3_scaled_to_fp16_bits(kp[t // ps, t % ps, 0], 0.25))
