"""IEEE-754 binary16 (FP16) decode and round-to-nearest-even encode, float64.

Test infrastructure only (see ``oracle/__init__.py``).

FP16 is the storage type of every tensor on the path ("Integrate FP32 v37
prefill and exact E4M3 bridge", Implementation: FP32 QK/PV accumulation,
"probabilities and final output retain FP16 storage").  The bridge's output is
defined as the FP16 value nearest to the exact scaled E4M3 value, ties to
even, which needs an encoder that rounds once from an exact float64 value.
"""

import numpy as np

_EXP_BIAS = 15
_MANT_BITS = 10


def fp16_bits_to_f64(bits):
    """Decode FP16 bit patterns (uint16) to float64 exactly.

    sign s, exponent e (5 bits), fraction f (10 bits):
      e == 0         -> (-1)^s * f * 2^-24            (zero / subnormal)
      1 <= e <= 30   -> (-1)^s * (1024 + f) * 2^(e-25)
      e == 31        -> +-inf when f == 0, NaN otherwise
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = (b >> 15) & 1
    e = (b >> _MANT_BITS) & 0x1F
    f = b & 0x3FF
    mag = np.where(e == 0, f.astype(np.float64) * 2.0 ** -24,
                   np.ldexp((1024 + f).astype(np.float64), (e - 25).astype(np.int32)))
    mag = np.where(e == 31, np.where(f == 0, np.inf, np.nan), mag)
    return np.where(s == 1, -mag, mag)


def f64_to_fp16_bits(x):
    """Round float64 values to the nearest FP16 value, ties to even; return bits.

    For finite |x| with binary exponent E (2^E <= |x| < 2^(E+1)), the FP16 grid
    spacing around x is q = 2^(max(E, -14) - 10) (the max() gives the fixed
    subnormal spacing 2^-24).  |x|/q is exact in float64 (a power-of-two
    scaling) and ``np.rint`` rounds it to the nearest integer, ties to even,
    which is exactly round-to-nearest-even on the FP16 grid.  A rounded
    magnitude of 2^16 or more overflows to infinity (IEEE: the largest finite
    FP16 is 65504 and values from 65520 up round to inf).  NaN maps to the
    quiet NaN 0x7E00 with the sign kept.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)
    _, ex = np.frexp(a_f)            # a = m * 2^ex with 0.5 <= m < 1  ->  E = ex - 1
    E = np.where(a_f > 0, ex - 1, -14)
    E = np.maximum(E, -14)
    q_exp = (E - _MANT_BITS).astype(np.int32)
    n = np.rint(np.ldexp(a_f, -q_exp))          # integer count of grid steps
    val = np.ldexp(n, q_exp)                    # rounded magnitude (exact)
    nn = n.astype(np.int64)
    Ee = E.astype(np.int64)
    sub = (Ee == -14) & (nn < 1024)             # subnormal (or zero) result
    up = nn == 2048                             # rounding carried into the next binade
    nn_n = np.where(up, 1024, nn)
    Ee_n = np.where(up, Ee + 1, Ee)
    normal_bits = ((Ee_n + _EXP_BIAS) << _MANT_BITS) | (nn_n - 1024)
    bits = np.where(sub, nn, normal_bits)
    overflow = (val >= 65536.0) | (Ee_n > 15)
    bits = np.where(finite & ~overflow, bits, 0x7C00)
    bits = np.where(np.isnan(x), 0x7E00, bits)
    bits = np.where(sign, bits | 0x8000, bits)
    return bits.astype(np.uint16)


def f64_to_fp16(x):
    """Round float64 to FP16 (RNE) and return the rounded values as float64."""
    return fp16_bits_to_f64(f64_to_fp16_bits(x))
