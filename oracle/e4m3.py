"""FP8 E4M3 decode and the paged E4M3 -> FP16 bridge, float64.

Test infrastructure only (see ``oracle/__init__.py``).

Format: the pages use the ``float8_e4m3fn`` flavour (FastVideo compare view,
fastvideo/distributed/projection_exchange.py and the FP4 key-quantisation
module name ``torch.float8_e4m3fn``): 1 sign bit, 4 exponent bits with bias 7,
3 fraction bits, no infinities, and the two codes with all exponent and
fraction bits set (0x7F, 0xFF) are NaN; the largest finite magnitude is 448
(the FP8 prefix round trip in prefix_quant.py divides by and clamps to 448).
The positive finite values follow the exact bit construction printed in the
FastVideo compare view (minimax_h3_swiglu_quant.cuh, ``scale_float``):
fraction m times 2^-9 when the exponent field is zero, and otherwise the FP32
number with biased exponent e + 120 and fraction m << 20, i.e.
(1 + m/8) * 2^(e - 7).  Negative codes are the sign-symmetric reading.

Bridge ("Integrate FP32 v37 prefill and exact E4M3 bridge", Purpose and
Implementation: an exact E4M3 paged-to-FP16 bridge with unit and non-unit
scales over the live length): token t of the logical sequence lives in
physical page ``page_table[t // page_size]`` at slot ``t % page_size``; the
output is the FP16 value nearest to decode(byte) * scale (one rounding of the
exact product, ties to even).  The product of a 4-bit significand and a 24-bit
FP32 scale is exact in float64, so computing it in float64 and rounding once
with the oracle's own FP16 encoder is the definition written out.
"""

import numpy as np

from .fp16 import f64_to_fp16_bits


def e4m3fn_decode(codes):
    """Decode E4M3 ("fn") bytes to float64.

    byte b: s = b >> 7, e = (b >> 3) & 15, m = b & 7
      b & 0x7F == 0x7F  -> NaN (sign kept)
      e == 0            -> (-1)^s * m * 2^-9
      otherwise         -> (-1)^s * (1 + m/8) * 2^(e - 7)
    """
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9,
                   (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int32)))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_scaled_to_fp16_bits(codes, scale):
    """RNE_fp16(decode(code) * scale) as uint16 bits; ``scale`` is an FP32 value.

    The float64 product decode(code) * float64(scale) is exact (4 + 24 <= 53
    significant bits), so the only rounding is the FP16 encode.
    """
    s = float(np.float32(scale))
    return f64_to_fp16_bits(e4m3fn_decode(codes) * s)


def paged_e4m3_to_fp16(k_pages, v_pages, page_table, kv_len, k_scale, v_scale):
    """The bridge: paged E4M3 K and V caches -> contiguous FP16 K and V.

    k_pages, v_pages : uint8 [num_phys_pages][page_size][Hkv][D]
    page_table       : int  [ceil(kv_len / page_size)]   logical -> physical page
    returns          : (k_bits, v_bits) uint16 [Hkv][kv_len][D] (FP16 bit patterns)

    Only the live length t < kv_len is produced.  Written as a per-token gather
    followed by an elementwise decode-and-round, exactly as the definition
    reads; a 256-entry table of the decoded-and-rounded values is that
    elementwise function evaluated once per code.
    """
    k_pages = np.asarray(k_pages, dtype=np.uint8)
    v_pages = np.asarray(v_pages, dtype=np.uint8)
    page_size = k_pages.shape[1]
    t = np.arange(kv_len)
    phys = np.asarray(page_table, dtype=np.int64)[t // page_size]
    slot = t % page_size
    k_tok = k_pages[phys, slot]            # [kv_len][Hkv][D]
    v_tok = v_pages[phys, slot]
    codes = np.arange(256, dtype=np.uint8)
    k_table = e4m3_scaled_to_fp16_bits(codes, k_scale)
    v_table = e4m3_scaled_to_fp16_bits(codes, v_scale)
    k_out = k_table[k_tok].transpose(1, 0, 2)   # [Hkv][kv_len][D]
    v_out = v_table[v_tok].transpose(1, 0, 2)
    return np.ascontiguousarray(k_out), np.ascontiguousarray(v_out)
