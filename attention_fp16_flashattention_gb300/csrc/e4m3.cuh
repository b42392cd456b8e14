// Exact FP8 E4M3 -> FP16 conversion with a scale, shared by the paged bridge
// and the paged decode kernel ("Integrate FP32 v37 prefill and exact E4M3
// bridge", Implementation: exact E4M3 byte conversion with unit and non-unit
// scales).  Decoding uses the hardware e4m3x2 -> f16x2 conversion, which is
// exact (every finite E4M3 value is an FP16 value).  The scaled result is the
// FP16 value nearest to the exact product, ties to even:
//   * if the FP32 scale is itself an FP16 value, one IEEE FP16 multiply of two
//     FP16 operands rounds the exact product once;
//   * otherwise the product is formed in FP32 with round-to-odd (truncated
//     product, sticky bit from the exact FMA residual) and rounded to FP16 once;
//     FP32 carries 24 >= 11 + 2 significant bits, so the double rounding through
//     round-to-odd equals a single rounding (Boldo and Melquiond, "Emulation of
//     FMA and correctly rounded sums: proved algorithms using rounding to odd",
//     IEEE Trans. Computers 57(4), 2008).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace gbattn {

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t out;
    const uint16_t in = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
    return out;
}

__device__ __forceinline__ uint32_t scale_f16x2(uint32_t h2, __half2 s2) {
    __half2 x = *reinterpret_cast<__half2*>(&h2);
    __half2 y = __hmul2(x, s2);
    return *reinterpret_cast<uint32_t*>(&y);
}

__device__ __forceinline__ __half scale_round_to_odd(__half h, float s) {
    const float x = __half2float(h);
    float p = __fmul_rz(x, s);
    const float r = __fmaf_rn(x, s, -p);
    if (r != 0.0f) p = __uint_as_float(__float_as_uint(p) | 1u);
    return __float2half_rn(p);
}

__device__ __forceinline__ uint32_t scale_f16x2_general(uint32_t h2, float s) {
    __half2 x = *reinterpret_cast<__half2*>(&h2);
    __half2 y = __halves2half2(scale_round_to_odd(__low2half(x), s),
                               scale_round_to_odd(__high2half(x), s));
    return *reinterpret_cast<uint32_t*>(&y);
}

template <bool kHalfScale>
__device__ __forceinline__ void convert16(uint4 in, __half2 s2, float s, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = e4m3x2_to_f16x2(w[i] & 0xFFFFu);
        o[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[i] = kHalfScale ? scale_f16x2(o[i], s2) : scale_f16x2_general(o[i], s);
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// True when the FP32 value s is exactly an FP16 value (normal or subnormal).
inline bool is_fp16_value(float s) {
    const __half h = __float2half_rn(s);
    return __half2float(h) == s;
}

}  // namespace gbattn
