// Paged FP8 E4M3 -> FP16 bridge ("Integrate FP32 v37 prefill and exact E4M3
// bridge", Purpose and Implementation: exact E4M3 byte conversion with unit
// and non-unit scales over the live length).
//
// Each thread turns 8 consecutive E4M3 bytes of one token into 8 FP16 values
// (one 8-byte load, one 16-byte store) for K and for V, so that every store
// instruction of a warp writes 512 contiguous bytes: whole 32-byte sectors.
// A thread handles four such chunks at a time (loads first), and the chunk's
// token, head and position come from shifts where the sizes are powers of two
// (the 64-bit divisions had made the kernel issue-bound).
// (With 16 bytes in and two 16-byte stores per thread, each store instruction
// wrote half of every sector it touched, and the same bytes took 16% longer.)
// The exact scaled conversion is in e4m3.cuh.
#include <cuda_fp16.h>

#include "e4m3.cuh"
#include "host.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

// Eight E4M3 bytes (two words) to eight scaled FP16 values (one 16-byte word).
template <bool kHalfScale>
__device__ __forceinline__ uint4 convert8(uint2 in, __half2 s2, float s) {
    uint32_t o[4] = {e4m3x2_to_f16x2(in.x & 0xFFFFu), e4m3x2_to_f16x2(in.x >> 16),
                     e4m3x2_to_f16x2(in.y & 0xFFFFu), e4m3x2_to_f16x2(in.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = kHalfScale ? scale_f16x2(o[i], s2) : scale_f16x2_general(o[i], s);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Where a chunk sits: token t, head h, chunk c of the row; the page table entry
// and the input and output offsets.  kPow2: chunks per token, chunks per row and
// the page size are powers of two (shifts and masks, passed as log2 values);
// otherwise 64-bit division.
struct BridgeGeom {
    int page_size, hkv, D;
    int log_ppt, log_cpr, log_page;   // log2 of chunks per token, chunks per row, page size
};

template <bool kPow2>
__device__ __forceinline__ void chunk_place(long long g, const BridgeGeom& q, long long& t, int& h, int& c) {
    if (kPow2) {
        t = g >> q.log_ppt;
        const int rem = static_cast<int>(g & ((1LL << q.log_ppt) - 1));
        h = rem >> q.log_cpr;
        c = rem & ((1 << q.log_cpr) - 1);
    } else {
        const int cpr = q.D >> 3;
        const long long per_token = static_cast<long long>(q.hkv) * cpr;
        t = g / per_token;
        const int rem = static_cast<int>(g - t * per_token);
        h = rem / cpr;
        c = rem - h * cpr;
    }
}

// Each thread takes chunks g and g + stride of the grid stride loop together:
// their four loads are in flight before the first store.  (Four chunks per
// thread kept more loads in flight but ran 5% slower: 41.6 against 39.6 us per
// call, 37.3 against 35.5 us back to back; eight chunks 45.7 us.)
template <bool kHalfScale, bool kPow2>
__global__ void __launch_bounds__(256) e4m3_bridge_kernel(
    const uint8_t* __restrict__ kp, const uint8_t* __restrict__ vp,
    const int32_t* __restrict__ table, int num_phys, int kv_len, BridgeGeom q,
    float ks, float vs, __half2 ks2, __half2 vs2, __half* __restrict__ ko,
    __half* __restrict__ vo, uint32_t* status) {
    constexpr int U = 2;
    const long long per_token = static_cast<long long>(q.hkv) * (q.D >> 3);
    const long long total = static_cast<long long>(kv_len) * per_token;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long g0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g0 < total;
         g0 += U * stride) {
        uint2 kin[U], vin[U];
        long long out_off[U];
        bool live[U], bad[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long g = g0 + u * stride;
            live[u] = g < total;
            bad[u] = false;
            kin[u] = vin[u] = make_uint2(0u, 0u);
            out_off[u] = 0;
            if (!live[u]) continue;
            long long t;
            int h, c;
            chunk_place<kPow2>(g, q, t, h, c);
            const long long tp = kPow2 ? (t >> q.log_page) : t / q.page_size;
            const int slot = static_cast<int>(kPow2 ? (t & ((1LL << q.log_page) - 1)) : t - tp * q.page_size);
            const int page = table[tp];
            out_off[u] = (static_cast<long long>(h) * kv_len + t) * q.D + static_cast<long long>(c) * 8;
            if (page < 0 || page >= num_phys) {
                bad[u] = true;
                if (c == 0 && h == 0 && slot == 0) atomicOr(status, kDevBadPage);
                continue;
            }
            const long long in_off =
                ((static_cast<long long>(page) * q.page_size + slot) * q.hkv + h) * q.D +
                static_cast<long long>(c) * 8;
            kin[u] = __ldcs(reinterpret_cast<const uint2*>(kp + in_off));
            vin[u] = __ldcs(reinterpret_cast<const uint2*>(vp + in_off));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (!live[u]) continue;
            const uint4 k16 = bad[u] ? make_uint4(0, 0, 0, 0) : convert8<kHalfScale>(kin[u], ks2, ks);
            const uint4 v16 = bad[u] ? make_uint4(0, 0, 0, 0) : convert8<kHalfScale>(vin[u], vs2, vs);
            __stcs(reinterpret_cast<uint4*>(ko + out_off[u]), k16);
            __stcs(reinterpret_cast<uint4*>(vo + out_off[u]), v16);
        }
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" int e4m3_paged_to_fp16(const uint8_t* k_pages, const uint8_t* v_pages,
                                  const int32_t* page_table, int num_phys_pages, int page_size,
                                  int kv_len, int Hkv, int D, float k_scale, float v_scale,
                                  void* k_out, void* v_out, void* stream) {
    CallRange nvtx_range("e4m3_paged_to_fp16");
    if (!k_pages || !v_pages || !page_table || !k_out || !v_out) return GBATTN_ERR_NULL;
    if (num_phys_pages <= 0 || page_size <= 0 || kv_len <= 0 || Hkv <= 0 || D <= 0)
        return GBATTN_ERR_SHAPE;
    if (D % 16 != 0) return GBATTN_ERR_UNSUPPORTED;
    if (!finite_positive(k_scale) || !finite_positive(v_scale)) return GBATTN_ERR_SCALE;
    if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_out) || !aligned16(v_out) ||
        (reinterpret_cast<uintptr_t>(page_table) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t in_bytes = static_cast<size_t>(num_phys_pages) * page_size * Hkv * D;
    const size_t out_bytes = static_cast<size_t>(kv_len) * Hkv * D * 2;
    const size_t tab_bytes = static_cast<size_t>((kv_len + page_size - 1) / page_size) * 4;
    const void* outs[2] = {k_out, v_out};
    for (const void* o : outs) {
        if (overlaps(o, out_bytes, k_pages, in_bytes) || overlaps(o, out_bytes, v_pages, in_bytes) ||
            overlaps(o, out_bytes, page_table, tab_bytes))
            return GBATTN_ERR_ALIAS;
    }
    if (overlaps(k_out, out_bytes, v_out, out_bytes)) return GBATTN_ERR_ALIAS;

    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    const long long total = static_cast<long long>(kv_len) * Hkv * (D / 8);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = static_cast<long long>(dev.num_sms) * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool half_scale = is_fp16_value(k_scale) && is_fp16_value(v_scale);
    const __half2 ks2 = __float2half2_rn(k_scale), vs2 = __float2half2_rn(v_scale);
    auto log2_exact = [](long long x) {   // log2 of a power of two, else -1
        if (x <= 0 || (x & (x - 1)) != 0) return -1;
        int l = 0;
        while ((1LL << l) < x) ++l;
        return l;
    };
    BridgeGeom q{page_size, Hkv, D, static_cast<int>(log2_exact(static_cast<long long>(Hkv) * (D / 8))),
                 static_cast<int>(log2_exact(D / 8)), static_cast<int>(log2_exact(page_size))};
    const bool pow2 = q.log_ppt >= 0 && q.log_cpr >= 0 && q.log_page >= 0;
    const unsigned nb = static_cast<unsigned>(blocks);
    __half* ko = static_cast<__half*>(k_out);
    __half* vo = static_cast<__half*>(v_out);
    if (half_scale && pow2)
        e4m3_bridge_kernel<true, true><<<nb, threads, 0, s>>>(k_pages, v_pages, page_table, num_phys_pages,
                                                               kv_len, q, k_scale, v_scale, ks2, vs2, ko, vo, dev.status);
    else if (half_scale)
        e4m3_bridge_kernel<true, false><<<nb, threads, 0, s>>>(k_pages, v_pages, page_table, num_phys_pages,
                                                                kv_len, q, k_scale, v_scale, ks2, vs2, ko, vo, dev.status);
    else if (pow2)
        e4m3_bridge_kernel<false, true><<<nb, threads, 0, s>>>(k_pages, v_pages, page_table, num_phys_pages,
                                                                kv_len, q, k_scale, v_scale, ks2, vs2, ko, vo, dev.status);
    else
        e4m3_bridge_kernel<false, false><<<nb, threads, 0, s>>>(k_pages, v_pages, page_table, num_phys_pages,
                                                                 kv_len, q, k_scale, v_scale, ks2, vs2, ko, vo, dev.status);
    count_launches(1);
    return launch_status();
}
