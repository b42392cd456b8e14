// VSA key-cube selection ("Integrate H3 SM70 execution, metrics and VSA
// diagnostics", Purpose: top-k = 64; FastVideo compare view,
// minimax_h3_fusions/query_pool.py and key_quant.py: FP32 tile means = FP32 sum
// divided by the token count).
//
// Two kernels:
//  1. vsa_pool_kernel: FP32 cube means of Q and K.  Each thread owns 8
//     consecutive channels of one cube and adds the cube's real tokens (all 64,
//     or the first valid-count slots of a boundary cube) in token order with
//     FP32 rounding after every addition, then divides by the count (correctly
//     rounded).  Video tokens start after `prefix` prefix tokens, which take no
//     part.  HBM-bound: Q and K are read once with 16-byte loads.
//  2. vsa_score_topk_kernel: 16 query cubes per CTA against all key cubes,
//     register-tiled (1 query x 4 keys per thread) with operands staged
//     d-major in shared memory.  Every score is an FP32 sum over d = 0..D-1, in
//     order, of FP32 products (no fused multiply-add, so both the product and the
//     sum are rounded).  The k-th largest score of a row is found with a 32-step
//     bitwise search on order-preserving integer keys; equal scores at the
//     threshold are taken from the lowest cube index up; the selection is
//     written in ascending cube order.
#include <cuda_fp16.h>

#include <mutex>

#include "host.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kMaxChunks = 32;      // 32-key chunks per row: supports up to 1024 cubes per head

__global__ void __launch_bounds__(kPoolThreads) vsa_pool_kernel(
    const __half* __restrict__ q, const __half* __restrict__ k, long long n_bh, int n_cubes,
    long long seq, int prefix, int D, int block, const int32_t* __restrict__ cube_valid,
    uint32_t* status, float* __restrict__ qm, float* __restrict__ km) {
    const __half* x = blockIdx.y == 0 ? q : k;
    float* out = blockIdx.y == 0 ? qm : km;
    const int groups = D >> 3;   // 8 channels per thread
    const long long gid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (gid >= n_bh * n_cubes * groups) return;
    long long cube, bh;                             // cube = bh * n_cubes + c
    int g, c;
    if (gid < (1LL << 31)) {                        // 32-bit index arithmetic when it fits
        const uint32_t gi = static_cast<uint32_t>(gid), cu = gi / static_cast<uint32_t>(groups);
        g = static_cast<int>(gi - cu * groups);
        const uint32_t b32 = cu / static_cast<uint32_t>(n_cubes);
        c = static_cast<int>(cu - b32 * n_cubes);
        cube = cu;
        bh = b32;
    } else {
        cube = gid / groups;
        g = static_cast<int>(gid - cube * groups);
        bh = cube / n_cubes;
        c = static_cast<int>(cube - bh * n_cubes);
    }
    // Real tokens of the cube: its first `count` slots (boundary cubes are padded).
    int count = block;
    if (cube_valid) {
        count = cube_valid[c];
        if (count < 1 || count > block) {
            if (g == 0 && bh == 0 && blockIdx.y == 0) atomicOr(status, kDevBadIndex);
            count = count < 1 ? 1 : block;
        }
    }
    const __half* base = x + (bh * seq + prefix + static_cast<long long>(c) * block) * D + g * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll 8
    for (int t = 0; t < count; ++t) {
        const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(base + static_cast<long long>(t) * D));
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            acc[2 * e] = __fadd_rn(acc[2 * e], f.x);
            acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], f.y);
        }
    }
    const float cnt = static_cast<float>(count);
    float4 lo, hi;
    lo.x = __fdiv_rn(acc[0], cnt); lo.y = __fdiv_rn(acc[1], cnt);
    lo.z = __fdiv_rn(acc[2], cnt); lo.w = __fdiv_rn(acc[3], cnt);
    hi.x = __fdiv_rn(acc[4], cnt); hi.y = __fdiv_rn(acc[5], cnt);
    hi.z = __fdiv_rn(acc[6], cnt); hi.w = __fdiv_rn(acc[7], cnt);
    float4* dst = reinterpret_cast<float4*>(out + cube * D + g * 8);
    dst[0] = lo;
    dst[1] = hi;
}

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kSelQ = 16;        // query cubes per CTA (about 75 KB of shared memory: 3 CTAs per SM)
constexpr int kSelKB = 64;       // key cubes per staged block
constexpr int kSelThreads = 256;
constexpr int kSelD = 128;

constexpr size_t sel_smem_bytes(int NC) {
    return (static_cast<size_t>(kSelD) * kSelQ + static_cast<size_t>(kSelD) * (kSelKB + 4) +
            static_cast<size_t>(kSelQ) * (NC + 1)) * sizeof(float);
}

// grid: (ceil(NC / kSelQ), B*H); block: kSelThreads; dynamic smem sel_smem_bytes(NC).
// Scores for 16 query cubes x all NC key cubes, each an FP32 sum over d in order of
// FP32 products (no FMA): thread (ty, tx) accumulates query ty against keys
// 4tx..4tx+3 of each 64-key block with both operands staged d-major.  Then each
// warp selects the top-k of two query rows; CH = 32-key chunks per row.
template <int CH>
__global__ void __launch_bounds__(kSelThreads) vsa_score_topk_kernel(
    const float* __restrict__ qm, const float* __restrict__ km, int NC, int topk,
    int32_t* __restrict__ idx) {
    extern __shared__ float sm[];
    float* sq = sm;                                   // [D][kSelQ]
    float* sk = sq + kSelD * kSelQ;                   // [D][kSelKB + 4]
    float* ss = sk + kSelD * (kSelKB + 4);            // [kSelQ][NC + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.y, q0 = blockIdx.x * kSelQ;
    const float* qbase = qm + static_cast<long long>(bh) * NC * kSelD;
    const float* kbase = km + static_cast<long long>(bh) * NC * kSelD;
    const int SK = kSelKB + 4, SS = NC + 1;
    // Stage Q (32 x 128) d-major: every thread issues its four 16-byte loads first.
    {
        float4 v[kSelQ * kSelD / 4 / kSelThreads];
#pragma unroll
        for (int r = 0; r < kSelQ * kSelD / 4 / kSelThreads; ++r) {
            const int i = tid + r * kSelThreads, q = i / (kSelD / 4), d4 = i % (kSelD / 4);
            v[r] = (q0 + q < NC) ? *reinterpret_cast<const float4*>(qbase + static_cast<long long>(q0 + q) * kSelD + 4 * d4)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int r = 0; r < kSelQ * kSelD / 4 / kSelThreads; ++r) {
            const int i = tid + r * kSelThreads, q = i / (kSelD / 4), d4 = i % (kSelD / 4);
            sq[(4 * d4 + 0) * kSelQ + q] = v[r].x;
            sq[(4 * d4 + 1) * kSelQ + q] = v[r].y;
            sq[(4 * d4 + 2) * kSelQ + q] = v[r].z;
            sq[(4 * d4 + 3) * kSelQ + q] = v[r].w;
        }
    }
    const int ty = tid >> 4, tx = tid & 15;
    // Key staging: lane = key (32 keys per warp), each lane one 32-byte sector of
    // 8 consecutive dims per item, so the d-major stores of a warp fill 32
    // consecutive words of one row (no bank conflicts) and every sector loaded
    // is used whole.  Warp w takes keys 32*(w&1) .. +31 and dim groups (w>>1) + 4r.
    const int sk_key = lane + 32 * (warp & 1), sk_g0 = warp >> 1;
    constexpr int kItems = kSelKB * kSelD / 8 / kSelThreads;   // 4
    for (int kb = 0; kb < NC; kb += kSelKB) {
        float4 v[2 * kItems];
        const bool live = kb + sk_key < NC;
        const float* krow = kbase + static_cast<long long>(kb + sk_key) * kSelD;
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int g = sk_g0 + 4 * r;   // dims 8g .. 8g+7
            v[2 * r] = live ? *reinterpret_cast<const float4*>(krow + 8 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[2 * r + 1] = live ? *reinterpret_cast<const float4*>(krow + 8 * g + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int g = sk_g0 + 4 * r;
            float* col = sk + (8 * g) * SK + sk_key;
            col[0 * SK] = v[2 * r].x;
            col[1 * SK] = v[2 * r].y;
            col[2 * SK] = v[2 * r].z;
            col[3 * SK] = v[2 * r].w;
            col[4 * SK] = v[2 * r + 1].x;
            col[5 * SK] = v[2 * r + 1].y;
            col[6 * SK] = v[2 * r + 1].z;
            col[7 * SK] = v[2 * r + 1].w;
        }
        __syncthreads();
        float acc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = 0.0f;
#pragma unroll 8
        for (int d = 0; d < kSelD; ++d) {
            const float qv = sq[d * kSelQ + ty];
            const float4 kv = *reinterpret_cast<const float4*>(sk + d * SK + 4 * tx);
            acc[0] = __fadd_rn(acc[0], __fmul_rn(qv, kv.x));
            acc[1] = __fadd_rn(acc[1], __fmul_rn(qv, kv.y));
            acc[2] = __fadd_rn(acc[2], __fmul_rn(qv, kv.z));
            acc[3] = __fadd_rn(acc[3], __fmul_rn(qv, kv.w));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (kb + 4 * tx + j < NC) ss[ty * SS + kb + 4 * tx + j] = acc[j];
    }
    __syncthreads();

    // Top-k: warp w owns query rows 2w, 2w+1.  Key c*32 + lane -> key[c].
    const int nchunks = (NC + 31) / 32;
    const uint32_t lt = (1u << lane) - 1u;
    for (int r = 0; r < kSelQ / (kSelThreads / 32); ++r) {
        const int ql = warp * (kSelQ / (kSelThreads / 32)) + r;
        const int qc = q0 + ql;
        if (qc >= NC) break;
        uint32_t key[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int kc = c * 32 + lane;
            key[c] = (c < nchunks && kc < NC) ? order_key(ss[ql * SS + kc]) : 0u;   // 0: below any score
        }
        // Threshold: the largest T such that at least topk keys are >= T.
        uint32_t T = 0;
#pragma unroll 1
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int cnt = 0;
#pragma unroll
            for (int c = 0; c < CH; ++c) cnt += (c < nchunks && key[c] >= cand) ? 1 : 0;
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            if (cnt >= topk) T = cand;
        }
        int greater = 0;
#pragma unroll
        for (int c = 0; c < CH; ++c) greater += (c < nchunks && key[c] > T) ? 1 : 0;
        greater = __reduce_add_sync(0xffffffffu, greater);
        int need = topk - greater;            // equal-to-threshold scores still to take
        int32_t* out = idx + (static_cast<long long>(bh) * NC + qc) * topk;
        int base = 0;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            if (c < nchunks) {
                const bool valid = c * 32 + lane < NC;
                const bool eq = valid && key[c] == T;
                const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
                const int take = min(need, __popc(eqm));
                const bool sel = valid && (key[c] > T || (eq && __popc(eqm & lt) < take));
                need -= take;
                const uint32_t selm = __ballot_sync(0xffffffffu, sel);
                if (sel) out[base + __popc(selm & lt)] = c * 32 + lane;
                base += __popc(selm);
            }
        }
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" size_t vsa_select_workspace_size(int B, int H, int S, int D, int block) {
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return 0;
    const size_t nc = static_cast<size_t>(S / block);
    return 2 * static_cast<size_t>(B) * H * nc * D * sizeof(float);
}

extern "C" int vsa_select_blocks(const void* q, const void* k, int B, int H, int S, int D,
                                 int block, int topk, int prefix, const int32_t* cube_valid,
                                 int32_t* idx, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    if (!q || !k || !idx) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || S <= 0 || topk <= 0 || prefix < 0 || prefix >= S)
        return GBATTN_ERR_SHAPE;
    if (D != 128 || block != 64) return GBATTN_ERR_UNSUPPORTED;
    if ((S - prefix) % block != 0) return GBATTN_ERR_SHAPE;
    const int NC = (S - prefix) / block;
    if (NC > kMaxChunks * 32 || topk > NC) return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    const size_t need = vsa_select_workspace_size(B, H, S, D, block);
    if (!workspace || workspace_bytes < need) return GBATTN_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(cube_valid) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t in_bytes = static_cast<size_t>(B) * H * S * D * 2;
    const size_t idx_bytes = static_cast<size_t>(B) * H * NC * topk * 4;
    if (overlaps(idx, idx_bytes, q, in_bytes) || overlaps(idx, idx_bytes, k, in_bytes) ||
        overlaps(workspace, need, q, in_bytes) || overlaps(workspace, need, k, in_bytes) ||
        overlaps(workspace, need, idx, idx_bytes))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* qm = static_cast<float*>(workspace);
    float* km = qm + static_cast<size_t>(B) * H * NC * D;
    const long long n_bh = static_cast<long long>(B) * H;
    const long long pool_threads = n_bh * NC * (D / 8);
    dim3 pgrid(static_cast<unsigned>((pool_threads + kPoolThreads - 1) / kPoolThreads), 2);
    vsa_pool_kernel<<<pgrid, kPoolThreads, 0, s>>>(static_cast<const __half*>(q),
                                                   static_cast<const __half*>(k), n_bh, NC, S,
                                                   prefix, D, block, cube_valid, dev.status, qm,
                                                   km);
    static std::once_flag attr_once[64];
    if (dev.device >= 0 && dev.device < 64)
        std::call_once(attr_once[dev.device], [] {
            cudaFuncSetAttribute(vsa_score_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sel_smem_bytes(16 * 32)));
            cudaFuncSetAttribute(vsa_score_topk_kernel<kMaxChunks>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sel_smem_bytes(kMaxChunks * 32)));
        });
    dim3 sgrid((NC + kSelQ - 1) / kSelQ, B * H);
    if (NC <= 16 * 32)
        vsa_score_topk_kernel<16><<<sgrid, kSelThreads, sel_smem_bytes(NC), s>>>(qm, km, NC, topk, idx);
    else
        vsa_score_topk_kernel<kMaxChunks><<<sgrid, kSelThreads, sel_smem_bytes(NC), s>>>(qm, km, NC, topk,
                                                                                       idx);
    count_launches(2);
    return launch_status();
}

// ------------------------------------------------------------------ query-cube pairing
//
// The sparse attention kernel processes two query cubes per CTA over the union
// of their selected key cubes; every key cube only one of the two selected is
// wasted work for the other.  Pairing cubes whose selections overlap most
// cuts that waste.  One CTA per head:
//   1. each cube's selection as a bitset over key cubes;
//   2. the overlap of every cube with the cubes up to kPairWindow index
//      positions away (neighbours in the cube grid are close in cube index);
//   3. kPairRounds rounds of "mutual best": every unpaired cube picks its
//      unpaired window partner of largest overlap (ties to the lower index);
//      two cubes that pick each other are paired;
//   4. the cubes still unpaired are paired in index order.
// The pairs are written in order of their first cube.  Any pairing gives the
// same attention result (up to summation order); this one only saves work.
namespace gbattn {
namespace {
constexpr int kPairThreads = 1024;   // one thread per cube
constexpr int kPairWindow = 32;
constexpr int kPairRounds = 4;
constexpr int kPairMaxCubes = 1024;
constexpr int kPairMaxWords = kPairMaxCubes / 32;

size_t pair_smem_bytes(int nc) {
    const int words = (nc + 31) / 32;
    return static_cast<size_t>(nc) * words * 4 + static_cast<size_t>(nc) * kPairWindow +
           static_cast<size_t>(nc) * 2 * 3 + 64 * 4;
}

// Exclusive prefix sum of v over the block (one value per thread); returns the
// total through *total.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, sh);
        if (lane >= sh) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kPairThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, sh);
            if (lane >= sh) t += y;
        }
        warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    *total = warp_tot[kPairThreads / 32 - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kPairThreads) vsa_pair_kernel(const int32_t* __restrict__ idx,
                                                                int nc, int topk,
                                                                int32_t* __restrict__ pairs) {
    extern __shared__ uint32_t psm[];
    __shared__ int warp_tot[32];
    const int words = (nc + 31) / 32;
    uint32_t* bits = psm;                                            // [words][nc] (transposed)
    uint8_t* ov = reinterpret_cast<uint8_t*>(bits + static_cast<size_t>(nc) * words);  // [W][nc]
    int16_t* partner = reinterpret_cast<int16_t*>(ov + static_cast<size_t>(nc) * kPairWindow);
    int16_t* best = partner + nc;
    int16_t* list = best + nc;
    const long long bh = blockIdx.x;
    const int32_t* sel = idx + bh * nc * static_cast<long long>(topk);
    const int a = threadIdx.x;
    const bool live = a < nc;

    for (int i = a; i < nc * words; i += kPairThreads) bits[i] = 0u;
    if (live) partner[a] = -1;
    __syncthreads();
    for (int e = a; e < nc * topk; e += kPairThreads) {
        const int c = e / topk;
        const int kc = sel[e];
        if (kc >= 0 && kc < nc) atomicOr(&bits[(kc >> 5) * nc + c], 1u << (kc & 31));
    }
    __syncthreads();
    // overlap of a and a + d (d = 1..W) at ov[(d - 1) * nc + a]
    if (live) {
        uint32_t mine[kPairMaxWords];
#pragma unroll
        for (int w = 0; w < kPairMaxWords; ++w) mine[w] = w < words ? bits[w * nc + a] : 0u;
        for (int d = 1; d <= kPairWindow; ++d) {
            const int b = a + d;
            int n = 0;
            if (b < nc) {
#pragma unroll
                for (int w = 0; w < kPairMaxWords; ++w)
                    if (w < words) n += __popc(mine[w] & bits[w * nc + b]);
            }
            ov[(d - 1) * nc + a] = static_cast<uint8_t>(n > 255 ? 255 : n);
        }
    }
    __syncthreads();
    for (int r = 0; r < kPairRounds; ++r) {
        int bb = -1;
        if (live && partner[a] < 0) {
            int bw = -1;
            for (int d = kPairWindow; d >= 1; --d) {      // b = a - d, ascending b
                const int b = a - d;
                if (b < 0 || partner[b] >= 0) continue;
                const int w = ov[(d - 1) * nc + b];
                if (w > bw) { bw = w; bb = b; }
            }
            for (int d = 1; d <= kPairWindow; ++d) {      // b = a + d, ascending b
                const int b = a + d;
                if (b >= nc) break;
                if (partner[b] >= 0) continue;
                const int w = ov[(d - 1) * nc + a];
                if (w > bw) { bw = w; bb = b; }
            }
        }
        if (live) best[a] = static_cast<int16_t>(bb);
        __syncthreads();
        if (live && partner[a] < 0 && bb >= 0 && best[bb] == a) partner[a] = static_cast<int16_t>(bb);
        __syncthreads();
    }
    // the cubes still unpaired pair up in index order
    int n_left = 0;
    const bool left = live && partner[a] < 0;
    const int lr = block_exclusive_scan(left ? 1 : 0, warp_tot, &n_left);
    if (left) list[lr] = static_cast<int16_t>(a);
    __syncthreads();
    if (left && (lr & 1) == 0 && lr + 1 < n_left) {
        const int b = list[lr + 1];
        partner[a] = static_cast<int16_t>(b);
        partner[b] = static_cast<int16_t>(a);
    }
    __syncthreads();
    // pairs in order of their first cube
    const int pb = live ? partner[a] : 0;
    const bool first = live && (pb > a || pb < 0);
    int n_out = 0;
    const int p = block_exclusive_scan(first ? 1 : 0, warp_tot, &n_out);
    if (first) {
        int32_t* out = pairs + (bh * static_cast<long long>((nc + 1) / 2) + p) * 2;
        out[0] = a;
        out[1] = pb > a ? pb : -1;
    }
}

}  // namespace
}  // namespace gbattn

extern "C" int vsa_pair_query_cubes(const int32_t* idx, int B, int H, int n_cubes, int topk,
                                    int32_t* pairs, void* stream) {
    if (!idx || !pairs) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || n_cubes <= 0 || topk <= 0 || topk > n_cubes) return GBATTN_ERR_SHAPE;
    if (n_cubes > kPairMaxCubes || static_cast<long long>(B) * H > 0x7FFFFFFFLL)
        return GBATTN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(pairs) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t ib = static_cast<size_t>(B) * H * n_cubes * topk * 4;
    const size_t pb = static_cast<size_t>(B) * H * ((n_cubes + 1) / 2) * 2 * 4;
    if (overlaps(pairs, pb, idx, ib)) return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    const size_t smem = pair_smem_bytes(n_cubes);
    static std::once_flag once[64];
    if (dev.device >= 0 && dev.device < 64)
        std::call_once(once[dev.device], [] {
            cudaFuncSetAttribute(vsa_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(pair_smem_bytes(kPairMaxCubes)));
        });
    vsa_pair_kernel<<<static_cast<unsigned>(static_cast<long long>(B) * H), kPairThreads, smem,
                      static_cast<cudaStream_t>(stream)>>>(idx, n_cubes, topk, pairs);
    count_launches(1);
    return launch_status();
}

// ------------------------------------------------------------------ no-allocation variant
//
// Some callers cannot allocate device memory when they call this library: a
// plugin inside a host program that fixed its memory budget at start-up and
// forbids later allocations, code whose device memory is entirely owned by a
// pool it cannot reach from here, or a latency-critical loop in which a
// cudaMalloc (which may synchronise the device) is not acceptable.  For them,
// vsa_select_blocks_noalloc runs the same selection with its scratch (the FP32
// pooled cube means) in a fixed array of kNoAllocScratchBytes that lives in
// this library's device image.  Every GPU that loads the library holds the
// array until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_select_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return GBATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GBATTN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GBATTN_OK;
}
}  // namespace

extern "C" int vsa_select_blocks_noalloc(const void* q, const void* k, int B, int H, int S, int D,
                                         int block, int topk, int prefix,
                                         const int32_t* cube_valid, int32_t* idx, void* stream) {
    if (!q || !k || !idx) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return GBATTN_ERR_SHAPE;
    const size_t need = vsa_select_workspace_size(B, H, S, D, block);
    if (need > kNoAllocScratchBytes) return GBATTN_ERR_WORKSPACE;   // sizes beyond the fixed scratch
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != GBATTN_OK) return rc;
    // The pool kernel overwrites every scratch byte it later reads, so the
    // previous call's contents need no clearing.
    return vsa_select_blocks(q, k, B, H, S, D, block, topk, prefix, cube_valid, idx, scratch,
                             kNoAllocScratchBytes, stream);
}
