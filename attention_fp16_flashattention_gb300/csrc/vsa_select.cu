// VSA key-cube selection ("Integrate H3 SM70 execution, metrics and VSA
// diagnostics", Purpose: top-k = 64; FastVideo compare view,
// minimax_h3_fusions/query_pool.py and key_quant.py: FP32 tile means = FP32 sum
// divided by the token count).
//
// Four kernels, each launched as a programmatic dependent of the one before:
//  1. vsa_pool_kernel: FP32 cube means of Q and K.  Each thread owns 8
//     consecutive channels of one cube and adds the cube's real tokens (all 64,
//     or the first valid-count slots of a boundary cube) in token order with
//     FP32 rounding after every addition, then divides by the count (correctly
//     rounded).  Video tokens start after `prefix` prefix tokens, which take no
//     part.  HBM-bound: Q and K are read once with 16-byte loads.  It also
//     writes each mean's Euclidean norm.
//  2. vsa_score_kernel: FP32 scores of every (query cube, key cube) pair, a
//     batched FFMA matrix product in 128 x 128 tiles.
//  3. vsa_topk_kernel: the selection ranks key cubes by the EXACT dot product
//     of the FP32 means.  One warp per query cube: the FP32 scores with a
//     rigorous error bound decide almost every key; the few keys whose FP32
//     score lies too close to the k-th value are ranked by exact integer scores
//     (limbs of the means on their 2^-53 grid).  Ties go to the lower cube
//     index; the selection is written in ascending cube order.
//  4. the same kernel in its fallback form: rows with more undecided keys than
//     one warp's in-place buffer holds (many equal scores) are ranked the same
//     way with room for every key.
#include <cuda_fp16.h>

#include <algorithm>
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
    uint32_t* status, float* __restrict__ qm, float* __restrict__ km, float* __restrict__ qn,
    float* __restrict__ kn, const __half* __restrict__ v, float* __restrict__ vm) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // score kernel may be placed
    // blockIdx.y: 0 = Q, 1 = K, 2 = V (the coarse branch's pooled values, no norm)
    const __half* x = blockIdx.y == 0 ? q : blockIdx.y == 1 ? k : v;
    float* out = blockIdx.y == 0 ? qm : blockIdx.y == 1 ? km : vm;
    float* out_n = blockIdx.y == 0 ? qn : blockIdx.y == 1 ? kn : nullptr;
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
    // Euclidean norm of the cube mean (it scales the score error bound): the
    // cube's 16 channel groups are 16 aligned lanes of one warp.
    float n2 = lo.x * lo.x + lo.y * lo.y + lo.z * lo.z + lo.w * lo.w + hi.x * hi.x + hi.y * hi.y +
               hi.z * hi.z + hi.w * hi.w;
    const unsigned grp = 0xFFFFu << (threadIdx.x & 16u);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) n2 += __shfl_xor_sync(grp, n2, off);
    if (g == 0 && out_n) out_n[cube] = sqrtf(n2);
}

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ---------------------------------------------------------------- exact scores
//
// Cube means of FP16 data are integer multiples of 2^-53 below 2^16 in
// magnitude (an FP32 sum of FP16 values stays on the 2^-24 grid; a nonzero sum
// over at most 64 tokens divided by the count is at least 2^-30, whose 24-bit
// significand ends at 2^-53 or above).  So M = x * 2^53 is an integer below
// 2^69, three signed 23-bit limbs, and sum_d Mq[d] Mk[d] -- the score times
// 2^106 -- is an integer formed exactly from int64 sums of limb products
// (each below 2^46; 128 dims x 3 products per position stay below 2^55).

constexpr uint32_t kLimbMask = (1u << 23) - 1u;

struct ExactScore {
    long long top;            // sign-carrying leading digit (weight 2^92)
    unsigned long long mid;   // digits of weight 2^69, 2^46 (23 bits each)
    unsigned long long low;   // digits of weight 2^23, 2^0
};

__device__ __forceinline__ bool exact_greater(const ExactScore& a, const ExactScore& b) {
    if (a.top != b.top) return a.top > b.top;
    if (a.mid != b.mid) return a.mid > b.mid;
    return a.low > b.low;
}
__device__ __forceinline__ bool exact_equal(const ExactScore& a, const ExactScore& b) {
    return a.top == b.top && a.mid == b.mid && a.low == b.low;
}

// The three limbs of x * 2^53 with x's sign.  Values off the grid (impossible
// for cube means of FP16 data) lose their bits below 2^-53; non-finite values
// count as 0 (their selection is unspecified, but stays a valid index list).
__device__ __forceinline__ void grid_limbs(float x, int& a0, int& a1, int& a2) {
    const uint32_t u = __float_as_uint(x);
    const int E = static_cast<int>((u >> 23) & 0xFFu);
    const uint32_t m = E == 255 ? 0u : ((u & 0x7FFFFFu) | (E ? 0x800000u : 0u));
    const int sh = (E ? E : 1) - 150 + 53;   // |x| * 2^53 = m * 2^sh
    auto limb = [&](int s) -> int {
        if (s >= 23 || s <= -32) return 0;
        const uint64_t v = s >= 0 ? (static_cast<uint64_t>(m) << s) : static_cast<uint64_t>(m >> -s);
        return static_cast<int>(v & kLimbMask);
    };
    const int sg = (u >> 31) ? -1 : 1;
    a0 = sg * limb(sh);
    a1 = sg * limb(sh - 23);
    a2 = sg * limb(sh - 46);
}

// Exact score of one query row against key row `krow` (128 FP32 means in global
// memory), by the whole warp: lane l takes dims 4l..4l+3, whose query limbs it
// holds in qa.  Every lane returns the same value.
__device__ __forceinline__ ExactScore exact_score_warp(const int (&qa)[4][3], const float* krow) {
    const int lane = threadIdx.x & 31;
    const float4 kv = *reinterpret_cast<const float4*>(krow + 4 * lane);
    const float kf[4] = {kv.x, kv.y, kv.z, kv.w};
    long long c[5] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int b0, b1, b2;
        grid_limbs(kf[e], b0, b1, b2);
        c[0] += static_cast<long long>(qa[e][0]) * b0;
        c[1] += static_cast<long long>(qa[e][0]) * b1 + static_cast<long long>(qa[e][1]) * b0;
        c[2] += static_cast<long long>(qa[e][0]) * b2 + static_cast<long long>(qa[e][1]) * b1 +
                static_cast<long long>(qa[e][2]) * b0;
        c[3] += static_cast<long long>(qa[e][1]) * b2 + static_cast<long long>(qa[e][2]) * b1;
        c[4] += static_cast<long long>(qa[e][2]) * b2;
    }
#pragma unroll
    for (int p = 0; p < 5; ++p)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c[p] += __shfl_xor_sync(0xffffffffu, c[p], off);
    // carry into 23-bit digits (arithmetic shifts are floor divisions)
    long long t = c[0];
    const unsigned long long d0 = static_cast<unsigned long long>(t) & kLimbMask;
    t = (t >> 23) + c[1];
    const unsigned long long d1 = static_cast<unsigned long long>(t) & kLimbMask;
    t = (t >> 23) + c[2];
    const unsigned long long d2 = static_cast<unsigned long long>(t) & kLimbMask;
    t = (t >> 23) + c[3];
    const unsigned long long d3 = static_cast<unsigned long long>(t) & kLimbMask;
    ExactScore r;
    r.top = (t >> 23) + c[4];
    r.mid = (d3 << 23) | d2;
    r.low = (d1 << 23) | d0;
    return r;
}

// Candidate buffer of one warp: the keys whose place around the k-th score the
// FP32 scores cannot decide, with their exact scores, and the chosen keys as
// bits (at most 1024 keys).
template <int CAP>
struct Cands {
    long long top[CAP];
    unsigned long long mid[CAP];
    unsigned long long low[CAP];
    int key[CAP];
    uint32_t chosen[32];
    uint32_t hist[256];   // selection histogram
    uint32_t list[32];    // keys of the bucket holding the k-th key
};

// ---------------------------------------------------------------- row selection
//
// One warp selects the topk keys of one query row (key c*32 + lane in chunk c).
// Scores s are FP32 with |s - exact| <= e for every key (e covers the FP32
// evaluation error of the dot product).  With s_k and s_k1 the k-th and
// (k+1)-th largest FP32 scores, a key with s < s_k - 2e is below k keys
// whose exact scores are all >= s_k - e (certainly out), and a key with
// s > s_k1 + 2e lies above the exact (k+1)-th score (certainly in).  The keys
// left between are ranked by their exact scores, ties to the lower index.
template <int CH>
struct RowClass {
    uint32_t in_m[CH];    // ballot masks per chunk
    uint32_t unc_m[CH];
    int n_in, n_unc;
};

// The k-th largest of the row's order keys by radix selection: four passes
// over 8-bit digits from the top, each a histogram of the keys that match the
// digits chosen so far, then a suffix scan over the 256 bins (8 per lane) for
// the digit holding the k-th key.
template <int CH>
__device__ __forceinline__ uint32_t kth_largest_key(const uint32_t (&key)[CH], const bool (&live)[CH],
                                                    int k, uint32_t* hist) {
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0, pmask = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
#pragma unroll
        for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0u;
        __syncwarp();
#pragma unroll
        for (int c = 0; c < CH; ++c)
            if (live[c] && (key[c] & pmask) == prefix) atomicAdd(&hist[(key[c] >> shift) & 0xFFu], 1u);
        __syncwarp();
        const uint4 b0 = *reinterpret_cast<const uint4*>(hist + lane * 8);
        const uint4 b1 = *reinterpret_cast<const uint4*>(hist + lane * 8 + 4);
        const uint32_t bins[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) mine += bins[i];
        uint32_t suf = mine;   // keys in lanes >= this lane (digits >= 8 * lane)
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf += y;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, suf >= static_cast<uint32_t>(k));
        const int L = 31 - __clz(hit);   // the highest lane whose suffix still holds k keys
        uint32_t above = __shfl_sync(0xffffffffu, suf - mine, L);   // keys in higher lanes
        int digit = 0;
        uint32_t gt = 0;
        if (lane == L) {
            uint32_t run = above;
            bool found = false;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (!found && run + bins[i] >= static_cast<uint32_t>(k)) {
                    digit = 8 * lane + i;
                    gt = run;
                    found = true;
                }
                run += bins[i];
            }
        }
        digit = __shfl_sync(0xffffffffu, digit, L);
        gt = __shfl_sync(0xffffffffu, gt, L);
        prefix |= static_cast<uint32_t>(digit) << shift;
        pmask |= 0xFFu << shift;
        k -= static_cast<int>(gt);
        __syncwarp();
    }
    return prefix;
}

// The k-th largest order key in one histogram pass when the scores are spread
// out: 256 equal buckets between the row's smallest and largest FP32 score
// (bucket = floor((s - min) * 256 / (max - min)), a non-decreasing function of
// s, so the buckets are in score order), a suffix scan over the buckets finds
// the one holding the k-th key, and if it holds at most 32 keys they are
// ranked directly.  Otherwise (many equal or clustered scores, or non-finite
// ones) the radix selection decides.
template <int CH>
__device__ __forceinline__ uint32_t kth_largest_key_fast(const float (&s)[CH], const uint32_t (&key)[CH],
                                                         const bool (&live)[CH], int k,
                                                         uint32_t* hist, uint32_t* list) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int c = 0; c < CH; ++c)
        if (live[c]) {
            kmin = min(kmin, key[c]);
            kmax = max(kmax, key[c]);
        }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    const float smin = key_float(kmin), smax = key_float(kmax);
    const float inv = 256.0f / (smax - smin);
    if (!(inv <= 3.0e38f)) return kth_largest_key<CH>(key, live, k, hist);   // equal, inf or nan
    auto bucket_of = [&](float x) { return min(255, __float2int_rz((x - smin) * inv)); };
#pragma unroll
    for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0u;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < CH; ++c)
        if (live[c]) atomicAdd(&hist[bucket_of(s[c])], 1u);
    __syncwarp();
    const uint4 b0 = *reinterpret_cast<const uint4*>(hist + lane * 8);
    const uint4 b1 = *reinterpret_cast<const uint4*>(hist + lane * 8 + 4);
    const uint32_t bins[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine += bins[i];
    uint32_t suf = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += y;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, suf >= static_cast<uint32_t>(k));
    const int L = 31 - __clz(hit);
    const uint32_t above = __shfl_sync(0xffffffffu, suf - mine, L);
    int bucket = 0;
    uint32_t gt = 0, nb = 0;
    if (lane == L) {
        uint32_t run = above;
        bool found = false;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (!found && run + bins[i] >= static_cast<uint32_t>(k)) {
                bucket = 8 * lane + i;
                gt = run;
                nb = bins[i];
                found = true;
            }
            run += bins[i];
        }
    }
    bucket = __shfl_sync(0xffffffffu, bucket, L);
    gt = __shfl_sync(0xffffffffu, gt, L);
    nb = __shfl_sync(0xffffffffu, nb, L);
    __syncwarp();
    if (nb > 32) return kth_largest_key<CH>(key, live, k, hist);
    // the bucket's keys, then the one with rank k - gt among them (ties counted)
    int base = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const bool in = live[c] && bucket_of(s[c]) == bucket;
        const uint32_t m = __ballot_sync(0xffffffffu, in);
        if (in) list[base + __popc(m & lt)] = key[c];
        base += __popc(m);
    }
    __syncwarp();
    const int kk = k - static_cast<int>(gt);
    const uint32_t mykey = lane < static_cast<int>(nb) ? list[lane] : 0u;
    int greater = 0, equal = 0;
    for (int j = 0; j < static_cast<int>(nb); ++j) {
        const uint32_t v = list[j];
        greater += v > mykey ? 1 : 0;
        equal += v == mykey ? 1 : 0;
    }
    const bool is_kth = lane < static_cast<int>(nb) && greater < kk && kk <= greater + equal;
    const uint32_t who = __ballot_sync(0xffffffffu, is_kth);
    const uint32_t T = __shfl_sync(0xffffffffu, mykey, __ffs(who) - 1);
    __syncwarp();
    return T;
}

template <int CH>
__device__ __forceinline__ void classify_row(const float (&s)[CH], int NC, int topk, float e,
                                             RowClass<CH>& rc, uint32_t* hist, uint32_t* list) {
    const int lane = threadIdx.x & 31;
    const int nchunks = (NC + 31) / 32;
    uint32_t key[CH];
    bool live[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        live[c] = c < nchunks && c * 32 + lane < NC;
        key[c] = live[c] ? order_key(s[c]) : 0u;
    }
    const uint32_t T = kth_largest_key_fast<CH>(s, key, live, topk, hist, list);
    int ge = 0;
    uint32_t below = 0;   // largest key value under T
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        if (live[c]) {
            ge += key[c] >= T ? 1 : 0;
            if (key[c] < T) below = max(below, key[c]);
        }
    }
    ge = __reduce_add_sync(0xffffffffu, ge);
    below = __reduce_max_sync(0xffffffffu, below);
    const uint32_t T1 = ge > topk ? T : below;          // the (k+1)-th largest key
    const float e2 = __fmul_ru(2.0f, e);
    const float thr_out = __fsub_rd(key_float(T), e2);
    const float thr_in = __fadd_ru(key_float(T1), e2);
    int n_in = 0, n_unc = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const bool in = live[c] && s[c] > thr_in;
        const bool unc = live[c] && !in && !(s[c] < thr_out);
        rc.in_m[c] = __ballot_sync(0xffffffffu, in);
        rc.unc_m[c] = __ballot_sync(0xffffffffu, unc);
        n_in += __popc(rc.in_m[c]);
        n_unc += __popc(rc.unc_m[c]);
    }
    rc.n_in = n_in;
    rc.n_unc = n_unc;
}

// Ranks the uncertain keys of a row by exact score and marks the best `need`
// in cb->chosen.  q_at(d) gives the row's query mean at dim d; kbase points at
// the key means of the head ([NC][128]).
template <int CH, int CAP, typename QAt>
__device__ __forceinline__ void resolve_exact(const RowClass<CH>& rc, int need, QAt q_at,
                                              const float* kbase, Cands<CAP>* cb) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    int base = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const uint32_t m = rc.unc_m[c];
        if ((m >> lane) & 1u) cb->key[base + __popc(m & lt)] = c * 32 + lane;
        base += __popc(m);
    }
    cb->chosen[lane] = 0u;
    int qa[4][3];
#pragma unroll
    for (int e = 0; e < 4; ++e) grid_limbs(q_at(4 * lane + e), qa[e][0], qa[e][1], qa[e][2]);
    __syncwarp();
    for (int i = 0; i < rc.n_unc; ++i) {
        const ExactScore x = exact_score_warp(qa, kbase + static_cast<long long>(cb->key[i]) * 128);
        if (lane == 0) {
            cb->top[i] = x.top;
            cb->mid[i] = x.mid;
            cb->low[i] = x.low;
        }
    }
    __syncwarp();
    for (int i = lane; i < rc.n_unc; i += 32) {
        const ExactScore xi{cb->top[i], cb->mid[i], cb->low[i]};
        const int ki = cb->key[i];
        int rank = 0;
        for (int v = 0; v < rc.n_unc; ++v) {
            const ExactScore xv{cb->top[v], cb->mid[v], cb->low[v]};
            rank += (exact_greater(xv, xi) || (exact_equal(xv, xi) && cb->key[v] < ki)) ? 1 : 0;
        }
        if (rank < need) atomicOr(&cb->chosen[ki >> 5], 1u << (ki & 31));
    }
    __syncwarp();
}

// Writes the row's selection (certainly-in keys plus the chosen uncertain keys)
// in ascending key order.
template <int CH, int CAP>
__device__ __forceinline__ void write_row(const RowClass<CH>& rc, const Cands<CAP>* cb, bool use_chosen,
                                          int NC, int topk, int32_t* out, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const int nchunks = (NC + 31) / 32;
    int base = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        if (c < nchunks) {
            const bool sel = ((rc.in_m[c] >> lane) & 1u) ||
                             (use_chosen && ((cb->chosen[c] >> lane) & 1u));
            const uint32_t m = __ballot_sync(0xffffffffu, sel);
            const int p = base + __popc(m & lt);
            if (sel && p < topk) out[p] = c * 32 + lane;
            base += __popc(m);
        }
    }
    if (base != topk && lane == 0) atomicOr(status, kDevBadIndex);   // never for finite inputs
}

// ---------------------------------------------------------------- score kernel
//
// Batched FP32 product S[bh] = Qm[bh] Km[bh]^T of the cube means ([NC][128]
// each), one 128 x 128 tile of S per CTA.  256 threads, each an 8 x 8 register
// tile (rows 4ty.., 64+4ty.., columns 4tx.., 64+4tx..); the two operand tiles
// pass through shared memory sixteen dims at a time, stored dim-major so that
// every operand read is a 16-byte load, with the next sixteen dims loaded into
// registers (two 16-byte loads per operand per thread) while the current ones
// are multiplied.  Every score is a sequence of FFMAs over d = 0..127, issued
// two scores at a time as packed FP32 pair FMAs (each lane an IEEE FMA with
// round to nearest, so the scores are those of scalar FFMAs).
// (Two CTAs fit on an SM.  A 4 x 8 thread tile with three CTAs per SM, for
// fewer idle SMs in the last wave, measured slower: 54 against 47 us.)
constexpr int kGT = 128;          // tile edge (query cubes x key cubes)
constexpr int kGK = 8;            // keys per stage of the coarse product
constexpr int kSK = 16;           // dims per stage of the score product
constexpr int kGThreads = 256;
constexpr int kGP = kGT + 4;      // shared-memory pitch (conflict-free transposing stores)
constexpr int kSelD = 128;

__host__ __device__ constexpr int score_ld(int NC) { return (NC + kGT - 1) / kGT * kGT; }

__global__ void __launch_bounds__(kGThreads, 2) vsa_score_kernel(const float* __restrict__ qm,
                                                                 const float* __restrict__ km,
                                                                 int NC, float* __restrict__ S) {
    __shared__ __align__(16) float As[2][kSK][kGP];
    __shared__ __align__(16) float Bs[2][kSK][kGP];
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the means come from the pool kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = threadIdx.x;
    const long long bh = blockIdx.z;
    const int m0 = blockIdx.y * kGT, n0 = blockIdx.x * kGT;
    const int LD = score_ld(NC);
    const float* A = qm + bh * NC * kSelD;
    const float* B = km + bh * NC * kSelD;
    // staging: thread t loads row lr, dims lk..lk+3 and lk+8..lk+11 of each stage
    constexpr int J = kSK / 8;
    const int lr = t >> 1, lk = (t & 1) * 4;
    const bool a_live = m0 + lr < NC, b_live = n0 + lr < NC;
    const float* a_src = A + static_cast<long long>(m0 + lr) * kSelD + lk;
    const float* b_src = B + static_cast<long long>(n0 + lr) * kSelD + lk;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 ra[J], rb[J];
    auto load = [&](int d0) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            ra[j] = a_live ? *reinterpret_cast<const float4*>(a_src + d0 + 8 * j) : zero;
            rb[j] = b_live ? *reinterpret_cast<const float4*>(b_src + d0 + 8 * j) : zero;
        }
    };
    auto stage = [&](int buf) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            As[buf][lk + 8 * j + 0][lr] = ra[j].x; As[buf][lk + 8 * j + 1][lr] = ra[j].y;
            As[buf][lk + 8 * j + 2][lr] = ra[j].z; As[buf][lk + 8 * j + 3][lr] = ra[j].w;
            Bs[buf][lk + 8 * j + 0][lr] = rb[j].x; Bs[buf][lk + 8 * j + 1][lr] = rb[j].y;
            Bs[buf][lk + 8 * j + 2][lr] = rb[j].z; Bs[buf][lk + 8 * j + 3][lr] = rb[j].w;
        }
    };
    load(0);
    stage(0);
    __syncthreads();
    const int ty = t >> 4, tx = t & 15;
    uint64_t acc[8][4];   // acc[i][p]: row i's scores at columns 2p, 2p+1 of the thread's 8
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[i][p] = 0ull;
    constexpr int NCH = kSelD / kSK;
#pragma unroll 1
    for (int ch = 0; ch < NCH; ++ch) {
        const int buf = ch & 1;
        if (ch + 1 < NCH) load((ch + 1) * kSK);
#pragma unroll
        for (int kk = 0; kk < kSK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const uint64_t bp[4] = {f2_pack(bv[0], bv[1]), f2_pack(bv[2], bv[3]),
                                    f2_pack(bv[4], bv[5]), f2_pack(bv[6], bv[7])};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t a2 = f2_pack(av[i], av[i]);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[i][p] = f2_fma(a2, bp[p], acc[i][p]);
            }
        }
        if (ch + 1 < NCH) stage(buf ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
        if (row >= NC) continue;
        float* dst = S + (bh * NC + row) * LD + n0;
        *reinterpret_cast<ulonglong2*>(dst + 4 * tx) = make_ulonglong2(acc[i][0], acc[i][1]);
        *reinterpret_cast<ulonglong2*>(dst + 64 + 4 * tx) = make_ulonglong2(acc[i][2], acc[i][3]);
    }
}

// ---------------------------------------------------------------- top-k kernels
//
// One warp per query row reads the row's FP32 scores and the cube norms, finds
// the k-th / (k+1)-th values by radix selection, classifies every key against
// the error bound and ranks the undecided ones by exact score.  The FP32 score
// of two 128-dim vectors (FFMA, any order; the means' grid keeps every partial
// sum on 2^-106 Z, so nothing underflows) is within gamma_128 sum|q||k| <=
// 2^-17 (1 + 2^-16) |q| |k| of the exact one; the norms are FP32 too, within
// 2^-17 relative, and e = 2^-15 |q^| max|k^| bounds the error with a factor of
// about 4 to spare.
// The main kernel (kTopkWarps warps per CTA, one row each) leaves rows with more
// than kCap undecided keys to the fallback kernel (kFbWarps warps per CTA,
// grid-stride over rows, room for every key of a row).
constexpr int kCap = 32;
constexpr int kTopkWarps = 8;
constexpr int kFbWarps = 2;
constexpr float kErrScale = 1.0f / 32768.0f;

// NCF: the cube count as a compile-time constant (a row of exactly CH chunks,
// so every per-key bounds test folds away), or 0 to take it from nc_arg.
// Rows of 16 chunks run four CTAs per SM (64 registers, a few spilled): the
// selection is issue-bound and the extra warps measured faster than three CTAs.
template <int CH, int CAP, bool FALLBACK, int NCF = 0>
__global__ void __launch_bounds__(FALLBACK ? kFbWarps * 32 : kTopkWarps * 32, FALLBACK ? 1 : (CH > 16 ? 2 : 4)) vsa_topk_kernel(
    float* __restrict__ S, const float* __restrict__ qm, const float* __restrict__ km,
    const float* __restrict__ qn, const float* __restrict__ kn, int nc_arg, int topk, long long rows,
    int32_t* __restrict__ deferred, int32_t* __restrict__ idx, uint32_t* status, float coarse_l2) {
    const int NC = NCF ? NCF : nc_arg;
    extern __shared__ __align__(16) uint8_t topk_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = FALLBACK ? kFbWarps : kTopkWarps;
    Cands<CAP>* cb = reinterpret_cast<Cands<CAP>*>(topk_smem) + warp;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // scores (and flags) of the kernel before
    if (!FALLBACK) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int LD = score_ld(NC);
    // main form: one row per warp; fallback form: warps stride over groups of 32
    // rows, each lane loading one row's flag, and visit the flagged rows
    const long long first = FALLBACK ? (static_cast<long long>(blockIdx.x) * kWarps + warp) * 32
                                     : static_cast<long long>(blockIdx.x) * kWarps + warp;
    const long long stride = FALLBACK ? static_cast<long long>(gridDim.x) * kWarps * 32 : rows;
    for (long long base = first; base < rows; base += stride) {
        uint32_t todo = 1u;
        if (FALLBACK) {
            const long long r = base + lane;
            todo = __ballot_sync(0xffffffffu, r < rows && deferred[r] != 0);
        }
        for (; todo; todo &= todo - 1) {
        const long long row = FALLBACK ? base + __ffs(todo) - 1 : base;
        const long long bh = row / NC;
        int32_t* out = idx + row * topk;
        float* srow = S + row * LD;
        float s[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) s[c] = c * 32 + lane < NC ? srow[c * 32 + lane] : 0.0f;
        // Coarse branch: the row's softmax over all key cubes replaces its scores
        // once the row is decided (a row left to the fallback keeps its scores
        // for it).  p = 2^((s - max) * scale * log2 e) / sum.
        auto write_probs = [&]() {
            if (coarse_l2 <= 0.0f) return;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < CH; ++c)
                if (c * 32 + lane < NC) mx = fmaxf(mx, s[c]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            float p[CH], l = 0.0f;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                p[c] = c * 32 + lane < NC ? exp2f((s[c] - mx) * coarse_l2) : 0.0f;
                l += p[c];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            const float inv = 1.0f / l;
#pragma unroll
            for (int c = 0; c < CH; ++c)
                if (c * 32 + lane < NC) srow[c * 32 + lane] = p[c] * inv;
        };
        RowClass<CH> rc;
        if (topk >= NC) {   // every key
#pragma unroll
            for (int c = 0; c < CH; ++c) rc.in_m[c] = __ballot_sync(0xffffffffu, c * 32 + lane < NC);
            if (!FALLBACK && lane == 0) deferred[row] = 0;
            write_row<CH, CAP>(rc, cb, false, NC, topk, out, status);
            write_probs();
            continue;
        }
        const float* nkh = kn + bh * NC;
        float nkmax = 0.0f;
#pragma unroll
        for (int c = 0; c < CH; ++c)
            if (c * 32 + lane < NC) nkmax = fmaxf(nkmax, nkh[c * 32 + lane]);
        nkmax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(nkmax)));   // >= 0
        const float e = __fmul_ru(__fmul_ru(qn[row], nkmax), kErrScale);
        classify_row<CH>(s, NC, topk, e, rc, cb->hist, cb->list);
        const int need = topk - rc.n_in;
        if (!FALLBACK && need > 0 && rc.n_unc > CAP) {   // left to the fallback kernel
            if (lane == 0) deferred[row] = 1;
            continue;
        }
        if (need > 0) {
            const float* qrow = qm + row * kSelD;
            resolve_exact<CH, CAP>(rc, need, [&](int d) { return qrow[d]; }, km + bh * NC * kSelD, cb);
        }
        if (!FALLBACK && lane == 0) deferred[row] = 0;
        write_row<CH, CAP>(rc, cb, need > 0, NC, topk, out, status);
        write_probs();
        __syncwarp();
        }
    }
}

template <int CH, int CAP, int WARPS>
constexpr size_t topk_smem_bytes() { return sizeof(Cands<CAP>) * WARPS; }

// ---------------------------------------------------------------- coarse branch
//
// O_c[bh] = P[bh] Vm[bh]: the probabilities of every query cube over all key
// cubes ([NC][NC], row stride score_ld(NC)) times the pooled values ([NC][128]),
// FP32 FFMA.  One 32 (query cubes) x 128 (dims) tile per CTA, 64 threads with
// 8 x 8 register tiles (rows 4ty.., 16+4ty.., dims 4tx.., 64+4tx..); the key
// dimension passes through shared memory eight keys at a time (P stored
// key-major, Vm row-major), the next eight loaded into registers meanwhile.
// (64-row tiles gave 192 CTAs for 24 heads of 512 cubes, 0.4 waves: 76 us.)
constexpr int kPvM = 32;
constexpr int kPvThreads = 64;

__global__ void __launch_bounds__(kPvThreads) vsa_coarse_pv_kernel(const float* __restrict__ P,
                                                                   const float* __restrict__ vm,
                                                                   int NC, float* __restrict__ oc) {
    __shared__ __align__(16) float As[2][kGK][kPvM + 4];
    __shared__ __align__(16) float Bs[2][kGK][kSelD];
    asm volatile("griddepcontrol.wait;" ::: "memory");   // probabilities of the top-k kernels
    const int t = threadIdx.x;
    const long long bh = blockIdx.y;
    const int m0 = blockIdx.x * kPvM;
    const int LD = score_ld(NC);
    const int ar = t >> 1, ak = (t & 1) * 4;          // P: row ar, keys ak..ak+3 of a stage
    const int bk = t >> 3, bd = (t & 7) * 4;          // Vm: key bk, dims bd + 32i (i < 4)
    const bool a_live = m0 + ar < NC;
    const float* a_src = P + (bh * NC + m0 + ar) * LD + ak;
    const float* b_src = vm + bh * NC * kSelD;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 ra, rb[4];
    auto load = [&](int kc) {
        ra = (a_live && kc + ak < NC) ? *reinterpret_cast<const float4*>(a_src + kc) : zero;
        const bool bl = kc + bk < NC;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            rb[i] = bl ? *reinterpret_cast<const float4*>(b_src + static_cast<long long>(kc + bk) * kSelD +
                                                          32 * i + bd)
                       : zero;
    };
    auto stage = [&](int buf) {
        As[buf][ak + 0][ar] = ra.x; As[buf][ak + 1][ar] = ra.y;
        As[buf][ak + 2][ar] = ra.z; As[buf][ak + 3][ar] = ra.w;
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<float4*>(&Bs[buf][bk][32 * i + bd]) = rb[i];
    };
    load(0);
    stage(0);
    __syncthreads();
    const int ty = t >> 4, tx = t & 15;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    const int nch = (NC + kGK - 1) / kGK;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        const int buf = ch & 1;
        if (ch + 1 < nch) load((ch + 1) * kGK);
#pragma unroll
        for (int kk = 0; kk < kGK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][16 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (ch + 1 < nch) stage(buf ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + (i < 4 ? 4 * ty + i : 16 + 4 * ty + i - 4);
        if (row >= NC) continue;
        float* dst = oc + (bh * NC + row) * kSelD;
        *reinterpret_cast<float4*>(dst + 4 * tx) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        *reinterpret_cast<float4*>(dst + 64 + 4 * tx) =
            make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

namespace {
// Workspace of the selection, each part 256-byte aligned: FP32 cube means of Q
// and K [rows][D], their norms [rows], one int32 "left to the fallback" flag per
// row, and the FP32 scores [rows][score_ld(NC)] (rows = B*H*NC query cubes).
struct SelectLayout {
    size_t qm, km, qn, kn, flags, scores, total;
    size_t vm, total_coarse;   // the coarse branch adds the pooled values
};
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
SelectLayout select_layout(size_t rows, int NC, int D) {
    SelectLayout L;
    L.qm = 0;
    L.km = L.qm + align256(rows * D * sizeof(float));
    L.qn = L.km + align256(rows * D * sizeof(float));
    L.kn = L.qn + align256(rows * sizeof(float));
    L.flags = L.kn + align256(rows * sizeof(float));
    L.scores = L.flags + align256(rows * sizeof(int32_t));
    L.total = L.scores + rows * static_cast<size_t>(score_ld(NC)) * sizeof(float);
    L.vm = align256(L.total);
    L.total_coarse = L.vm + rows * D * sizeof(float);
    return L;
}
}  // namespace

extern "C" size_t vsa_select_workspace_size(int B, int H, int S, int D, int block) {
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return 0;
    const int nc = S / block;
    return select_layout(static_cast<size_t>(B) * H * nc, nc, D).total;
}

extern "C" size_t vsa_select_coarse_workspace_size(int B, int H, int S, int D, int block) {
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return 0;
    const int nc = S / block;
    return select_layout(static_cast<size_t>(B) * H * nc, nc, D).total_coarse;
}

namespace {
// The selection (v == nullptr) or the selection plus the coarse branch.
int select_impl(const void* q, const void* k, const void* v, int B, int H, int S, int D,
                int block, int topk, int prefix, const int32_t* cube_valid, float scale,
                int32_t* idx, float* o_coarse, void* workspace, size_t workspace_bytes,
                void* stream) {
    const bool coarse = v != nullptr;
    if (!q || !k || !idx || (coarse && !o_coarse)) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || S <= 0 || topk <= 0 || prefix < 0 || prefix >= S)
        return GBATTN_ERR_SHAPE;
    if (D != 128 || block != 64) return GBATTN_ERR_UNSUPPORTED;
    if ((S - prefix) % block != 0) return GBATTN_ERR_SHAPE;
    const int NC = (S - prefix) / block;
    if (NC > kMaxChunks * 32 || topk > NC) return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    if (coarse && !finite_positive(scale)) return GBATTN_ERR_SCALE;
    const size_t need = coarse ? vsa_select_coarse_workspace_size(B, H, S, D, block)
                               : vsa_select_workspace_size(B, H, S, D, block);
    if (!workspace || workspace_bytes < need) return GBATTN_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(workspace) || !aligned16(v) ||
        !aligned16(o_coarse) || (reinterpret_cast<uintptr_t>(idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(cube_valid) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t in_bytes = static_cast<size_t>(B) * H * S * D * 2;
    const size_t idx_bytes = static_cast<size_t>(B) * H * NC * topk * 4;
    const size_t oc_bytes = static_cast<size_t>(B) * H * NC * D * 4;
    if (overlaps(idx, idx_bytes, q, in_bytes) || overlaps(idx, idx_bytes, k, in_bytes) ||
        overlaps(workspace, need, q, in_bytes) || overlaps(workspace, need, k, in_bytes) ||
        overlaps(workspace, need, idx, idx_bytes) || overlaps(idx, idx_bytes, v, in_bytes) ||
        overlaps(workspace, need, v, in_bytes) || overlaps(o_coarse, oc_bytes, q, in_bytes) ||
        overlaps(o_coarse, oc_bytes, k, in_bytes) || overlaps(o_coarse, oc_bytes, v, in_bytes) ||
        overlaps(o_coarse, oc_bytes, idx, idx_bytes) || overlaps(o_coarse, oc_bytes, workspace, need))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    if (dev.device < 0 || dev.device >= 64) return GBATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long n_bh = static_cast<long long>(B) * H;
    const long long rows = n_bh * NC;
    const SelectLayout L = select_layout(static_cast<size_t>(rows), NC, D);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* qm = reinterpret_cast<float*>(ws + L.qm);
    float* km = reinterpret_cast<float*>(ws + L.km);
    float* qn = reinterpret_cast<float*>(ws + L.qn);
    float* kn = reinterpret_cast<float*>(ws + L.kn);
    int32_t* deferred = reinterpret_cast<int32_t*>(ws + L.flags);
    float* scores = reinterpret_cast<float*>(ws + L.scores);
    float* vm = coarse ? reinterpret_cast<float*>(ws + L.vm) : nullptr;
    const float coarse_l2 = coarse ? scale * 1.4426950408889634f : 0.0f;

    static std::once_flag attr_once[64];
    static int attr_rc[64];
    std::call_once(attr_once[dev.device], [&] {
        bool ok = cudaFuncSetAttribute(vsa_topk_kernel<32, 1024, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(topk_smem_bytes<32, 1024, kFbWarps>())) ==
                  cudaSuccess;
        ok &= cudaFuncSetAttribute(vsa_topk_kernel<16, 512, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(topk_smem_bytes<16, 512, kFbWarps>())) ==
              cudaSuccess;
        attr_rc[dev.device] = ok ? GBATTN_OK : GBATTN_ERR_CUDA;
    });
    if (attr_rc[dev.device] != GBATTN_OK) {
        cudaGetLastError();
        return GBATTN_ERR_CUDA;
    }

    const long long pool_threads = rows * (D / 8);
    dim3 pgrid(static_cast<unsigned>((pool_threads + kPoolThreads - 1) / kPoolThreads), coarse ? 3 : 2);
    vsa_pool_kernel<<<pgrid, kPoolThreads, 0, s>>>(static_cast<const __half*>(q),
                                                   static_cast<const __half*>(k), n_bh, NC, S,
                                                   prefix, D, block, cube_valid, dev.status, qm,
                                                   km, qn, kn, static_cast<const __half*>(v), vm);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return GBATTN_ERR_CUDA;

    // The other three kernels are programmatic dependent launches: their CTAs
    // are placed as the previous grid retires and wait (griddepcontrol.wait)
    // for all of its results.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float *cqm = qm, *ckm = km, *cqn = qn, *ckn = kn, *cs = scores;
    auto launched = [&](cudaError_t e) {
        count_launches(1);
        if (e == cudaSuccess) return true;
        cudaGetLastError();
        return false;
    };
    const unsigned tiles = static_cast<unsigned>((NC + kGT - 1) / kGT);
    cfg.gridDim = dim3(tiles, tiles, static_cast<unsigned>(n_bh));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = 0;
    if (!launched(cudaLaunchKernelEx(&cfg, vsa_score_kernel, cqm, ckm, NC, scores)))
        return GBATTN_ERR_CUDA;
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kTopkWarps - 1) / kTopkWarps));
    cfg.blockDim = dim3(kTopkWarps * 32);
    cudaError_t e;
    if (NC <= 512) {
        cfg.dynamicSmemBytes = topk_smem_bytes<16, kCap, kTopkWarps>();
        e = NC == 512 ? cudaLaunchKernelEx(&cfg, vsa_topk_kernel<16, kCap, false, 512>, scores, cqm,
                                           ckm, cqn, ckn, NC, topk, rows, deferred, idx, dev.status,
                                           coarse_l2)
                      : cudaLaunchKernelEx(&cfg, vsa_topk_kernel<16, kCap, false>, scores, cqm, ckm,
                                           cqn, ckn, NC, topk, rows, deferred, idx, dev.status,
                                           coarse_l2);
    } else {
        cfg.dynamicSmemBytes = topk_smem_bytes<32, kCap, kTopkWarps>();
        e = NC == 1024 ? cudaLaunchKernelEx(&cfg, vsa_topk_kernel<32, kCap, false, 1024>, scores, cqm,
                                            ckm, cqn, ckn, NC, topk, rows, deferred, idx, dev.status,
                                            coarse_l2)
                       : cudaLaunchKernelEx(&cfg, vsa_topk_kernel<32, kCap, false>, scores, cqm, ckm,
                                            cqn, ckn, NC, topk, rows, deferred, idx, dev.status,
                                            coarse_l2);
    }
    if (!launched(e)) return GBATTN_ERR_CUDA;
    const long long fb_ctas = std::min<long long>((rows + 32 * kFbWarps - 1) / (32 * kFbWarps),
                                                  2LL * dev.num_sms);
    cfg.gridDim = dim3(static_cast<unsigned>(fb_ctas));
    cfg.blockDim = dim3(kFbWarps * 32);
    if (NC <= 512) {
        cfg.dynamicSmemBytes = topk_smem_bytes<16, 512, kFbWarps>();
        e = cudaLaunchKernelEx(&cfg, vsa_topk_kernel<16, 512, true>, scores, cqm, ckm, cqn, ckn, NC,
                               topk, rows, deferred, idx, dev.status, coarse_l2);
    } else {
        cfg.dynamicSmemBytes = topk_smem_bytes<32, 1024, kFbWarps>();
        e = cudaLaunchKernelEx(&cfg, vsa_topk_kernel<32, 1024, true>, scores, cqm, ckm, cqn, ckn, NC,
                               topk, rows, deferred, idx, dev.status, coarse_l2);
    }
    if (!launched(e)) return GBATTN_ERR_CUDA;
    if (coarse) {
        cfg.gridDim = dim3(static_cast<unsigned>((NC + kPvM - 1) / kPvM), static_cast<unsigned>(n_bh));
        cfg.blockDim = dim3(kPvThreads);
        cfg.dynamicSmemBytes = 0;
        const float* cvm = vm;
        if (!launched(cudaLaunchKernelEx(&cfg, vsa_coarse_pv_kernel, cs, cvm, NC, o_coarse)))
            return GBATTN_ERR_CUDA;
    }
    return launch_status();
}
}  // namespace

extern "C" int vsa_select_blocks(const void* q, const void* k, int B, int H, int S, int D,
                                 int block, int topk, int prefix, const int32_t* cube_valid,
                                 int32_t* idx, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    CallRange nvtx_range("vsa_select_blocks");
    return select_impl(q, k, nullptr, B, H, S, D, block, topk, prefix, cube_valid, 0.0f, idx,
                       nullptr, workspace, workspace_bytes, stream);
}

extern "C" int vsa_select_blocks_coarse(const void* q, const void* k, const void* v, int B, int H,
                                        int S, int D, int block, int topk, int prefix,
                                        const int32_t* cube_valid, float scale, int32_t* idx,
                                        float* o_coarse, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    CallRange nvtx_range("vsa_select_blocks_coarse");
    if (!v) return GBATTN_ERR_NULL;
    return select_impl(q, k, v, B, H, S, D, block, topk, prefix, cube_valid, scale, idx, o_coarse,
                       workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ query-cube pairing
//
// The sparse attention kernel processes two query cubes per item over the union
// of their selected key cubes; every key cube only one of the two selected is
// wasted work for the other.  The pairing is the greedy one: the pair of
// largest selection overlap first (ties: the lower cube indices), then the
// largest among the cubes left, and so on.  Three kernels compute it:
//   vsa_pair_bits_kernel (a warp per cube): every cube's selection as a bitset
//     over key cubes, into the workspace;
//   vsa_pair_cand_kernel (a warp per four cubes): every cube's kPairCand (32)
//     best partners over all cubes of the head, by overlap then index, into the
//     workspace;
//   vsa_pair_kernel (a CTA per head): rounds of "mutual best": each unpaired
//     cube takes the first unpaired cube of its list, and two cubes that take
//     each other pair up.  Such a pair is the heaviest one left at both its
//     cubes, so the greedy order pairs it too.  A cube whose list has run out
//     waits for the second phase: rounds of mutual best over all cubes still
//     unpaired (full overlap scans), which complete the greedy pairing.  A
//     lone cube of an odd count stays alone.
// The pairs are written longest union first (ties: lower first cube): the
// persistent sparse kernel hands its items out in this order, so the long
// ones do not end the launch.  Any pairing gives the same attention result
// (up to summation order); this one only saves work.
namespace gbattn {
namespace {
constexpr int kPairThreads = 1024;   // vsa_pair_kernel: one thread per cube
constexpr int kPairMaxCubes = 1024;
constexpr int kPairCand = 32;        // candidates kept per cube (one per lane)
constexpr int kCandThreads = 128;    // vsa_pair_cand_kernel: four warps

__host__ __device__ inline int pair_words(int nc) { return (nc + 31) / 32; }
// selection bitsets padded to whole 16-byte rows (vector loads)
__host__ __device__ inline int pair_row_words(int nc) { return (pair_words(nc) + 3) & ~3; }
__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Cubes per warp of vsa_pair_cand_kernel: four when a lane's share of the
// partners (one in 32) fits 16 registers per cube, else two.
inline int cand_cubes_per_warp(int nc) { return nc <= 512 ? 4 : 2; }

size_t cand_smem_bytes(int nc) {
    return static_cast<size_t>(nc) * pair_row_words(nc) * 4 + kCandThreads * 4;
}

// vsa_pair_kernel's shared memory: bitset rows, candidate lists, then int16
// arrays (partner, best, list, first cube of each pair) and the pairs' tiles.
__host__ __device__ inline size_t pair_lists_offset(int nc) {
    return static_cast<size_t>(nc) * pair_row_words(nc) * 4;
}
__host__ __device__ inline size_t pair_arrays_offset(int nc) {
    return pair_lists_offset(nc) + static_cast<size_t>(nc) * kPairCand * 2;
}
__host__ __device__ inline size_t pair_tiles_offset(int nc) {
    return pair_arrays_offset(nc) + align16(static_cast<size_t>(nc) * 2 * 4);
}
size_t pair_smem_bytes(int nc) { return pair_tiles_offset(nc) + align16(static_cast<size_t>(nc + 8) * 2); }

// Workspace: the bitset rows, then the candidate lists.
size_t pair_bits_bytes(int B, int H, int nc) {
    return static_cast<size_t>(B) * H * nc * pair_row_words(nc) * 4;
}

// Candidate key: overlap in the high half, then the lower index first.
__device__ __forceinline__ uint32_t cand_key(int overlap, int b) {
    return (static_cast<uint32_t>(overlap) << 16) | static_cast<uint32_t>(0xFFFF - b);
}

// Exclusive prefix sum of v over the block (one value per thread); returns the
// total through *total.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_warps = static_cast<int>(blockDim.x) >> 5;
    int x = v;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, sh);
        if (lane >= sh) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < n_warps ? warp_tot[lane] : 0;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, sh);
            if (lane >= sh) t += y;
        }
        warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    *total = warp_tot[n_warps - 1];
    __syncthreads();
    return before;
}

// Every cube's selection as a bitset over key cubes (one warp per cube): lane i
// takes entries i, i + 32, ...; each word of the row is the OR over the lanes of
// the bits that fall in it, and lane w stores word w.  Entries out of range are
// skipped.  Rows are row_words long (whole 16-byte units).
__global__ void __launch_bounds__(256) vsa_pair_bits_kernel(const int32_t* __restrict__ idx,
                                                            long long rows, int nc, int topk,
                                                            uint32_t* __restrict__ bits) {
    const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;   // warp-uniform
    const int rw = pair_row_words(nc);
    const int32_t* sel = idx + r * topk;
    uint32_t mine = 0u;   // word `lane` of the row
    for (int base = 0; base < topk; base += 32) {
        const int kc = base + lane < topk ? sel[base + lane] : -1;
        const bool ok = kc >= 0 && kc < nc;
        const int w = ok ? (kc >> 5) : -1;
        const uint32_t bit = ok ? 1u << (kc & 31) : 0u;
        for (int ww = 0; ww < rw; ++ww) {
            const uint32_t v = __reduce_or_sync(0xffffffffu, w == ww ? bit : 0u);
            if (lane == ww) mine |= v;
        }
    }
    if (lane < rw) bits[r * rw + lane] = mine;
}

// 16-byte chunk q and word w of bitset row b (rows of rw words).
__device__ __forceinline__ uint4 row_chunk(const uint32_t* bits, int rw, int b, int q) {
    return reinterpret_cast<const uint4*>(bits + b * rw)[q];
}
__device__ __forceinline__ uint32_t row_word(const uint32_t* bits, int rw, int b, int w) {
    return bits[b * rw + w];
}

// Copy a head's bitset rows (nc rows of row_words words) into shared memory.
__device__ void load_rows(const uint32_t* __restrict__ src, int nc, int rw, uint32_t* dst) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < nc * (rw >> 2); i += blockDim.x) d4[i] = s4[i];
    __syncthreads();
}

__device__ __forceinline__ int popc_and4(uint4 x, uint4 y) {
    return __popc(x.x & y.x) + __popc(x.y & y.y) + __popc(x.z & y.z) + __popc(x.w & y.w);
}

// Each warp takes CPW cubes a; lane l holds the overlaps of those cubes with the
// partners b = l + 32 i (i < CPL), each partner row read once for all CPW cubes.
// A cube's kPairCand best partners (overlap, then the lower index) come from a
// bitwise search for the overlap threshold tau (the largest value that at least
// kPairCand partners reach), every partner above tau, the lowest-index partners
// at tau, and a 32-lane bitonic sort of their keys.
// NCF: the cube count as a compile-time constant (every bounds test and the
// row length fold away), or 0 to take it from nc_arg.
template <int CPL, int CPW, int NCF = 0>
__global__ void __launch_bounds__(kCandThreads) vsa_pair_cand_kernel(const uint32_t* __restrict__ gbits,
                                                                     int nc_arg, int top_bit,
                                                                     int16_t* __restrict__ cand) {
    const int nc = NCF ? NCF : nc_arg;
    extern __shared__ uint32_t csm[];
    const int rw = pair_row_words(nc);
    uint32_t* bits = csm;                                   // [nc][rw]
    uint32_t* stage = csm + static_cast<size_t>(nc) * rw;   // [warps][32] keys
    const long long bh = blockIdx.y;
    load_rows(gbits + bh * nc * static_cast<long long>(rw), nc, rw, bits);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a0 = (static_cast<int>(blockIdx.x) * (kCandThreads / 32) + warp) * CPW;
    if (a0 >= nc) return;   // warp-uniform; no block barrier follows
    int acc[CPW][CPL];
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int i = 0; i < CPL; ++i) acc[c][i] = 0;
    for (int q = 0; q < (rw >> 2); ++q) {
        uint4 A[CPW];
#pragma unroll
        for (int c = 0; c < CPW; ++c)
            A[c] = a0 + c < nc ? row_chunk(bits, rw, a0 + c, q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int b = lane + 32 * i;
            if (b < nc) {
                const uint4 Bv = row_chunk(bits, rw, b, q);
#pragma unroll
                for (int c = 0; c < CPW; ++c) acc[c][i] += popc_and4(A[c], Bv);
            }
        }
    }
    const unsigned lt = (1u << lane) - 1u;
    uint32_t* st = stage + warp * 32;
    const int want = min(kPairCand, nc - 1);
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
        const int a = a0 + c;
        if (a >= nc) break;   // warp-uniform
        // -1 marks no partner (past the end, or the cube itself)
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int b = lane + 32 * i;
            if (b >= nc || b == a) acc[c][i] = -1;
        }
        int tau = 0;
        for (int bit = top_bit; bit >= 0; --bit) {   // overlaps are at most topk < 2^(top_bit+1)
            const int trial = tau | (1 << bit);
            int n = 0;
#pragma unroll
            for (int i = 0; i < CPL; ++i) n += acc[c][i] >= trial;
            if (static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n))) >= want) tau = trial;
        }
        int need = want;   // partners at tau still to take
        {
            int above = 0;
#pragma unroll
            for (int i = 0; i < CPL; ++i) above += acc[c][i] > tau;
            need -= static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(above)));
        }
        int slot = 0;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {   // index order: i, then lane
            const int v = acc[c][i];
            const unsigned meq = __ballot_sync(0xffffffffu, v == tau);
            const bool take = v > tau || (v == tau && __popc(meq & lt) < need);
            need -= min(need, __popc(meq));
            const unsigned mt = __ballot_sync(0xffffffffu, take);
            const int at = slot + __popc(mt & lt);   // below want by the choice of tau
            if (take && at < 32) st[at] = cand_key(v, lane + 32 * i);
            slot += __popc(mt);
        }
        __syncwarp();
        uint32_t k = lane < want ? st[lane] : 0u;
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const uint32_t o = __shfl_xor_sync(0xffffffffu, k, stride);
                k = (((lane & stride) == 0) == ((lane & size) == 0)) ? max(k, o) : min(k, o);
            }
        cand[(bh * nc + a) * kPairCand + lane] =
            static_cast<int16_t>(k == 0u ? -1 : 0xFFFF - static_cast<int>(k & 0xFFFFu));
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kPairThreads) vsa_pair_kernel(const uint32_t* __restrict__ gbits,
                                                                const int16_t* __restrict__ cand,
                                                                int nc,
                                                                int32_t* __restrict__ pairs) {
    extern __shared__ uint32_t psm[];
    __shared__ int warp_tot[32];
    const int words = pair_row_words(nc);
    uint8_t* base = reinterpret_cast<uint8_t*>(psm);
    uint32_t* bits = psm;                                                         // [nc][words]
    int16_t* cl = reinterpret_cast<int16_t*>(base + pair_lists_offset(nc));       // [nc][kPairCand]
    int16_t* partner = reinterpret_cast<int16_t*>(base + pair_arrays_offset(nc));
    int16_t* best = partner + nc;
    int16_t* list = best + nc;
    int16_t* p_first = list + nc;
    int16_t* p_tiles = reinterpret_cast<int16_t*>(base + pair_tiles_offset(nc));  // 16-byte aligned
    const long long bh = blockIdx.x;
    const int a = threadIdx.x;
    const int lane = a & 31, warp = a >> 5;
    const bool live = a < nc;
    load_rows(gbits + bh * nc * static_cast<long long>(words), nc, words, bits);
    {
        const uint4* src = reinterpret_cast<const uint4*>(cand + bh * nc * kPairCand);
        uint4* dst = reinterpret_cast<uint4*>(cl);
        for (int i = a; i < nc * kPairCand / 8; i += kPairThreads) dst[i] = src[i];
    }
    if (live) partner[a] = -1;
    for (int i = a; i < nc + 8; i += kPairThreads) p_tiles[i] = -1;
    __syncthreads();
    // phase 1: mutual best over the candidate lists (each round pairs at least one
    // pair or ends the phase); a list is read eight entries at a time, the eight
    // partner lookups together
    for (int r = 0; r < nc; ++r) {
        int bb = -1;
        if (live && partner[a] < 0) {
            const uint4* L = reinterpret_cast<const uint4*>(cl + a * kPairCand);
            for (int q = 0; q < kPairCand / 8 && bb < 0; ++q) {
                const uint4 v = L[q];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                int c8[8], p8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) c8[e] = static_cast<int16_t>((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
#pragma unroll
                for (int e = 0; e < 8; ++e) p8[e] = (c8[e] >= 0 && c8[e] < nc) ? partner[c8[e]] : 0;
                bool end = false;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (bb >= 0 || end) continue;
                    if (c8[e] < 0 || c8[e] >= nc) end = true;
                    else if (p8[e] < 0) bb = c8[e];
                }
                if (end) break;
            }
        }
        if (live) best[a] = static_cast<int16_t>(bb);
        __syncthreads();
        const bool pair_now = live && partner[a] < 0 && bb >= 0 && best[bb] == a;
        if (pair_now) partner[a] = static_cast<int16_t>(bb);
        if (!__syncthreads_or(pair_now)) break;
    }
    // phase 2: mutual best over all cubes still unpaired (the heaviest pair left
    // is always mutual, so each round pairs at least one pair); a warp scans the
    // partners of one unpaired cube at a time, a lane every 32nd of them
    for (int r = 0; r < nc; ++r) {
        int n_left = 0;
        const bool left = live && partner[a] < 0;
        const int lr = block_exclusive_scan(left ? 1 : 0, warp_tot, &n_left);
        if (left) list[lr] = static_cast<int16_t>(a);
        __syncthreads();
        if (n_left < 2) break;
        for (int li = warp; li < n_left; li += kPairThreads / 32) {
            const int me = list[li];
            uint32_t bk = 0u;
            int bb = -1;
            for (int j = lane; j < n_left; j += 32) {
                const int b = list[j];
                if (b == me) continue;
                int n = 0;
                for (int q = 0; q < (words >> 2); ++q)
                    n += popc_and4(row_chunk(bits, words, me, q), row_chunk(bits, words, b, q));
                const uint32_t k = cand_key(n, b);
                if (k > bk) {
                    bk = k;
                    bb = b;
                }
            }
            const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
            const unsigned who = __ballot_sync(0xffffffffu, mk != 0u && bk == mk);
            const int win = who ? __shfl_sync(0xffffffffu, bb, __ffs(who) - 1) : -1;
            if (lane == 0) best[me] = static_cast<int16_t>(win);
        }
        __syncthreads();
        const int me = a < n_left ? list[a] : -1;
        const int bb = me >= 0 ? best[me] : -1;
        const bool pair_now = me >= 0 && bb >= 0 && best[bb] == me;
        if (pair_now) partner[me] = static_cast<int16_t>(bb);
        if (!__syncthreads_or(pair_now)) break;
    }
    // (phase 2 leaves at most one cube; should any more be left, they pair up in
    // index order, so that the output is always a pairing)
    {
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
    }
    // every pair once (by its lower cube; a lone cube by itself) with its union's tiles
    const int pb = live ? partner[a] : 0;
    const bool first = live && (pb > a || pb < 0);
    int n_pairs = 0;
    const int slot = block_exclusive_scan(first ? 1 : 0, warp_tot, &n_pairs);
    int tiles = 0;
    if (first) {
        int u = 0;
        for (int w = 0; w < words; ++w)
            u += __popc(row_word(bits, words, a, w) | (pb >= 0 ? row_word(bits, words, pb, w) : 0u));
        tiles = (u + 1) / 2;
        p_first[slot] = static_cast<int16_t>(a);
        p_tiles[slot] = static_cast<int16_t>(tiles);
    }
    __syncthreads();
    // rank: more tiles first, then the lower first cube (slots are in cube order);
    // the padding past the last pair holds -1
    if (first) {
        int rank = 0;
        const uint4* t8 = reinterpret_cast<const uint4*>(p_tiles);
        for (int j8 = 0; j8 < (n_pairs + 7) / 8; ++j8) {
            const uint4 v = t8[j8];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int tj = static_cast<int16_t>((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                const int j = j8 * 8 + e;
                rank += (tj > tiles) || (tj == tiles && j < slot);
            }
        }
        if (rank < (nc + 1) / 2) {   // always true for a pairing
            int32_t* out = pairs + (bh * static_cast<long long>((nc + 1) / 2) + rank) * 2;
            out[0] = a;
            out[1] = pb > a ? pb : -1;
        }
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" size_t vsa_pair_workspace_size(int B, int H, int n_cubes) {
    if (B <= 0 || H <= 0 || n_cubes <= 0) return 0;
    return pair_bits_bytes(B, H, n_cubes) +
           ((static_cast<size_t>(B) * H * n_cubes * kPairCand * 2 + 15) & ~static_cast<size_t>(15));
}

extern "C" int vsa_pair_query_cubes(const int32_t* idx, int B, int H, int n_cubes, int topk,
                                    int32_t* pairs, void* workspace, size_t workspace_bytes,
                                    void* stream) {
    CallRange nvtx_range("vsa_pair_query_cubes");
    if (!idx || !pairs) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || n_cubes <= 0 || topk <= 0 || topk > n_cubes) return GBATTN_ERR_SHAPE;
    if (n_cubes > kPairMaxCubes || static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(pairs) & 3u) ||
        !aligned16(workspace))
        return GBATTN_ERR_ALIGN;
    const size_t wb = vsa_pair_workspace_size(B, H, n_cubes);
    if (!workspace || workspace_bytes < wb) return GBATTN_ERR_WORKSPACE;
    const size_t ib = static_cast<size_t>(B) * H * n_cubes * topk * 4;
    const size_t pb = static_cast<size_t>(B) * H * ((n_cubes + 1) / 2) * 2 * 4;
    if (overlaps(pairs, pb, idx, ib) || overlaps(workspace, wb, idx, ib) ||
        overlaps(workspace, wb, pairs, pb))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    static std::once_flag once[64];
    if (dev.device >= 0 && dev.device < 64)
        std::call_once(once[dev.device], [] {
            cudaFuncSetAttribute(vsa_pair_cand_kernel<16, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cand_smem_bytes(kPairMaxCubes)));
            cudaFuncSetAttribute(vsa_pair_cand_kernel<16, 4, 512>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cand_smem_bytes(kPairMaxCubes)));
            cudaFuncSetAttribute(vsa_pair_cand_kernel<32, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cand_smem_bytes(kPairMaxCubes)));
            cudaFuncSetAttribute(vsa_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(pair_smem_bytes(kPairMaxCubes)));
        });
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* gbits = static_cast<uint32_t*>(workspace);
    int16_t* cand = reinterpret_cast<int16_t*>(static_cast<uint8_t*>(workspace) +
                                               pair_bits_bytes(B, H, n_cubes));
    const long long rows = static_cast<long long>(B) * H * n_cubes;
    vsa_pair_bits_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, s>>>(
        idx, rows, n_cubes, topk, gbits);
    const int cpw = cand_cubes_per_warp(n_cubes);
    const int per_cta = (kCandThreads / 32) * cpw;
    const dim3 cgrid((n_cubes + per_cta - 1) / per_cta, static_cast<unsigned>(B * H));
    int top_bit = 0;   // the highest bit an overlap (at most topk) can have
    while ((2 << top_bit) <= topk) ++top_bit;
    if (n_cubes == 512)
        vsa_pair_cand_kernel<16, 4, 512><<<cgrid, kCandThreads, cand_smem_bytes(n_cubes), s>>>(
            gbits, n_cubes, top_bit, cand);
    else if (cpw == 4)
        vsa_pair_cand_kernel<16, 4><<<cgrid, kCandThreads, cand_smem_bytes(n_cubes), s>>>(gbits, n_cubes, top_bit, cand);
    else
        vsa_pair_cand_kernel<32, 2><<<cgrid, kCandThreads, cand_smem_bytes(n_cubes), s>>>(gbits, n_cubes, top_bit, cand);
    vsa_pair_kernel<<<static_cast<unsigned>(B * H), kPairThreads, pair_smem_bytes(n_cubes), s>>>(
        gbits, cand, n_cubes, pairs);
    count_launches(3);
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
// pooled cube means, their norms, one flag per query cube and the FP32 scores)
// in a fixed array of
// kNoAllocScratchBytes that lives in this library's device image.  Every GPU
// that loads the library holds the array until the process exits.
namespace {
// 48 MiB + 192 KiB: the whole workspace of 16384 query cubes at 512 cubes per
// head and D = 128 (B*H*S <= 1,048,576 tokens x heads at S = 32768, e.g. B=1,
// H=32): means 16 MiB, norms and flags 192 KiB, scores 32 MiB.
constexpr size_t kNoAllocScratchBytes = (48u << 20) + (192u << 10);

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
    CallRange nvtx_range("vsa_select_blocks_noalloc");
    if (!q || !k || !idx) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return GBATTN_ERR_SHAPE;
    const size_t need = vsa_select_workspace_size(B, H, S, D, block);
    if (need > kNoAllocScratchBytes) return GBATTN_ERR_WORKSPACE;   // sizes beyond the fixed scratch
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != GBATTN_OK) return rc;
    // Every scratch byte a call reads was written earlier in the same call (the
    // pool kernel writes the means and norms, the score kernel every score read,
    // the top-k kernel every row's flag), so the previous call's contents need
    // no clearing.
    return vsa_select_blocks(q, k, B, H, S, D, block, topk, prefix, cube_valid, idx, scratch,
                             kNoAllocScratchBytes, stream);
}
