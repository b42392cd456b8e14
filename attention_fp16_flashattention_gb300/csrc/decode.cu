// Decode attention over a paged FP8 E4M3 KV cache ("Integrate FP32 v37
// prefill and exact E4M3 bridge": Implementation, the exact E4M3 paged -> FP16
// bridge; Validation, the E4M3 decode wave kernels and the 256000-input
// decode).  The newest nq tokens of each sequence attend, causally among
// themselves, to its whole cache; the K and V values are exactly the bridge's
// FP16 values RNE_fp16(decode(byte) * scale), formed in registers from the
// cached bytes and never written back to memory.
//
// Work split (balanced whatever the lengths): a stream is one (sequence, KV
// head, group of <= 8 query rows); its work is ceil(kv_len / 16) tiles of 16
// cached tokens.  The streams' tiles are laid end to end and every warp of a
// persistent grid (8 warps per SM) takes an equal contiguous range of them.
//   * Each warp runs its own pipeline: a ring of 16-token stages filled by TMA
//     (128-byte swizzle, one box per 128-byte half of the head width for K and
//     V) issued by one elected lane, with the page-table entries of the next 32
//     tiles prefetched one per lane.
//   * Per tile the warp computes S^T = K Q^T and O^T += V^T P^T on mma.sync
//     (m16n8k16, FP16 in, FP32 accumulate): tokens (QK) and head-width rows
//     (PV) fill the M dimension, the <= 8 query rows fill N.  The E4M3 bytes
//     become MMA fragments directly: for QK each byte pair of a token row is
//     one FP16x2 register (the reduction index is permuted identically in Q);
//     for PV a byte permute pairs the same column of two token rows.
//   * Probabilities leave the QK accumulators as FP16 hi + lo halves (p = hi +
//     lo to about 22 bits), transposed into PV operands by movmatrix, so P
//     keeps FP32-level precision; softmax state is FP32 in log2 units with a
//     lazy rescale (the reference max moves only when a score passes it by
//     more than 2^8).
//   * When its range leaves a stream, the warp writes that stream segment's
//     unnormalised O, max and sum (a partial record); a merge kernel combines
//     the records of every query row and writes O (FP16) and lse.
#include <cuda_fp16.h>
#include <mutex>

#include "e4m3.cuh"
#include "host.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kTile = 16;        // tokens per tile (one MMA M block)
// Warps per CTA, each with its own pipeline.  Two warps per scheduler hide each
// other's conversion and MMA latency chains; eight warps with two stages hold
// the same bytes in flight (128 KB per SM) as four with four.
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 8;         // query rows per stream (MMA N)
constexpr int kMaxSeqs = 4096;   // sequences per launch (prefix table in shared memory)
constexpr float kRescale = 8.0f;

// Scale handling: RNE_fp16(decode(b) * s) equals decode(b) * s exactly when
// s = 2^a with -15 <= a <= 7 (a 4-bit significand stays inside the FP16 range
// and subnormal grid), and then the scale is applied to the FP32 scores and
// outputs instead (a power-of-two factor commutes with every FP32 rounding);
// an FP16-valued scale uses one FP16 multiply; any other scale the
// round-to-odd product.
enum ScaleMode { kScaleFolded = 0, kScaleHalf = 1, kScaleGeneral = 2 };

template <int D>
struct Cfg {
    static constexpr int kHalves = D / 128;
    static constexpr int kStages = D == 256 ? 2 : 4;          // 16 KB per warp
    static constexpr int kBox = kTile * 128;                     // one TMA box
    static constexpr int kStageBytes = 2 * kHalves * kBox;       // K halves, then V halves
    static constexpr int kSteps = D / 16;                        // QK k-steps, PV d-blocks
    static constexpr int kRing = kWarps * kStages * kStageBytes;
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static constexpr int kSmem = kRing + kBarBytes + 4 * (kMaxSeqs + 1) + 16 + 1024;
};

struct DecodeArgs {
    const __half* q;
    const int32_t* table;
    const int32_t* kv_lens;
    float* part_o;        // [record][kRows][D], unnormalised
    float2* part_ml;      // [record][kRows]: (max in log2 units, sum)
    uint32_t* prefix_out; // [B + 1]: tiles of all streams of the sequences before b
    uint32_t* status;
    uint64_t wait_limit;
    int fault;   // test hook: 1 = no stage is loaded, 2 = loads stop after two ring rounds
    int B, Hq, Hkv, nq, G, row_groups, num_phys, ps, max_pages, max_kv;
    float sl2;            // softmax scale * log2(e) (* k_scale when folded)
    float ks, vs;
    __half2 ks2, vs2;
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <int kMode>
__device__ __forceinline__ uint32_t cvt_scaled(uint32_t two_bytes, __half2 s2, float s) {
    const uint32_t h = e4m3x2_to_f16x2(two_bytes);
    if (kMode == kScaleHalf) return scale_f16x2(h, s2);
    if (kMode == kScaleGeneral) return scale_f16x2_general(h, s);
    return h;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Head-width position of PV output row m of d-block j held by lane group g:
// rows g and g + 8 are the adjacent bytes 2*(j%8) and 2*(j%8) + 1 of 16-byte
// column g in half j/8.
__device__ __forceinline__ int pv_col(int j, int g) { return 128 * (j >> 3) + 16 * g + 2 * (j & 7); }

// Tiles of one stream of a sequence (0 for a rejected length).
__device__ __forceinline__ uint32_t seq_tiles(int len, int nq, int max_kv) {
    return (len >= nq && len <= max_kv) ? static_cast<uint32_t>((len + kTile - 1) / kTile) : 0u;
}

// First tile of warp w when W warps share U tiles.
__device__ __forceinline__ uint32_t warp_start(uint32_t w, uint32_t W, uint32_t U) {
    return static_cast<uint32_t>(static_cast<unsigned long long>(w) * U / W);
}

// The warp whose range holds tile u (the last w with warp_start(w) <= u).
__device__ __forceinline__ uint32_t warp_of(uint32_t u, uint32_t W, uint32_t U) {
    return static_cast<uint32_t>(((static_cast<unsigned long long>(u) + 1) * W - 1) / U);
}

// Where tile u lives: sequence b, stream within the sequence (hk * row_groups +
// rg), tile t within the stream, and the stream's tile range.
struct TileLoc {
    int b, sis, t;
    uint32_t s_end;
};

__device__ __forceinline__ TileLoc locate(uint32_t u, const uint32_t* prefix, int B, int per_seq) {
    int lo = 0, hi = B - 1;   // largest b with prefix[b] <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    TileLoc L;
    L.b = lo;
    const uint32_t T = (prefix[lo + 1] - prefix[lo]) / per_seq;
    const uint32_t off = u - prefix[lo];
    L.sis = static_cast<int>(off / T);
    L.t = static_cast<int>(off - L.sis * T);
    L.s_end = prefix[lo] + (L.sis + 1) * T;
    return L;
}

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                        DecodeArgs a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t warp_sums[kWarps];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRing);
    uint32_t* prefix = reinterpret_cast<uint32_t*>(smem + C::kRing + C::kBarBytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(prefix + kMaxSeqs + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_seq = a.Hkv * a.row_groups;

    // ---- tile prefix over sequences (block-wide scan of per-sequence tile counts)
    {
        constexpr int kPer = (kMaxSeqs + 1 + kThreads - 1) / kThreads;
        const int b0 = threadIdx.x * kPer;
        uint32_t local[kPer];
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int b = b0 + i;
            uint32_t n = 0;
            if (b < a.B) {
                n = seq_tiles(a.kv_lens[b], a.nq, a.max_kv) * static_cast<uint32_t>(per_seq);
                if (n == 0 && blockIdx.x == 0) atomicOr(a.status, kDevBadLength);
            }
            local[i] = n;
            sum += n;
        }
        uint32_t incl = sum;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, sh);
            if (lane >= sh) incl += y;
        }
        if (lane == 31) warp_sums[warp] = incl;
        if (threadIdx.x == 0) {
            for (int s = 0; s < kWarps * C::kStages; ++s) mbar_init(&bars[s], 1);
            *abort_flag = 0;
            mbar_init_fence();
        }
        __syncthreads();
        uint32_t run = incl - sum;
        for (int w = 0; w < warp; ++w) run += warp_sums[w];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int b = b0 + i;
            if (b <= a.B) prefix[b] = run;   // prefix[B] = total
            run += local[i];
        }
        __syncthreads();
        if (blockIdx.x == 0)
            for (int b = threadIdx.x; b <= a.B; b += kThreads) a.prefix_out[b] = prefix[b];
    }
    // The merge grid may start launching now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t U = prefix[a.B];
    const uint32_t W = gridDim.x * kWarps;
    const uint32_t w = blockIdx.x * kWarps + warp;
    const uint32_t u_beg = warp_start(w, W, U), u_end = warp_start(w + 1, W, U);
    if (u_beg >= u_end) return;

    const WaitCtl wc{a.wait_limit, a.status, abort_flag};
    uint8_t* ring = smem + warp * C::kStages * C::kStageBytes;
    uint64_t* full = bars + warp * C::kStages;
    if (lane == 0) {
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }

    // First cache row ([page * ps + slot] space) of tile u, with its KV head in
    // the high bits' place: returned as (row, hk) packed in 64 bits.
    auto tile_src = [&](uint32_t u) -> long long {
        if (u >= u_end) return 0;
        const TileLoc L = locate(u, prefix, a.B, per_seq);
        const int tok = L.t * kTile;
        int page = a.table[static_cast<long long>(L.b) * a.max_pages + tok / a.ps];
        if (page < 0 || page >= a.num_phys) {
            atomicOr(a.status, kDevBadPage);
            page = 0;
        }
        const int hk = L.sis / a.row_groups;
        return (static_cast<long long>(hk) << 32) | static_cast<uint32_t>(page * a.ps + tok % a.ps);
    };
    auto issue = [&](uint32_t k, long long src) {   // stage k of this warp's range
        if (elect_one()) {
            const int slot = k % C::kStages;
            uint8_t* dst = ring + slot * C::kStageBytes;
            const int row = static_cast<int>(src & 0xFFFFFFFFLL), hk = static_cast<int>(src >> 32);
            mbar_arrive_expect_tx(&full[slot], C::kStageBytes);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(dst + h * C::kBox, &tk, &full[slot], 128 * h, hk, row);
                tma_load_3d(dst + (C::kHalves + h) * C::kBox, &tv, &full[slot], 128 * h, hk, row);
            }
        }
        __syncwarp();
    };

    const uint32_t n_tiles = u_end - u_beg;
    // test hook: the waits for stages never loaded run out (bounded) mid-range
    const uint32_t n_load = a.fault == 1 ? 0u
                            : a.fault == 2 ? min(n_tiles, static_cast<uint32_t>(2 * C::kStages))
                                           : n_tiles;
    long long src_cur = tile_src(u_beg + lane);          // tiles 0..31 of the range, one per lane
    long long src_next = tile_src(u_beg + 32 + lane);    // tiles 32..63
    uint32_t issued = 0;
    for (; issued < static_cast<uint32_t>(C::kStages - 1) && issued < n_load; ++issued)
        issue(issued, __shfl_sync(0xffffffffu, src_cur, issued));

    const int g = lane >> 2, c = lane & 3;
    const int grp = a.Hq / a.Hkv;
    float o[C::kSteps][4];
    float m_ref[2], l_sum[2];
    uint32_t qf[C::kSteps][2];
    TileLoc L = locate(u_beg, prefix, a.B, per_seq);
    int kv_len = 0, lim0 = 0, lim1 = 0, first_masked = 0;
    long long rec_id = 0;
    // Start of a stream segment: state reset and the Q operand of the stream's rows.
    auto begin_stream = [&]() {
        kv_len = a.kv_lens[L.b];
        const int hk = L.sis / a.row_groups, rg = L.sis - hk * a.row_groups;
        rec_id = static_cast<long long>(w) + static_cast<long long>(L.b) * per_seq + L.sis;
        const int r0 = rg * kRows + 2 * c, r1 = r0 + 1;
        lim0 = r0 < a.G ? kv_len - a.nq + (r0 % a.nq) : kv_len - 1;
        lim1 = r1 < a.G ? kv_len - a.nq + (r1 % a.nq) : kv_len - 1;
        first_masked = kv_len - a.nq + 1;
        // Q^T operand: k-step st covers, for lane quad c, the head-width
        // positions 128*(st/8) + 16*(2c + (st%8)/4) + 4*(st%4) + {0,1} and
        // {2,3}; the K operand reads the same positions.
        const int r = rg * kRows + g;
        const __half* qp = nullptr;
        if (r < a.G)
            qp = a.q + ((static_cast<long long>(L.b) * a.Hq + hk * grp + r / a.nq) * a.nq +
                        (r % a.nq)) * D;
#pragma unroll
        for (int st = 0; st < C::kSteps; ++st) {
            const int e = 128 * (st >> 3) + 16 * (2 * c + ((st & 7) >> 2)) + 4 * (st & 3);
            uint2 v = make_uint2(0, 0);
            if (qp) v = *reinterpret_cast<const uint2*>(qp + e);
            qf[st][0] = v.x;
            qf[st][1] = v.y;
        }
#pragma unroll
        for (int j = 0; j < C::kSteps; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
        m_ref[0] = m_ref[1] = -INFINITY;
        l_sum[0] = l_sum[1] = 0.0f;
    };
    begin_stream();

    bool aborted = false;
    for (uint32_t k = 0; k < n_tiles; ++k) {
        // keep the ring kStages - 1 tiles ahead
        if (issued < n_load) {
            if ((issued & 31u) == 0) {
                src_cur = src_next;
                src_next = tile_src(u_beg + issued + 32 + lane);
            }
            issue(issued, __shfl_sync(0xffffffffu, src_cur, issued & 31u));
            ++issued;
        }
        const int slot = k % C::kStages;
        if (!wait_warp(&full[slot], (k / C::kStages) & 1, wc)) {
            aborted = true;
            break;
        }
        const uint8_t* kst = ring + slot * C::kStageBytes;
        const uint8_t* vst = kst + C::kHalves * C::kBox;
        const int tb = L.t * kTile;   // first token of the tile

        // ---- S^T = K Q^T: 16 tokens (rows) x 8 query rows
        float acc[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[x][0] = acc[x][1] = acc[x][2] = acc[x][3] = 0.0f;
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int col = ((2 * c + qq) ^ g) << 4;   // rows g and g + 8: same swizzle phase
                const uint4 k0 = *reinterpret_cast<const uint4*>(kst + h * C::kBox + g * 128 + col);
                const uint4 k1 =
                    *reinterpret_cast<const uint4*>(kst + h * C::kBox + (g + 8) * 128 + col);
                const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
                const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const int st = 8 * h + 4 * qq + i4;
                    mma_16816(acc[st & 3], cvt_scaled<kMode>(w0[i4] & 0xFFFFu, a.ks2, a.ks),
                              cvt_scaled<kMode>(w1[i4] & 0xFFFFu, a.ks2, a.ks),
                              cvt_scaled<kMode>(w0[i4] >> 16, a.ks2, a.ks),
                              cvt_scaled<kMode>(w1[i4] >> 16, a.ks2, a.ks), qf[st][0], qf[st][1]);
                }
            }
        }
        // x[0]: token g, query 2c; x[1]: token g, query 2c+1; x[2], x[3]: token g+8.
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = ((acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e])) * a.sl2;
        if (tb + kTile > first_masked) {
            const int t0 = tb + g, t1 = tb + g + 8;
            if (t0 > lim0) x[0] = -INFINITY;
            if (t0 > lim1) x[1] = -INFINITY;
            if (t1 > lim0) x[2] = -INFINITY;
            if (t1 > lim1) x[3] = -INFINITY;
        }
        // ---- online softmax for this lane's query columns 2c, 2c+1
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const bool up0 = mx0 > m_ref[0] + kRescale, up1 = mx1 > m_ref[1] + kRescale;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float n0 = up0 ? mx0 : m_ref[0], n1 = up1 ? mx1 : m_ref[1];
            const float al0 = up0 ? fast_exp2(m_ref[0] - n0) : 1.0f;
            const float al1 = up1 ? fast_exp2(m_ref[1] - n1) : 1.0f;
            m_ref[0] = n0;
            m_ref[1] = n1;
            l_sum[0] *= al0;
            l_sum[1] *= al1;
#pragma unroll
            for (int j = 0; j < C::kSteps; ++j) {
                o[j][0] *= al0;
                o[j][2] *= al0;
                o[j][1] *= al1;
                o[j][3] *= al1;
            }
        }
        const float mu0 = m_ref[0] == -INFINITY ? 0.0f : m_ref[0];
        const float mu1 = m_ref[1] == -INFINITY ? 0.0f : m_ref[1];
        const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
        const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
        l_sum[0] += p0 + p2;
        l_sum[1] += p1 + p3;
        // ---- P^T operands: hi and lo FP16 halves, transposed by movmatrix
        const __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(p0 - f01.x, p1 - f01.y);
        const __half2 l23 = __floats2half2_rn(p2 - f23.x, p3 - f23.y);
        const uint32_t bh0 = movmatrix_trans(h2_bits(h01)), bh1 = movmatrix_trans(h2_bits(h23));
        const uint32_t bl0 = movmatrix_trans(h2_bits(l01)), bl1 = movmatrix_trans(h2_bits(l23));
        // ---- O^T += V^T P^T: V rows (tokens) 2c, 2c+1, 2c+8, 2c+9, column g
        const int v0 = 2 * c;
        const bool vtail = tb + kTile > kv_len;
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) {
            const uint8_t* vh = vst + h * C::kBox;
            uint4 ra = *reinterpret_cast<const uint4*>(vh + v0 * 128 + ((g ^ v0) << 4));
            uint4 rb = *reinterpret_cast<const uint4*>(vh + (v0 + 1) * 128 + ((g ^ (v0 + 1)) << 4));
            uint4 rc = *reinterpret_cast<const uint4*>(vh + (v0 + 8) * 128 + ((g ^ v0) << 4));
            uint4 rd = *reinterpret_cast<const uint4*>(vh + (v0 + 9) * 128 + ((g ^ (v0 + 1)) << 4));
            if (vtail) {   // tokens past the cache end may hold any byte (even NaN codes)
                const uint4 z = make_uint4(0, 0, 0, 0);
                if (tb + v0 >= kv_len) ra = z;
                if (tb + v0 + 1 >= kv_len) rb = z;
                if (tb + v0 + 8 >= kv_len) rc = z;
                if (tb + v0 + 9 >= kv_len) rd = z;
            }
            const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
            const uint32_t wc8[4] = {rc.x, rc.y, rc.z, rc.w}, wd[4] = {rd.x, rd.y, rd.z, rd.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const uint32_t e01 = __byte_perm(wa[wi], wb[wi], 0x5140);
                const uint32_t e89 = __byte_perm(wc8[wi], wd[wi], 0x5140);
                const uint32_t d01 = __byte_perm(wa[wi], wb[wi], 0x7362);
                const uint32_t d89 = __byte_perm(wc8[wi], wd[wi], 0x7362);
                {
                    const int j = 8 * h + 2 * wi;
                    const uint32_t x0 = cvt_scaled<kMode>(e01 & 0xFFFFu, a.vs2, a.vs);
                    const uint32_t x1 = cvt_scaled<kMode>(e01 >> 16, a.vs2, a.vs);
                    const uint32_t x2 = cvt_scaled<kMode>(e89 & 0xFFFFu, a.vs2, a.vs);
                    const uint32_t x3 = cvt_scaled<kMode>(e89 >> 16, a.vs2, a.vs);
                    mma_16816(o[j], x0, x1, x2, x3, bh0, bh1);
                    mma_16816(o[j], x0, x1, x2, x3, bl0, bl1);
                }
                {
                    const int j = 8 * h + 2 * wi + 1;
                    const uint32_t x0 = cvt_scaled<kMode>(d01 & 0xFFFFu, a.vs2, a.vs);
                    const uint32_t x1 = cvt_scaled<kMode>(d01 >> 16, a.vs2, a.vs);
                    const uint32_t x2 = cvt_scaled<kMode>(d89 & 0xFFFFu, a.vs2, a.vs);
                    const uint32_t x3 = cvt_scaled<kMode>(d89 >> 16, a.vs2, a.vs);
                    mma_16816(o[j], x0, x1, x2, x3, bh0, bh1);
                    mma_16816(o[j], x0, x1, x2, x3, bl0, bl1);
                }
            }
        }

        // ---- end of a stream segment: write the partial record, move on
        const uint32_t u = u_beg + k;
        if (u + 1 == L.s_end || k + 1 == n_tiles) {
            float ls0 = l_sum[0], ls1 = l_sum[1];
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                ls0 += __shfl_xor_sync(0xffffffffu, ls0, sh);
                ls1 += __shfl_xor_sync(0xffffffffu, ls1, sh);
            }
            float* po = a.part_o + rec_id * kRows * D;
            const int rbase = (L.sis % a.row_groups) * kRows;   // query rows of padding are skipped
            const bool real0 = rbase + 2 * c < a.G, real1 = rbase + 2 * c + 1 < a.G;
#pragma unroll
            for (int j = 0; j < C::kSteps; ++j) {
                const int d = pv_col(j, g);
                if (real0)
                    *reinterpret_cast<float2*>(po + (2 * c) * D + d) = make_float2(o[j][0], o[j][2]);
                if (real1)
                    *reinterpret_cast<float2*>(po + (2 * c + 1) * D + d) =
                        make_float2(o[j][1], o[j][3]);
            }
            if (g == 0) {
                if (real0) a.part_ml[rec_id * kRows + 2 * c] = make_float2(m_ref[0], ls0);
                if (real1) a.part_ml[rec_id * kRows + 2 * c + 1] = make_float2(m_ref[1], ls1);
            }
            if (k + 1 < n_tiles) {
                L = locate(u + 1, prefix, a.B, per_seq);
                begin_stream();
            }
        } else {
            ++L.t;
        }
    }
    if (aborted) {
        // Stages already issued must land before the CTA's shared memory goes away.
        if (lane == 0) {
            for (uint32_t k = issued > C::kStages ? issued - C::kStages : 0; k < issued; ++k) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[k % C::kStages], (k / C::kStages) & 1))
                    if (global_timer_ns() - t0 > a.wait_limit) break;
            }
        }
        __syncwarp();
    }
}

// Combine the partial records of every query row: with m_r, l_r the max (log2
// units) and sum of record r, M = max_r m_r, L = sum_r 2^(m_r - M) l_r,
// O = out_mul * sum_r 2^(m_r - M) O_r / L and lse = (M + log2 L) ln 2.  The
// records of a row are those of the warps whose tile ranges meet its stream.
// One CTA takes one row and a 32-wide slice of the head width: 8 lanes cover
// the slice (one float4 each) and 64 lane groups take every 64th record, so
// many record loads are in flight at once.  Each lane group folds its records
// in one pass (a running max, as in the online softmax), and the groups' results
// are folded the same way.  A rejected sequence (no tiles) gets O = 0,
// lse = -inf.
template <int D>
__global__ void __launch_bounds__(512, 2) decode_merge_kernel(const float* __restrict__ part_o,
                                                           const float2* __restrict__ part_ml,
                                                           const uint32_t* __restrict__ prefix,
                                                           int B, int Hq, int Hkv, int nq,
                                                           int row_groups, uint32_t W, float out_mul,
                                                           __half* __restrict__ o,
                                                           float* __restrict__ lse) {
    __shared__ float red[16];
    __shared__ float4 part[16][8];
    __shared__ float lpart[16];
    const long long row = blockIdx.x;
    const int slice = blockIdx.y;
    const int tid = threadIdx.x, f4 = tid & 7, rl = tid >> 3;
    const int per_b = Hq * nq;
    const int b = static_cast<int>(row / per_b);
    const int within = static_cast<int>(row - static_cast<long long>(b) * per_b);
    const int head = within / nq, i = within - head * nq;
    const int grp = Hq / Hkv;
    const int hk = head / grp, r = (head - hk * grp) * nq + i;
    const int rg = r / kRows, n = r - rg * kRows;
    const int per_seq = Hkv * row_groups;
    // Launched as a programmatic dependent of the decode grid: wait for its
    // prefix table and records before reading them.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t U = prefix[B];
    const uint32_t T = (prefix[b + 1] - prefix[b]) / per_seq;

    uint32_t w0 = 1, w1 = 0;   // empty unless the sequence has tiles
    long long s_index = 0;
    if (T > 0) {
        const int sis = hk * row_groups + rg;
        const uint32_t u0 = prefix[b] + sis * T;
        w0 = warp_of(u0, W, U);
        w1 = warp_of(u0 + T - 1, W, U);
        s_index = static_cast<long long>(b) * per_seq + sis;
    }
    // With at least as many tiles as warps every warp range is non-empty, and
    // the per-record emptiness test (two 64-bit divisions) is skipped.
    const bool all_busy = U >= W;
    // One pass: every lane keeps its own running max, sum and weighted O slice
    // over its records, and the lanes are then folded pairwise.
    float mx = -INFINITY, lw = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // Records are fetched 6 per lane group at a time, all loads issued before
    // any of them is used, so one round of L2 latency covers 384 records.
    constexpr int kBatch = 6;
    for (uint32_t wb = w0 + rl; wb <= w1; wb += 64 * kBatch) {
        float2 ml[kBatch];
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const uint32_t w = wb + 64 * j;
            ml[j] = make_float2(-INFINITY, 0.0f);
            v[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (w <= w1 && (all_busy || warp_start(w, W, U) < warp_start(w + 1, W, U))) {
                const long long rec = (w + s_index) * kRows + n;
                ml[j] = part_ml[rec];
                v[j] = *reinterpret_cast<const float4*>(part_o + rec * D + slice * 32 + f4 * 4);
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (ml[j].x > mx) {   // a larger max: rescale what this lane holds
                const float sc = mx == -INFINITY ? 0.0f : exp2f(mx - ml[j].x);
                acc = make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
                lw *= sc;
                mx = ml[j].x;
            }
            const float wc = ml[j].x == -INFINITY ? 0.0f : exp2f(ml[j].x - mx);
            acc = make_float4(acc.x + wc * v[j].x, acc.y + wc * v[j].y, acc.z + wc * v[j].z,
                              acc.w + wc * v[j].w);
            lw += wc * ml[j].y;
        }
    }
    // (m1, l1, a1) <- the combination of (m1, l1, a1) and (m2, l2, a2)
    auto fold = [](float& m1, float& l1, float4& a1, float m2, float l2, float4 a2) {
        const float m = fmaxf(m1, m2);
        const float s1 = m1 == -INFINITY ? 0.0f : exp2f(m1 - m);
        const float s2 = m2 == -INFINITY ? 0.0f : exp2f(m2 - m);
        a1 = make_float4(a1.x * s1 + a2.x * s2, a1.y * s1 + a2.y * s2, a1.z * s1 + a2.z * s2,
                         a1.w * s1 + a2.w * s2);
        l1 = l1 * s1 + l2 * s2;
        m1 = m;
    };
    // Fold the 64 record lanes: 4 per warp by shuffles, then the 16 warps.
#pragma unroll
    for (int sh = 8; sh < 32; sh <<= 1) {
        const float4 ao = make_float4(__shfl_xor_sync(0xffffffffu, acc.x, sh),
                                      __shfl_xor_sync(0xffffffffu, acc.y, sh),
                                      __shfl_xor_sync(0xffffffffu, acc.z, sh),
                                      __shfl_xor_sync(0xffffffffu, acc.w, sh));
        const float lo = __shfl_xor_sync(0xffffffffu, lw, sh);
        const float mo = __shfl_xor_sync(0xffffffffu, mx, sh);
        fold(mx, lw, acc, mo, lo, ao);
    }
    const int wid = tid >> 5;
    if ((tid & 31) < 8) {
        part[wid][f4] = acc;
        if (f4 == 0) {
            lpart[wid] = lw;
            red[wid] = mx;
        }
    }
    __syncthreads();
    if (tid >= 8) return;
    float M = red[0], L = lpart[0];
    float4 sacc = part[0][f4];
#pragma unroll
    for (int k = 1; k < 16; ++k) fold(M, L, sacc, red[k], lpart[k], part[k][f4]);
    const float inv = L > 0.0f ? out_mul / L : 0.0f;
    uint2 out;
    out.x = pack_half2(sacc.x * inv, sacc.y * inv);
    out.y = pack_half2(sacc.z * inv, sacc.w * inv);
    *reinterpret_cast<uint2*>(o + row * D + slice * 32 + f4 * 4) = out;
    if (lse && slice == 0 && f4 == 0)
        lse[row] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

bool power_of_two_in(float s, int lo, int hi) {
    int e = 0;
    const float m = frexpf(s, &e);   // s = m * 2^e, m in [0.5, 1)
    return m == 0.5f && e - 1 >= lo && e - 1 <= hi;
}

int scale_mode(float ks, float vs) {
    if (power_of_two_in(ks, -15, 7) && power_of_two_in(vs, -15, 7)) return kScaleFolded;
    if (is_fp16_value(ks) && is_fp16_value(vs)) return kScaleHalf;
    return kScaleGeneral;
}

size_t record_bytes(int D) { return static_cast<size_t>(kRows) * (static_cast<size_t>(D) * 4 + 8); }

// Workspace: partial records for W warps plus one per stream boundary, then the
// (B + 1)-entry tile prefix.
size_t decode_workspace(long long warps, long long streams, int B, int D) {
    return static_cast<size_t>(warps + streams) * record_bytes(D) +
           (static_cast<size_t>(B) + 1) * 4 + 16;
}

int sm_count_or_default() {
    DeviceState d;
    return current_device(&d) == GBATTN_OK ? d.num_sms : 148;
}

template <int D, int kMode>
int launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, int ctas, const DecodeArgs& a,
                  cudaStream_t s) {
    static std::once_flag once[64];
    static int rc[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBATTN_ERR_CUDA;
    std::call_once(once[dev], [&] {
        rc[dev] = cudaFuncSetAttribute(paged_decode_kernel<D, kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<D>::kSmem) == cudaSuccess
                      ? GBATTN_OK
                      : GBATTN_ERR_CUDA;
    });
    if (rc[dev] != GBATTN_OK) return rc[dev];
    paged_decode_kernel<D, kMode><<<ctas, kThreads, Cfg<D>::kSmem, s>>>(tk, tv, a);
    count_launches(1);
    return launch_status();
}

template <int D>
int launch_decode_mode(int mode, const CUtensorMap& tk, const CUtensorMap& tv, int ctas,
                       const DecodeArgs& a, cudaStream_t s) {
    if (mode == kScaleFolded) return launch_decode<D, kScaleFolded>(tk, tv, ctas, a, s);
    if (mode == kScaleHalf) return launch_decode<D, kScaleHalf>(tk, tv, ctas, a, s);
    return launch_decode<D, kScaleGeneral>(tk, tv, ctas, a, s);
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" size_t attn_paged_decode_workspace_size(int B, int Hq, int Hkv, int nq, int max_kv_len,
                                                   int D) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || nq <= 0 || max_kv_len <= 0 || D <= 0 || Hq % Hkv != 0)
        return 0;
    const int rgs = (Hq / Hkv * nq + kRows - 1) / kRows;
    const long long warps = static_cast<long long>(sm_count_or_default()) * kWarps;
    return decode_workspace(warps, static_cast<long long>(B) * Hkv * rgs, B, D);
}

extern "C" int attn_paged_decode_fwd(const void* q, const uint8_t* k_pages, const uint8_t* v_pages,
                                     const int32_t* page_table, const int32_t* kv_lens, void* o,
                                     float* lse, int B, int Hq, int Hkv, int nq, int D,
                                     int num_phys_pages, int page_size, int max_pages,
                                     int max_kv_len, float k_scale, float v_scale, float scale,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    CallRange nvtx_range("attn_paged_decode_fwd");
    if (!q || !k_pages || !v_pages || !page_table || !kv_lens || !o) return GBATTN_ERR_NULL;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || nq <= 0 || num_phys_pages <= 0 || page_size <= 0 ||
        max_pages <= 0 || max_kv_len <= 0)
        return GBATTN_ERR_SHAPE;
    if (Hq % Hkv != 0 || nq > max_kv_len ||
        static_cast<long long>(max_kv_len) > static_cast<long long>(max_pages) * page_size)
        return GBATTN_ERR_SHAPE;
    if (D != 128 && D != 256) return GBATTN_ERR_UNSUPPORTED;
    if (page_size < 16 || (page_size & (page_size - 1)) != 0 ||
        static_cast<long long>(num_phys_pages) * page_size > 0x7FFFFFFFLL)
        return GBATTN_ERR_UNSUPPORTED;
    if (B > kMaxSeqs) return GBATTN_ERR_UNSUPPORTED;
    const int G = Hq / Hkv * nq;
    const int rgs = (G + kRows - 1) / kRows;
    const long long streams = static_cast<long long>(B) * Hkv * rgs;
    const long long max_tiles = streams * ((max_kv_len + kTile - 1) / kTile);
    if (max_tiles > 0x7FFFFFFFLL || static_cast<long long>(B) * Hq * nq > 0x7FFFFFFFLL)
        return GBATTN_ERR_SHAPE;
    if (!finite_positive(scale) || !finite_positive(k_scale) || !finite_positive(v_scale))
        return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(kv_lens) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    const long long rows = static_cast<long long>(B) * Hq * nq;
    const size_t qb = static_cast<size_t>(rows) * D * 2;
    const size_t pb = static_cast<size_t>(num_phys_pages) * page_size * Hkv * D;
    const size_t tb = static_cast<size_t>(B) * max_pages * 4;
    const size_t kb = static_cast<size_t>(B) * 4;
    const size_t lb = static_cast<size_t>(rows) * 4;
    if (overlaps(o, qb, q, qb) || overlaps(o, qb, k_pages, pb) || overlaps(o, qb, v_pages, pb) ||
        overlaps(o, qb, page_table, tb) || overlaps(o, qb, kv_lens, kb) ||
        overlaps(lse, lb, q, qb) || overlaps(lse, lb, k_pages, pb) ||
        overlaps(lse, lb, v_pages, pb) || overlaps(lse, lb, page_table, tb) ||
        overlaps(lse, lb, kv_lens, kb) || overlaps(lse, lb, o, qb))
        return GBATTN_ERR_ALIAS;
    if (!workspace) return GBATTN_ERR_WORKSPACE;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;

    // One CTA of 8 warps per SM; fewer when the workspace holds fewer records.
    long long ctas = dev.num_sms;
    while (ctas > 1 && decode_workspace(ctas * kWarps, streams, B, D) > workspace_bytes) --ctas;
    const size_t wb = decode_workspace(ctas * kWarps, streams, B, D);
    if (wb > workspace_bytes) return GBATTN_ERR_WORKSPACE;
    if (overlaps(workspace, wb, q, qb) || overlaps(workspace, wb, k_pages, pb) ||
        overlaps(workspace, wb, v_pages, pb) || overlaps(workspace, wb, page_table, tb) ||
        overlaps(workspace, wb, kv_lens, kb) || overlaps(workspace, wb, o, qb) ||
        overlaps(workspace, wb, lse, lb))
        return GBATTN_ERR_ALIAS;

    CUtensorMap tk, tv;
    const uint64_t total_rows = static_cast<uint64_t>(num_phys_pages) * page_size;
    if (encode_tmap_u8_pages(&tk, k_pages, D, Hkv, total_rows, kTile) != GBATTN_OK ||
        encode_tmap_u8_pages(&tv, v_pages, D, Hkv, total_rows, kTile) != GBATTN_OK)
        return GBATTN_ERR_CUDA;

    const int mode = scale_mode(k_scale, v_scale);
    const size_t n_rec = static_cast<size_t>(ctas * kWarps + streams);
    DecodeArgs a{};
    a.q = static_cast<const __half*>(q);
    a.table = page_table;
    a.kv_lens = kv_lens;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = reinterpret_cast<float2*>(a.part_o + n_rec * kRows * D);
    a.prefix_out = reinterpret_cast<uint32_t*>(a.part_ml + n_rec * kRows);
    a.status = dev.status;
    a.wait_limit = wait_limit_ns();
    a.fault = fault_mode();
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.nq = nq;
    a.G = G;
    a.row_groups = rgs;
    a.num_phys = num_phys_pages;
    a.ps = page_size;
    a.max_pages = max_pages;
    a.max_kv = max_kv_len;
    a.sl2 = scale * 1.4426950408889634f * (mode == kScaleFolded ? k_scale : 1.0f);
    a.ks = k_scale;
    a.vs = v_scale;
    a.ks2 = __float2half2_rn(k_scale);
    a.vs2 = __float2half2_rn(v_scale);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = D == 256 ? launch_decode_mode<256>(mode, tk, tv, static_cast<int>(ctas), a, s)
                  : launch_decode_mode<128>(mode, tk, tv, static_cast<int>(ctas), a, s);
    if (rc != GBATTN_OK) return rc;
    const float out_mul = mode == kScaleFolded ? v_scale : 1.0f;
    const uint32_t W = static_cast<uint32_t>(ctas * kWarps);
    // The merge is a programmatic dependent launch: its CTAs are placed as
    // decode CTAs retire and wait (griddepcontrol.wait) for the whole decode
    // grid, which hides the launch gap between the two kernels.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), D / 32);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    __half* oh = static_cast<__half*>(o);
    const cudaError_t e =
        D == 256 ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<256>, a.part_o,
                                      static_cast<const float2*>(a.part_ml),
                                      static_cast<const uint32_t*>(a.prefix_out), B, Hq, Hkv, nq,
                                      rgs, W, out_mul, oh, lse)
                 : cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, a.part_o,
                                      static_cast<const float2*>(a.part_ml),
                                      static_cast<const uint32_t*>(a.prefix_out), B, Hq, Hkv, nq,
                                      rgs, W, out_mul, oh, lse);
    count_launches(1);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GBATTN_ERR_CUDA;
    }
    return launch_status();
}
