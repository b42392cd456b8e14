// Dense non-causal attention on sm_103a, D = 128: O = softmax(scale * Q K^T) V
// with FP16 Q/K/V/P/O, FP32 accumulation in tensor memory and an FP32 online
// softmax ("Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation:
// FP32 QK/PV accumulation, FP16 probabilities and output).
//
// The one-query-tile-per-CTA form of the attention pipeline in attn.cu (which
// also runs causal, masked, paged and VSA attention and, for VSA, persistent
// CTAs), kept as its own kernel: with everything but the dense path taken out,
// the compiler schedules its loops measurably better (2-4% on dense video
// attention on GB300) than the same path inside the general kernel.
//
// One CTA owns a 128-row query tile of one head and walks every 128-key tile
// (two adjacent 64-key halves).  Warp roles (352 threads):
//   warp 0      TMA producer: Q once, then K and V tiles through a 4-slot ring in
//               the order the MMAs consume them (K0 .. K2, V0, K3, V1, ...).
//   warp 1      allocates tensor memory and issues S = Q K_t^T (SMEM x SMEM).
//   warp 10     issues O += P_j V_j (P from TMEM).  Each issuing warp is
//               converged and one elected lane issues each group.
//   warps 2..9  softmax: two threads per query row (TMEM lane = row), one per
//               64-key half of the tile; they exchange the partial row max;
//               exp2 with packed FP32 pairs, row sum, P -> FP16 into TMEM; lazy
//               O rescaling (only when the running max grows by more than 2^8),
//               each thread on its half of O; epilogue O / l.
// Tensor memory (512 columns): three S buffers of 128 FP32 columns (P_j
// overwrites the first 64 columns of its buffer as FP16 pairs), then O.  QK runs
// up to three tiles ahead; QK_t waits for PV_{t-3}, which read P from its buffer.
//
// Every wait is bounded in time (see WaitCtl): a wait that runs out records
// GBATTN_DEV_WAIT_TIMEOUT in the device status word, the CTA stops, waits a
// bounded time for its copies and MMAs in flight, frees tensor memory and exits.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "host.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kD = 128;              // head width
constexpr int kBM = 128;             // query rows per CTA
constexpr int kBN = 128;             // keys per tile (two halves of 64)
constexpr int kNS = 4;               // K/V ring slots
constexpr int kNSB = 3;              // S buffers in TMEM (QK lookahead)
constexpr int kThreads = 352;
constexpr int kPvWarp = 10;
constexpr int kSoftmaxThreads = 256;
constexpr int kChunk = 128 * 128;    // 128 rows x 64 FP16 columns
constexpr int kHalf = 64 * 128;      // 64 rows x 64 columns
constexpr int kKch = kD / 64;
constexpr int kQBytes = kBM * kD * 2;
constexpr int kSlotBytes = kBN * kD * 2;
constexpr uint32_t kTO = kNSB * 128;  // first TMEM column of O
static_assert(kTO + kD <= 512, "tensor memory budget");
constexpr uint32_t kIdescQK = idesc_f16(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = idesc_f16(kBM, kD, false, true);
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s for draining after an abort

struct DenseArgs {
    int seq_q, seq_k;   // query rows and keys per head
    int hq;             // heads per batch entry
    float scale_log2;   // scale * log2(e)
    __half* o;
    long long o_sb, o_sh, o_sr;   // element strides of O between batch entries, heads, rows
    float* lse;         // optional natural-log LSE [B*H][seq_q]
    uint32_t* status;
    uint64_t wait_limit;
    int fault;          // test hook: 1 = the TMA warp never loads Q; 2 = it stops after 2*NS K/V items
};

struct Ctrl {
    uint64_t q_full;
    uint64_t full[kNS];
    uint64_t empty[kNS];
    uint64_t s_full[kNSB];    // QK_j done (buffer j % NSB)
    uint64_t p_full[kNSB];    // P_j written (buffer j % NSB)
    uint64_t pv_done[kNSB];   // PV_j done (barrier j % NSB).  QK_j is issued after
                              // PV_{j-NSB}, so once S_j is visible the previous phase
                              // of every barrier awaited below has completed.
    uint64_t drain;
    uint64_t drain_pv;        // the PV issuer's own drain after an abort
    uint64_t xchg[4];         // per row quarter: the two half-row threads exchange values
    uint32_t tmem_base;
    int abort;
};

// Values exchanged between the two threads that share a query row.
struct Exchange {
    float mx[2][2][128];   // [tile parity][column half][row] partial row max
    float l[2][128];       // [column half][row] partial row sum (epilogue)
};

constexpr int kCtrlBytes = 256 + static_cast<int>(sizeof(Exchange));
static_assert(sizeof(Ctrl) <= 256, "control block");
constexpr int kSmemBytes = 1024 + kQBytes + kNS * kSlotBytes + kCtrlBytes;

// Bounded wait that ignores the abort flag (used only to drain after an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainNs) return;
    }
}

// Item order of the K/V ring = the MMA warps' consumption order with a QK
// lookahead of L tiles: K_0 .. K_{L-1}, then (V_j, K_{j+L}) while j + L < n,
// then the remaining V_j.
__device__ __forceinline__ void ring_item(int it, int n, int L, int& tile, bool& is_v) {
    const int k0 = min(n, L);
    if (it < k0) { tile = it; is_v = false; return; }
    const int r = it - k0;
    const int m = max(n - L, 0);
    if (r < 2 * m) {
        if (r & 1) { tile = (r >> 1) + L; is_v = false; }
        else { tile = r >> 1; is_v = true; }
        return;
    }
    tile = m + (r - 2 * m);
    is_v = true;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_dense_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const DenseArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + kQBytes;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(sKV + kNS * kSlotBytes);
    Exchange* ex = reinterpret_cast<Exchange*>(reinterpret_cast<uint8_t*>(ctrl) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = static_cast<int>(blockIdx.y);
    const int q_row0 = static_cast<int>(blockIdx.x) * kBM;
    const int n_tiles = (a.seq_k + kBN - 1) / kBN;
    // 4-D tensor-map coordinates (head, batch entry)
    const int qb = bh / a.hq, qh = bh - qb * a.hq;

    // ---- prologue
    if (threadIdx.x == 0) {
        mbar_init(&ctrl->q_full, 1);
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&ctrl->full[i], 1);
            mbar_init(&ctrl->empty[i], 1);
        }
        for (int i = 0; i < kNSB; ++i) {
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->p_full[i], kSoftmaxThreads);
        }
        for (int i = 0; i < kNSB; ++i) mbar_init(&ctrl->pv_done[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&ctrl->xchg[i], 64);
        mbar_init(&ctrl->drain, 1);
        mbar_init(&ctrl->drain_pv, 1);
        ctrl->abort = 0;
        mbar_init_fence();
    }
    // The query tile's copy (one elected lane of the TMA warp).
    auto issue_q = [&]() {
        if (elect_one()) {
            mbar_arrive_expect_tx(&ctrl->q_full, kQBytes);
#pragma unroll
            for (int c = 0; c < kKch; ++c)
                tma_load_4d(sQ + c * kChunk, &tmQ, &ctrl->q_full, c * 64, q_row0, qh, qb);
        }
        __syncwarp();
    };
    const bool load_q = a.fault != 1;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        __syncwarp();   // the barriers thread 0 initialised are visible to the warp
    }
    if (warp == 1) {
        tmem_alloc(&ctrl->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const WaitCtl w{a.wait_limit, a.status, &ctrl->abort};

    // S_t = Q K_t^T into S buffer buf; O += P_j V_j with P_j read from S buffer buf.
    auto issue_qk = [&](int slot, int buf) {
        const uint32_t qa = smem_addr(sQ);
        const uint32_t ka = smem_addr(sKV + slot * kSlotBytes);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16) {
            const uint32_t off = (k16 >> 2) * kChunk + (k16 & 3) * 32;
            mma_ss(tmem + buf * 128, sdesc_sw128(qa + off, 16, 1024),
                   sdesc_sw128(ka + off, 16, 1024), kIdescQK, k16 > 0 ? 1u : 0u);
        }
    };
    auto issue_pv = [&](int slot, int buf, bool acc) {
        const uint32_t va = smem_addr(sKV + slot * kSlotBytes);
#pragma unroll
        for (int k16 = 0; k16 < kBN / 16; ++k16)
            mma_ts(tmem + kTO, tmem + buf * 128 + k16 * 8,
                   sdesc_sw128(va + k16 * 2048, kChunk, 1024), kIdescPV,
                   (acc || k16 > 0) ? 1u : 0u);
    };
    // Ring positions (the TMA warp's load order, see ring_item) of K_t and V_j.
    auto pos_k = [&](int t) { return t < kNSB ? t : kNSB + 2 * (t - kNSB) + 1; };
    auto pos_v = [&](int j) { return min(n_tiles, kNSB) + j + min(j, max(0, n_tiles - kNSB)); };

    if (warp == 0) {
        // ================= TMA producer (whole warp; one elected lane issues)
        if (n_tiles > 0) {
            int last_it[kNS] = {-1, -1, -1, -1};
            if (load_q) issue_q();
            bool ok = true;
            for (int it = 0; it < 2 * n_tiles; ++it) {
                if (a.fault == 2 && it >= 2 * kNS) {   // test hook: stop mid-stream, drain, leave
                    ok = false;
                    break;
                }
                const int slot = it % kNS;
                if (!wait_warp(&ctrl->empty[slot], ((it / kNS) & 1) ^ 1u, w)) { ok = false; break; }
                int t;
                bool is_v;
                ring_item(it, n_tiles, kNSB, t, is_v);
                const int k0 = t * kBN, k1 = k0 + 64;
                const CUtensorMap* m = is_v ? &tmV : &tmK;
                uint8_t* dst = sKV + slot * kSlotBytes;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&ctrl->full[slot], kSlotBytes);
#pragma unroll
                    for (int c = 0; c < kKch; ++c) {
                        tma_load_4d(dst + c * kChunk, m, &ctrl->full[slot], c * 64, k0, qh, qb);
                        tma_load_4d(dst + c * kChunk + kHalf, m, &ctrl->full[slot], c * 64, k1, qh, qb);
                    }
                }
                __syncwarp();
                last_it[slot] = it;
            }
            if (!ok && lane == 0) {   // let copies in flight land before the CTA exits
                if (load_q) drain_wait(&ctrl->q_full, 0);
                for (int s = 0; s < kNS; ++s)
                    if (last_it[s] >= 0) drain_wait(&ctrl->full[s], (last_it[s] / kNS) & 1);
            }
        }
    } else if (warp == 1) {
        // ================= QK issuer (whole warp waits; one elected lane issues
        // each group of MMAs and its commits).  QK_t overwrites the S buffer that
        // PV_{t-NSB} read P_{t-NSB} from, so it waits for that PV to finish.  A
        // parity wait on a slot is unambiguous only if the slot's previous item is
        // known to have landed: here it is either an earlier K (this warp waited
        // for it) or a V_i that precedes K_t in the ring, so i <= t-NSB (K_t
        // follows V_{t-NSB}) and PV_i finished with PV_{t-NSB}.
        if (n_tiles > 0) {
            bool ok = wait_warp(&ctrl->q_full, 0, w);
            for (int t = 0; ok && t < n_tiles; ++t) {
                const int pos = pos_k(t);
                const int slot = pos % kNS;
                const int buf = t % kNSB;
                if (t >= kNSB) ok = wait_warp(&ctrl->pv_done[buf], ((t - kNSB) / kNSB) & 1, w);
                ok = ok && wait_warp(&ctrl->full[slot], (pos / kNS) & 1, w);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_qk(slot, buf);
                    mma_commit(&ctrl->s_full[buf]);
                    mma_commit(&ctrl->empty[slot]);
                }
                __syncwarp();
            }
            if (!ok) {   // wait for issued MMAs before tensor memory is freed
                if (elect_one()) mma_commit(&ctrl->drain);
                __syncwarp();
                if (lane == 0) drain_wait(&ctrl->drain, 0);
            }
        }
    } else if (warp == kPvWarp) {
        // ================= PV issuer (whole warp waits, one elected lane issues).
        // PV_j waits for P_j (the softmax is done with S_j, so every QK_t with
        // t <= j has finished) and for V_j in the ring.  The slot's previous item
        // is an earlier V (this warp waited for it) or a K_t with t <= j, both
        // known to have landed (the 4-slot ring never puts a later K there).
        if (n_tiles > 0) {
            bool ok = true;
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int pos = pos_v(j);
                const int slot = pos % kNS;
                const int buf = j % kNSB;
                ok = wait_warp(&ctrl->p_full[buf], (j / kNSB) & 1, w);
                ok = ok && wait_warp(&ctrl->full[slot], (pos / kNS) & 1, w);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_pv(slot, buf, j > 0);
                    mma_commit(&ctrl->empty[slot]);
                    mma_commit(&ctrl->pv_done[buf]);
                }
                __syncwarp();
            }
            if (!ok) {   // wait for issued MMAs before tensor memory is freed
                if (elect_one()) mma_commit(&ctrl->drain_pv);
                __syncwarp();
                if (lane == 0) drain_wait(&ctrl->drain_pv, 0);
            }
        }
    } else {
        // ================= softmax / correction / epilogue (warps 2..9)
        // Two threads share each query row: warps 2..5 own key columns 0..63 of
        // every tile, warps 6..9 columns 64..127 (TMEM lane quarter = warp % 4).
        // They exchange their partial row max each tile (and the row sums at the
        // end) through shared memory, ordered by the per-quarter xchg mbarrier.
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const long long row_g = static_cast<long long>(q_row0) + row;
        uint64_t* xbar = &ctrl->xchg[quarter];
        const int lim = a.seq_k;   // keys >= lim are invisible (past the end)
        const float sl2 = a.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        float m_run = -INFINITY, l = 0.0f;
        uint32_t xphase = 0;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int buf = j % kNSB;
            const uint32_t sbuf = tl + buf * 128;
            ok = wait_warp(&ctrl->s_full[buf], (j / kNSB) & 1, w);
            if (!ok) break;
            tc_fence_after();
            uint32_t s[64];
            tmem_ld32(sbuf + half * 64, s);
            tmem_ld32(sbuf + half * 64 + 32, s + 32);
            tmem_ld_wait();

            const int kh = j * kBN + half * 64;
            if (kh + 64 > lim) {   // keys past the end
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (kh + c >= lim) s[c] = __float_as_uint(-INFINITY);
            }
            // row max of the 64 values with four independent chains (short latency):
            // s[0..3] start the chains, s[4..59] in seven steps of eight, s[60..63] last
            float m4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) m4[k] = __uint_as_float(s[k]);
#pragma unroll
            for (int c = 4; c < 60; c += 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    m4[k] = max3f(m4[k], __uint_as_float(s[c + k]), __uint_as_float(s[c + 4 + k]));
            }
            m4[0] = max3f(m4[0], __uint_as_float(s[60]), __uint_as_float(s[61]));
            m4[1] = max3f(m4[1], __uint_as_float(s[62]), __uint_as_float(s[63]));
            const float pm = fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
            ex->mx[j & 1][half][row] = pm;
            tc_fence_before();   // our S loads are ordered before the partner's P stores
            mbar_arrive(xbar);
            ok = wait_warp(xbar, xphase, w);
            xphase ^= 1u;
            if (!ok) break;
            tc_fence_after();
            const float mx = fmaxf(pm, ex->mx[j & 1][half ^ 1][row]);
            const float m_new = fmaxf(m_run, mx * sl2);
            const bool need = m_new > m_run + 8.0f;
            float alpha = 1.0f;
            if (need) {
                alpha = fast_exp2(m_run - m_new);
                m_run = m_new;
            }
            const bool warp_need = __any_sync(0xffffffffu, need);
            const float m_use = m_run == -INFINITY ? 0.0f : m_run;
            const uint64_t negm = f2_pack(-m_use, -m_use);
            uint64_t rs[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) rs[k] = f2_pack(0.0f, 0.0f);
            uint32_t p2[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                 sl2x2, negm),
                          x0, x1);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                rs[i & 3] = f2_add(rs[i & 3], f2_pack(p0, p1));   // four independent sums
                p2[i] = pack_half2(p0, p1);
            }
            float r0, r1, r2, r3, r4, r5, r6, r7;
            f2_unpack(rs[0], r0, r1);
            f2_unpack(rs[1], r2, r3);
            f2_unpack(rs[2], r4, r5);
            f2_unpack(rs[3], r6, r7);
            l = l * alpha + (((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7)));
            // P_j over the first 64 columns of its S buffer; both threads of the
            // row have loaded their S halves (they passed the exchange above).
            tmem_st32(sbuf + half * 32, p2);
            tmem_st_wait();
            if (warp_need && j > 0) {   // rescale this thread's half of O after PV_{j-1}
                ok = wait_warp(&ctrl->pv_done[(j - 1) % kNSB], ((j - 1) / kNSB) & 1, w);
                if (!ok) break;
                tc_fence_after();
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int cc = 0; cc < kD / 64; ++cc) {
                    const uint32_t col = tl + kTO + half * (kD / 2) + cc * 32;
                    uint32_t o[32];
                    tmem_ld32(col, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float y0, y1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2),
                                  y0, y1);
                        o[2 * e] = __float_as_uint(y0);
                        o[2 * e + 1] = __float_as_uint(y1);
                    }
                    tmem_st32(col, o);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(&ctrl->p_full[buf]);
        }
        if (ok && n_tiles > 0) {
            ok = wait_warp(&ctrl->pv_done[(n_tiles - 1) % kNSB], ((n_tiles - 1) / kNSB) & 1, w);
            tc_fence_after();
        }
        if (ok) {   // combine the two partial row sums
            ex->l[half][row] = l;
            mbar_arrive(xbar);
            ok = wait_warp(xbar, xphase, w);
            if (ok) l += ex->l[half ^ 1][row];
        }
        if (ok) {
            const bool row_ok = row_g < a.seq_q;
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            const float lse2 = l > 0.0f ? m_run + __log2f(l) : -INFINITY;
            const long long orow = static_cast<long long>(bh) * a.seq_q + row_g;
#pragma unroll 1
            for (int cc = 0; cc < kD / 64; ++cc) {
                const int c0 = half * (kD / 2) + cc * 32;   // first output column of this chunk
                uint32_t o[32];
                if (n_tiles > 0) {
                    tmem_ld32(tl + kTO + c0, o);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (!row_ok) continue;
                uint4* dst = reinterpret_cast<uint4*>(a.o + qb * a.o_sb + qh * a.o_sh + row_g * a.o_sr + c0);
                float y[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) y[e] = __uint_as_float(o[e]) * inv_l;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t hw[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f) hw[f] = pack_half2(y[8 * e + 2 * f], y[8 * e + 2 * f + 1]);
                    dst[e] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                }
            }
            if (row_ok && half == 0 && a.lse) a.lse[orow] = lse2 * 0.69314718055994531f;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" int attn_dense_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Sq, int Skv, int D, const int64_t* q_strides,
                              const int64_t* kv_strides, const int64_t* o_strides, float scale,
                              void* stream) {
    CallRange nvtx_range("attn_dense_fwd");
    if (!q || !k || !v || !o) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || Sq <= 0 || Skv <= 0) return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    if (D != kD) return GBATTN_ERR_UNSUPPORTED;
    Strides qs, kvs, os;
    if (!make_strides(q_strides, B, H, Sq, D, false, &qs) ||
        !make_strides(kv_strides, B, H, Skv, D, false, &kvs) ||
        !make_strides(o_strides, B, H, Sq, D, true, &os))
        return GBATTN_ERR_SHAPE;
    if (!finite_positive(scale)) return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t qb = strided_bytes(qs, B, H, Sq, D);
    const size_t kb = strided_bytes(kvs, B, H, Skv, D);
    const size_t ob = strided_bytes(os, B, H, Sq, D);
    const size_t lb = static_cast<size_t>(B) * H * Sq * 4;
    if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, kb) ||
        overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
        overlaps(lse, lb, o, ob))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    DenseArgs a{};
    a.seq_q = Sq;
    a.seq_k = Skv;
    a.hq = H;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.o = static_cast<__half*>(o);
    a.o_sb = os.b;
    a.o_sh = os.h;
    a.o_sr = os.r;
    a.lse = lse;
    a.status = dev.status;
    a.wait_limit = wait_limit_ns();
    a.fault = fault_mode();
    // 4-D maps (D, S, heads, batch) with the callers' strides; boxes past a head's
    // last row read zeros and never cross into another head
    CUtensorMap tq, tk, tv;
    if (encode_tmap_f16_4d(&tq, q, D, Sq, H, B, qs.r, qs.h, qs.b, 64, kBM) != GBATTN_OK ||
        encode_tmap_f16_4d(&tk, k, D, Skv, H, B, kvs.r, kvs.h, kvs.b, 64, 64) != GBATTN_OK ||
        encode_tmap_f16_4d(&tv, v, D, Skv, H, B, kvs.r, kvs.h, kvs.b, 64, 64) != GBATTN_OK)
        return GBATTN_ERR_CUDA;
    static std::once_flag once[64];
    static int attr_rc[64];
    if (dev.device < 0 || dev.device >= 64) return GBATTN_ERR_CUDA;
    std::call_once(once[dev.device], [&] {
        attr_rc[dev.device] = cudaFuncSetAttribute(attn_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemBytes) == cudaSuccess
                                  ? GBATTN_OK
                                  : GBATTN_ERR_CUDA;
    });
    if (attr_rc[dev.device] != GBATTN_OK) return attr_rc[dev.device];
    const dim3 grid((Sq + kBM - 1) / kBM, B * H);
    attn_dense_kernel<<<grid, kThreads, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(tq, tk, tv, a);
    count_launches(1);
    return launch_status();
}
