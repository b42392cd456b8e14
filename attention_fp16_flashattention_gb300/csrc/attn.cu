// Fused forward attention on sm_103a: O = softmax(scale * Q K^T + mask) V with
// FP16 Q/K/V/P/O, FP32 accumulation in tensor memory and an FP32 online softmax
// ("Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation: FP32
// QK/PV accumulation, FP32 prefix/tail state and final merge, FP16
// probabilities and output).  This file holds the causal (plain and paged
// E4M3), masked and VSA modes; dense attention has its own copy of the
// pipeline in attn_dense.cu.
//
// A work item is a 128-row query tile with a list of 128-key tiles.  Each key
// tile is two 64-key halves; for causal and masked attention the halves are
// adjacent, for VSA they are two selected 64-token cubes (the two-query-half x
// two-key-half blocks with a 4-bit quadrant mask of block_lists.py in the
// FastVideo compare view).  Causal and masked launches run one CTA per item;
// the VSA modes run persistent CTAs (one per SM) whose scheduler warp draws
// items from a counter and builds their tile lists one item ahead.
//
// Warp roles (320 threads at D=256, 384 with the mask warp or the VSA scheduler,
// 448 with the paged converters):
//   warp 0      TMA producer: each item's Q, then K and V tiles through an
//               NS-slot ring in the order the MMAs consume them (K0 .. K_{NSB-1},
//               V0, K_NSB, V1, ...); items follow each other in the ring.
//   warp 1      allocates tensor memory and issues S = Q K_t^T (SMEM x SMEM);
//               at D=128 only these, at D=256 also every PV, in order.
//   warp 10     (D=128) issues O += P_j V_j (P from TMEM), so that neither MMA
//               stream waits behind the other's barrier waits.  Each issuing
//               warp is converged and one elected lane issues each group.
//   warps 2..9  softmax: two threads per query row (TMEM lane = row), one per
//               64-key half of the tile; they exchange the partial row max;
//               exp2 with packed FP32 pairs, row sum, P -> FP16 into TMEM; lazy
//               O rescaling (only when the running max grows by more than 2^8),
//               each thread on its half of O; epilogue O / l.
//   warp 11     (masked) loads each tile's 128 x 128 mask block two tiles ahead;
//               (VSA) the scheduler.
//   warps 10..13 (paged causal) convert E4M3 page rows to FP16 in shared memory.
// Tensor memory (512 columns): NSB S buffers of 128 FP32 columns (3 for D=128,
// 2 for D=256); P_j overwrites the first 64 columns of its S buffer as FP16
// pairs; O [NSB*128, NSB*128 + D) FP32.  QK runs up to NSB tiles ahead; with
// two issuing warps QK_t waits for PV_{t-NSB} (which read P from its buffer).
//
// Every wait is bounded in time (see WaitCtl): a wait that runs out records
// GBATTN_DEV_WAIT_TIMEOUT in the device status word, the CTA stops, waits a
// bounded time for its copies and MMAs in flight, frees tensor memory and exits.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "e4m3.cuh"
#include "host.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int BM = 128;             // query rows per CTA
constexpr int BN = 128;             // keys per tile (two halves of 64)
constexpr int kSoftmaxThreads = 256;
constexpr int kMaxSparseTiles = 512;
constexpr int kMaxTopk = 512;
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s for draining after an abort
constexpr size_t kSparseWorkspaceBytes = 16;    // the item counter (int32), padded
constexpr uint64_t kItemWaitNs = 20000000000ull;   // 20 s: the scheduler's wait for a free item slot

// kMasked: dense with an additive FP16 mask [Sq][Skv] per (batch, head) slice.
// kSparseFull: kSparse with the full VSA layout (prefix queries, boundary cubes).
// kCausalPaged: kCausal reading K/V as E4M3 pages (converted in shared memory).
enum Mode { kDense = 0, kCausal = 1, kSparse = 2, kMasked = 3, kSparseFull = 4, kCausalPaged = 5 };
__host__ __device__ constexpr bool is_sparse(int mode) { return mode == kSparse || mode == kSparseFull; }
__host__ __device__ constexpr bool is_causal(int mode) { return mode == kCausal || mode == kCausalPaged; }
// The D=128 modes issue their MMAs from two warps: warp 1 the QK groups and
// warp 10 the PV groups, so that neither stream waits behind the other's
// barrier waits.  The D=256 causal modes keep one issuing warp: with only two
// S buffers in tensor memory, waiting for PV_j to finish before QK_{j+2}
// reuses its buffer would stall the softmax.
__host__ __device__ constexpr bool dual_issue(int mode) { return !(mode == kCausal || mode == kCausalPaged); }
constexpr int kPvWarp = 10;
// threads per CTA: the PV issuer adds a warp (10); the paged mode adds four
// converter warps (10..13), the masked mode a mask-loading warp (11), the VSA
// modes a scheduler warp (11)
// Persistent CTAs (one per SM, each running items until none is left) pay
// where items are short and uneven: the VSA modes.  The other modes launch one
// CTA per item; their item loop then runs once, with a compile-time bound.
__host__ __device__ constexpr bool persistent(int mode) { return is_sparse(mode); }
__host__ __device__ constexpr int threads_for(int mode) {
    return mode == kCausalPaged ? 448 : mode == kMasked ? 384 : is_sparse(mode) ? 384 : (dual_issue(mode) ? 352 : 320);
}
constexpr int kMaskWarp = 11;
constexpr int kConvThreads = 128;

struct AttnArgs {
    int seq_q;          // query rows per head
    int seq_k;          // keys per KV head
    int heads_q;        // B * Hq (rows of the grid)
    int hq;             // query heads per batch entry
    int hkv;            // KV heads per batch entry
    int group;          // Hq / Hkv
    int q_real;         // causal: real queries
    int kv_prefix;      // causal: KV - Q_real
    int n_chunks;       // causal: key-range chunks per query tile
    int n_cubes;        // sparse: S / 64
    int topk;           // sparse
    float scale_log2;   // scale * log2(e)
    float scale;        // masked: the softmax scale itself
    __half* o;
    long long o_sb, o_sh, o_sr;   // element strides of O between batch entries, heads, rows
    float* lse;         // optional natural-log LSE (dense [B*H][seq_q])
    float* part_o;      // causal, n_chunks > 1: [C][heads_q][seq_q][D] FP32, normalised
    float* part_lse;    // causal, n_chunks > 1: [C][heads_q][seq_q] log2-sum-exp2
    const int32_t* idx; // sparse: [heads][n_cubes][topk]
    int prefix;         // sparse: prefix tokens before the video cubes (multiple of BM)
    const int32_t* page_table;   // paged: [B][max_pages] logical -> physical page
    int num_phys, page_size, max_pages, page_box;   // paged: pool, rows per TMA box
    int scale_mode;     // paged: 0 folded power of two, 1 FP16-valued, 2 general
    float ks, vs;       // paged: dequantisation scales
    __half2 ks2, vs2;
    float out_mul;      // v_scale when folded (applied to O), else 1
    const int32_t* pairs;   // sparse: [heads][ceil(n_cubes/2)][2] query-cube pairs, or null
                            //         (cubes 2p, 2p+1); a second entry of -1 means none
    const int32_t* cube_valid;   // sparse: real tokens per cube, or null (all full)
    const float* coarse;         // sparse: coarse-branch output [heads][n_cubes][D] FP32, or null
    const __half* gate;          // sparse: gate [heads][seq_q][D] FP16 (with coarse)
    const __half* mask; // masked: additive mask, row stride seq_k
    long long mask_sb;  // masked: elements between batch slices (0 = shared)
    long long mask_sh;  // masked: elements between head slices (0 = shared)
    uint32_t* status;
    uint64_t wait_limit;
    int fault;          // test hook: 1 = the TMA warp never loads Q; 2 = it stops after 2*NS K/V items
    int n_items;        // work items of the launch (query tiles, x key chunks for causal)
    int items_x;        // items per head row of the item order (see decode_item)
    int* sched;         // item counter (zero between launches), or null: static split
    int nsm;            // host: SMs of the device
};

constexpr int kSmemMax = 232448;   // dynamic shared memory a CTA may opt into (227 KB)

struct Ctrl {
    uint64_t q_full[2];    // query buffer b loaded
    uint64_t q_empty[2];   // the last QK of the item that used query buffer b is done
    uint64_t full[5];
    uint64_t empty[5];
    uint64_t s_full[3];    // QK_g done (buffer g % NSB), g counting every tile of the CTA
    uint64_t p_full[3];    // P_g written (buffer g % NSB)
    uint64_t pv_done[3];   // PV_g done (barrier g % NSB).  QK_g is issued after
                           // PV_{g-NSB}, so once S_g is visible the previous phase
                           // of every barrier awaited below has completed.
    uint64_t item_full[2];    // the scheduler warp wrote item slot s
    uint64_t item_empty[2];   // every consumer warp is done with item slot s
    uint64_t o_free;          // the softmax warps have read O of their last item out of TMEM
    uint64_t drain;
    uint64_t drain_pv;     // the PV issuer's own drain after an abort
    uint64_t xchg[4];      // per row quarter: the two half-row threads exchange values
    uint64_t raw_full[2];  // paged: E4M3 bytes of a slot landed (converters may read)
    uint64_t conv_read[2]; // paged: every converter holds its bytes (the slot may be overwritten)
    uint32_t tmem_base;
    int abort;
};

// Values exchanged between the two threads that share a query row.
struct Exchange {
    float mx[2][2][128];   // [tile parity][column half][row] partial row max
    float l[2][128];       // [column half][row] partial row sum (epilogue)
};

constexpr int kCtrlReserve = 512;
constexpr int kCtrlBytes = kCtrlReserve + static_cast<int>(sizeof(Exchange));
static_assert(sizeof(Ctrl) <= kCtrlReserve, "control block");

// One work item: a 128-row query tile of one head (a VSA video item: a pair of
// 64-row query cubes) and, for causal attention, one key chunk.
struct Item {
    int valid;      // 0: no more work for this CTA
    int bh;         // query head (batch-major)
    int kv_bh;      // key/value head
    int q_row0;     // first query row (VSA: of the first cube)
    int tile0;      // first 128-key tile (dense and causal)
    int n_tiles;    // key tiles of the item
    int chunk;      // causal key chunk
    int rbase0;     // first token row of each 64-row query half (-1: no second cube)
    int rbase1;
};

// The key tiles of a VSA item as its consumers read them.
struct SparseSlot {
    int key0[kMaxSparseTiles];   // first key of each 64-key tile half
    int key1[kMaxSparseTiles];
    // What the softmax reads per tile, in one word: quadrant bits | real keys of
    // the first half << 8 | real keys of the second half << 16.
    uint32_t info[kMaxSparseTiles];
};

// The scheduler warp's working space while it builds a VSA tile list.
struct SparseScratch {
    int list_a[kMaxTopk];
    int list_b[kMaxTopk];
    uint32_t bits_a[32];            // the two cube sets (at most 1024 cubes)
    uint32_t bits_b[32];
    uint8_t mask_hi[kMaxSparseTiles];   // quadrant bits of each tile's second half
    uint8_t mask[kMaxSparseTiles];
    uint8_t kv0[kMaxSparseTiles];   // real keys in each 64-key half (boundary cubes)
    uint8_t kv1[kMaxSparseTiles];
};

// Masked mode: the mask warp stages each tile's 128 rows x 128 keys of the mask
// (two 64-key boxes of 16 KB, TMA, 128-byte swizzle) in two slots, two tiles
// ahead; the slots' full and empty barriers follow them.
constexpr int kMaskSlotBytes = 128 * 256;
constexpr int kMaskStageBytes = 2 * kMaskSlotBytes + 4 * 8;

template <int D, int MODE>
struct Cfg {
    // K/V ring slots (the masked mode gives one D=128 slot to its mask stages; the
    // VSA modes, whose key cubes are gathered from across the head and miss L2
    // more often, take a fifth in place of a second query buffer)
    static constexpr int NS = D == 128 ? (MODE == 3 ? 3 : is_sparse(MODE) ? 5 : 4) : 2;
    static constexpr int NSB = D == 128 ? 3 : 2;         // S buffers in TMEM (QK lookahead)
    static constexpr int CHUNK = 128 * 128;               // 128 rows x 64 FP16 columns
    static constexpr int HALF = 64 * 128;                 // 64 rows x 64 columns
    static constexpr int KCH = D / 64;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int SLOT_BYTES = BN * D * 2;
    // everything but the query buffers
    static constexpr int REST = 1024 + NS * SLOT_BYTES + kCtrlBytes + 2 * static_cast<int>(sizeof(Item)) +
                                (is_sparse(MODE) ? static_cast<int>(2 * sizeof(SparseSlot) + sizeof(SparseScratch)) : 0) +
                                (MODE == kMasked ? kMaskStageBytes : 0);
    // Two query buffers where they fit: the next item's query tile then loads
    // while the last QKs of the current item still read theirs.
    static constexpr int QB = persistent(MODE) && !is_sparse(MODE) && REST + 2 * Q_BYTES <= kSmemMax ? 2 : 1;
    static constexpr int SMEM = REST + QB * Q_BYTES;
    static_assert(SMEM <= kSmemMax, "shared memory budget");
    // TMEM columns: S buffer b at b*128 (P of that tile overwrites its first 64
    // columns as FP16 pairs), O after the S buffers.
    static constexpr uint32_t T_O = NSB * 128;
    static_assert(T_O + D <= 512, "tensor memory budget");
    static constexpr uint32_t IDESC_QK = idesc_f16(BM, BN, false, false);
    static constexpr uint32_t IDESC_PV = idesc_f16(BM, D, false, true);
};

template <int D, int MODE>
constexpr int smem_bytes() {
    return Cfg<D, MODE>::SMEM;
}

// Consumer warps of an item slot: TMA, QK issuer, PV issuer (D=128), eight
// softmax warps, and the mask warp or the four converter warps.
__host__ __device__ constexpr int consumer_warps(int mode) {
    return 2 + (dual_issue(mode) ? 1 : 0) + kSoftmaxThreads / 32 + (mode == kMasked ? 1 : 0) +
           (mode == kCausalPaged ? kConvThreads / 32 : 0);
}

// Bounded wait that ignores the abort flag (used only to drain after an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainNs) return;
    }
}

// Item order of the K/V ring = the MMA warp's consumption order with a QK
// lookahead of L tiles: K_0 .. K_{L-1}, then (V_j, K_{j+L}) while j + L < n,
// then the remaining V_j.  Items follow each other in the ring.
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

// Position in a ring of N buffers, advanced one step at a time: idx = count % N,
// phase = (count / N) & 1, without a division in the loops.
template <int N>
struct Cursor {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void step() {
        if (++idx == N) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// Ring slot and phase of ring position pos (unsigned: a power-of-two ring is a mask).
template <int N>
__device__ __forceinline__ int slot_of(int pos) { return static_cast<int>(static_cast<unsigned>(pos) % N); }
template <int N>
__device__ __forceinline__ uint32_t phase_of(int pos) { return (static_cast<unsigned>(pos) / N) & 1u; }

// Real tokens of video cube c (boundary cubes are padded); out-of-range counts
// are flagged and clamped.
__device__ __forceinline__ int cube_count(const AttnArgs& a, int c) {
    if (!a.cube_valid) return 64;
    const int n = a.cube_valid[c];
    if (n < 1 || n > 64) {
        atomicOr(a.status, kDevBadIndex);
        return n < 1 ? 1 : 64;
    }
    return n;
}

// Tile list of a VSA item, built by the scheduler warp.  Prefix query tiles
// (qtile < prefix / BM) attend densely: every 128-key prefix tile, then the
// video cubes two by two.  Video query-cube pairs merge their two strictly
// ascending cube lists into tiles of two cubes; entries that are out of range
// or not ascending are skipped and flagged.  Video keys sit at prefix + 64 *
// cube.  Returns the number of tiles (warp-uniform).
template <bool kFull>
__device__ int build_sparse_tiles(SparseScratch* sc, SparseSlot* sl, const AttnArgs& a, int bh,
                                  int qtile, int ca, int cb) {
    const int lane = threadIdx.x & 31;
    const int n_pre = kFull ? a.prefix / BM : 0;
    const int kbase = kFull ? a.prefix : 0;
    if (kFull && qtile < n_pre) {
        const int nt = n_pre + (a.n_cubes + 1) / 2;
        for (int t = lane; t < nt; t += 32) {
            if (t < n_pre) {
                sl->key0[t] = t * BN;
                sl->key1[t] = t * BN + 64;
                sc->kv0[t] = sc->kv1[t] = 64;
                sc->mask[t] = 0xF;
            } else {
                const int c0 = 2 * (t - n_pre), c1 = c0 + 1;
                sl->key0[t] = a.prefix + 64 * c0;
                sc->kv0[t] = static_cast<uint8_t>(cube_count(a, c0));
                if (c1 < a.n_cubes) {
                    sl->key1[t] = a.prefix + 64 * c1;
                    sc->kv1[t] = static_cast<uint8_t>(cube_count(a, c1));
                    sc->mask[t] = 0xF;
                } else {   // odd cube count: the second half repeats the cube, masked
                    sl->key1[t] = sl->key0[t];
                    sc->kv1[t] = sc->kv0[t];
                    sc->mask[t] = 0x5;
                }
            }
        }
        return nt;
    }
    const int na = a.topk;
    const int nb = cb >= 0 ? a.topk : 0;
    const int32_t* la = a.idx + (static_cast<long long>(bh) * a.n_cubes + ca) * a.topk;
    const int32_t* lb = a.idx + (static_cast<long long>(bh) * a.n_cubes + (cb >= 0 ? cb : ca)) * a.topk;
    for (int i = lane; i < na; i += 32) sc->list_a[i] = la[i];
    for (int i = lane; i < nb; i += 32) sc->list_b[i] = lb[i];
    sc->bits_a[lane] = 0u;
    sc->bits_b[lane] = 0u;
    __syncwarp();
    // Set of each list: an entry counts when it lies in range and exceeds every
    // entry before it (a list that is not strictly ascending is flagged and its
    // offending entries skipped).
    bool bad = false;
    for (int lst = 0; lst < 2; ++lst) {
        const int n = lst == 0 ? na : nb;
        const int* L = lst == 0 ? sc->list_a : sc->list_b;
        uint32_t* bits = lst == 0 ? sc->bits_a : sc->bits_b;
        int run_max = -1;
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            const int v = i < n ? L[i] : -1;
            int pre = (v >= 0 && v < a.n_cubes) ? v : -1;   // inclusive prefix max (in range)
#pragma unroll
            for (int sh = 1; sh < 32; sh <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, pre, sh);
                if (lane >= sh) pre = max(pre, y);
            }
            int before = __shfl_up_sync(0xffffffffu, pre, 1);
            if (lane == 0) before = -1;
            before = max(before, run_max);
            if (i < n) {
                if (v > before && v < a.n_cubes) atomicOr(&bits[v >> 5], 1u << (v & 31));
                else bad = true;
            }
            run_max = max(run_max, __shfl_sync(0xffffffffu, pre, 31));
        }
    }
    __syncwarp();
    // Union in ascending cube order: word w of the sets belongs to lane w; a warp
    // prefix sum of the popcounts places every cube; consecutive cubes pair up
    // into 128-key tiles.
    const uint32_t ua = sc->bits_a[lane], ub = sc->bits_b[lane], uu = ua | ub;
    const int cnt = __popc(uu);
    int incl = cnt;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, sh);
        if (lane >= sh) incl += y;
    }
    const int nu = __shfl_sync(0xffffffffu, incl, 31);
    int pos = incl - cnt;
    for (uint32_t rest = uu; rest; rest &= rest - 1, ++pos) {
        const int bit = __ffs(rest) - 1;
        const int c = lane * 32 + bit;
        const uint32_t f = ((ua >> bit) & 1u) | (((ub >> bit) & 1u) << 1);
        const int t = pos >> 1;
        if ((pos & 1) == 0) {
            sl->key0[t] = kbase + c * 64;
            sc->mask[t] = static_cast<uint8_t>((f & 1) | ((f >> 1) << 2));
            if (pos == nu - 1) {   // odd union: the second half repeats the cube, fully masked
                sl->key1[t] = kbase + c * 64;
                sc->mask_hi[t] = 0;
            }
        } else {
            sl->key1[t] = kbase + c * 64;
            sc->mask_hi[t] = static_cast<uint8_t>(((f & 1) << 1) | ((f >> 1) << 3));
        }
    }
    __syncwarp();
    const int nt = (nu + 1) / 2;
    for (int t = lane; t < nt; t += 32) sc->mask[t] |= sc->mask_hi[t];
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, kDevBadIndex);
    return nt;
}

// The next item of a CTA (lane 0 draws, the warp gets it).  With a counter the
// items go to whichever CTA asks first; every CTA draws once past the last
// item, and the draw that sees the last of those values (n_items + grid - 1:
// no CTA draws after it) puts the counter back to zero for the next launch.
// A draw outside [0, n_items + grid) means the counter did not start at zero:
// it is flagged and ends the CTA's work.  Without a counter, CTA c takes items
// c, c + grid, c + 2 grid, ...
__device__ __forceinline__ long long next_item(const AttnArgs& a, int k) {
    long long id = 0;
    if (a.sched) {
        if ((threadIdx.x & 31) == 0) {
            const int last = a.n_items + static_cast<int>(gridDim.x) - 1;
            const int v = atomicAdd(a.sched, 1);
            if (v == last) atomicExch(a.sched, 0);
            if (v < 0 || v > last) atomicOr(a.status, kDevBadIndex);
            id = (v < 0 || v > last) ? a.n_items : v;
        }
        id = __shfl_sync(0xffffffffu, id, 0);
    } else {
        id = static_cast<long long>(blockIdx.x) + static_cast<long long>(k) * gridDim.x;
    }
    return id;
}

// Work decode of item id (everything but the VSA tile list).  The item order
// is the order the CTAs of a one-item-per-CTA launch would start in.
template <int MODE>
__device__ Item decode_item(const AttnArgs& a, int id, int& qtile) {
    Item it{};
    it.valid = 1;
    int bh;
    if (MODE == kMasked) {
        // heads fastest, so that the items of all heads of a query tile run
        // together and share that tile's mask rows in L2
        bh = id % a.heads_q;
        qtile = id / a.heads_q;
    } else if (MODE == kSparseFull) {
        // the long prefix tiles of every head first, then each head's cube pairs
        const int n_pre = a.prefix / BM;
        const int n_pairs = a.items_x - n_pre;
        const int pre_all = n_pre * a.heads_q;
        if (id < pre_all) {
            bh = id / n_pre;
            qtile = id - bh * n_pre;
        } else {
            const int r = id - pre_all;
            bh = r / n_pairs;
            qtile = n_pre + (r - bh * n_pairs);
        }
    } else if (is_causal(MODE)) {
        // heads fastest, then query tiles, then key chunks, so that the items in
        // flight walk one key window together (and the query heads that share a
        // KV head read each K/V tile from L2 at about the same time)
        const int n_qt = a.items_x / a.n_chunks;
        bh = id % a.heads_q;
        const int r = id / a.heads_q;
        qtile = r % n_qt;
        it.chunk = r / n_qt;
    } else {
        qtile = id % a.items_x;
        bh = id / a.items_x;
    }
    it.bh = bh;
    it.q_row0 = qtile * BM;
    it.kv_bh = bh;
    if (is_causal(MODE)) {
        const int b = bh / a.hq, h = bh - b * a.hq;
        it.kv_bh = b * a.hkv + h / a.group;
        const long long kend = min(static_cast<long long>(a.seq_k),
                                   static_cast<long long>(a.kv_prefix) + it.q_row0 + BM);
        const int T = static_cast<int>((kend + BN - 1) / BN);
        it.tile0 = static_cast<int>(static_cast<long long>(it.chunk) * T / a.n_chunks);
        it.n_tiles = static_cast<int>(static_cast<long long>(it.chunk + 1) * T / a.n_chunks) - it.tile0;
    } else if (MODE == kDense || MODE == kMasked) {
        it.n_tiles = (a.seq_k + BN - 1) / BN;
    }
    it.rbase0 = it.q_row0;
    it.rbase1 = it.q_row0 + 64;
    return it;
}

// PS (causal modes only): the probabilities enter the PV product as two FP16
// halves, hi = RNE(p) and lo = RNE(p - hi), about 22 bits of p, instead of one
// FP16 value.  P_lo takes columns 64..127 of its S buffer (both threads of a
// row have read their S halves before either writes), and PV issues a second
// group of MMAs over it.
//
// Items: every role loops over the CTA's items until it gets an invalid one
// (persistent VSA modes; the other modes run one item per CTA and their loop
// has a compile-time bound of one).  Every role keeps running counts (tiles,
// ring items, query buffer uses) across items, so each barrier's phases simply
// continue; the first PV of an item overwrites O once the softmax warps have
// read the previous item's O (o_free).
template <int D, int MODE, bool PS = false>
__global__ void __launch_bounds__(threads_for(MODE), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmM,
                    const AttnArgs a) {
    using C = Cfg<D, MODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                              // C::QB query buffers
    uint8_t* sKV = smem + C::QB * C::Q_BYTES;
    // masked mode: mask stages (1024-aligned) and their barriers after the ring
    uint8_t* sMask = sKV + C::NS * C::SLOT_BYTES;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sMask + 2 * kMaskSlotBytes);   // full[2], empty[2]
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(sKV + C::NS * C::SLOT_BYTES +
                                         (MODE == kMasked ? kMaskStageBytes : 0));
    Exchange* ex = reinterpret_cast<Exchange*>(reinterpret_cast<uint8_t*>(ctrl) + kCtrlReserve);
    Item* items = reinterpret_cast<Item*>(reinterpret_cast<uint8_t*>(ctrl) + kCtrlBytes);
    SparseSlot* slots = reinterpret_cast<SparseSlot*>(items + 2);
    SparseScratch* scratch = reinterpret_cast<SparseScratch*>(slots + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // VSA items differ in length and need their tile lists built: a scheduler warp
    // draws them and fills two item slots ahead of the consumers.  Every other
    // item is a uniform query tile (and key chunk) that each warp decodes itself.
    constexpr bool kSched = is_sparse(MODE);
    constexpr bool kPersist = persistent(MODE);
    constexpr int kSchedWarp = kSched ? threads_for(MODE) / 32 - 1 : -1;

    // ---- prologue
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::QB; ++i) {
            mbar_init(&ctrl->q_full[i], 1);
            mbar_init(&ctrl->q_empty[i], 1);
        }
        for (int i = 0; i < C::NS; ++i) {
            // paged: the four converter warps complete a slot, not the TMA bytes
            mbar_init(&ctrl->full[i], MODE == kCausalPaged ? kConvThreads / 32 : 1);
            mbar_init(&ctrl->empty[i], 1);
        }
        if (MODE == kCausalPaged)
            for (int i = 0; i < 2; ++i) {
                mbar_init(&ctrl->raw_full[i], 1);
                mbar_init(&ctrl->conv_read[i], kConvThreads / 32);
            }
        for (int i = 0; i < C::NSB; ++i) {
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->p_full[i], kSoftmaxThreads);
            mbar_init(&ctrl->pv_done[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&ctrl->xchg[i], 64);
        if (MODE == kMasked)
            for (int i = 0; i < 2; ++i) {
                mbar_init(&mbar[i], 1);                          // the slot's bytes landed
                mbar_init(&mbar[2 + i], kSoftmaxThreads / 32);   // every softmax warp read it
            }
        if (kSched)
            for (int i = 0; i < 2; ++i) {
                mbar_init(&ctrl->item_full[i], 1);
                mbar_init(&ctrl->item_empty[i], consumer_warps(MODE));
            }
        mbar_init(&ctrl->o_free, kSoftmaxThreads / 32);
        mbar_init(&ctrl->drain, 1);
        mbar_init(&ctrl->drain_pv, 1);
        ctrl->abort = 0;
        mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (MODE == kMasked || is_sparse(MODE)) tma_prefetch_desc(&tmM);
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
    const bool load_q = a.fault != 1;

    // The CTA's k-th item.  VSA: from item slot k & 1 (false: the wait ended in
    // an abort); otherwise item blockIdx.x + k * gridDim.x, decoded here.
    auto get_item = [&](int k, Item& cur) -> bool {
        if (kSched) {
            if (!wait_warp(&ctrl->item_full[k & 1], (k >> 1) & 1, w)) return false;
            cur = items[k & 1];
        } else {
            const long long id = static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x +
                                 static_cast<long long>(k) * gridDim.x * gridDim.y;
            int qtile = 0;
            if (id < a.n_items) cur = decode_item<MODE>(a, static_cast<int>(id), qtile);
            else cur.valid = 0;
        }
        return true;
    };
    auto item_release = [&](int k) {
        if (kSched) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->item_empty[k & 1]);
        }
    };
    auto tile_keys = [&](const Item& it, const SparseSlot* sl, int t, int& k0, int& k1) {
        if (is_sparse(MODE)) {
            k0 = sl->key0[t];
            k1 = sl->key1[t];
        } else {
            k0 = (it.tile0 + t) * BN;
            k1 = k0 + 64;
        }
    };
    // S_g = Q K^T into S buffer buf; O += P V with P read from S buffer buf.
    auto issue_qk = [&](int qbuf, int slot, int buf) {
        const uint32_t qa = smem_addr(sQ + qbuf * C::Q_BYTES);
        const uint32_t ka = smem_addr(sKV + slot * C::SLOT_BYTES);
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16) {
            const uint32_t off = (k16 >> 2) * C::CHUNK + (k16 & 3) * 32;
            mma_ss(tmem + buf * 128, sdesc_sw128(qa + off, 16, 1024),
                   sdesc_sw128(ka + off, 16, 1024), C::IDESC_QK, k16 > 0 ? 1u : 0u);
        }
    };
    auto issue_pv = [&](int slot, int buf, bool acc) {
        const uint32_t va = smem_addr(sKV + slot * C::SLOT_BYTES);
#pragma unroll
        for (int k16 = 0; k16 < BN / 16; ++k16)
            mma_ts(tmem + C::T_O, tmem + buf * 128 + k16 * 8,
                   sdesc_sw128(va + k16 * 2048, C::CHUNK, 1024), C::IDESC_PV,
                   (acc || k16 > 0) ? 1u : 0u);
        if (PS) {   // O += P_lo V (columns 64.. of the buffer)
#pragma unroll
            for (int k16 = 0; k16 < BN / 16; ++k16)
                mma_ts(tmem + C::T_O, tmem + buf * 128 + 64 + k16 * 8,
                       sdesc_sw128(va + k16 * 2048, C::CHUNK, 1024), C::IDESC_PV, 1u);
        }
    };
    // Ring positions within an item of n tiles (the TMA warp's load order, see
    // ring_item) of K_t and V_j.
    auto pos_k = [&](int t) { return t < C::NSB ? t : C::NSB + 2 * (t - C::NSB) + 1; };
    auto pos_v = [&](int j, int n) { return min(n, C::NSB) + j + min(j, max(0, n - C::NSB)); };

    if (kSched && warp == kSchedWarp) {
        // ================= scheduler: draws items, decodes them (and builds the
        // VSA tile lists) into the two item slots, one item ahead of the consumers
        // (a slot frees when a whole item has run, so this wait has a long limit
        // and sleeps between polls; an abort elsewhere still ends it)
        const WaitCtl w_item{a.wait_limit > kItemWaitNs ? a.wait_limit : kItemWaitNs, a.status, &ctrl->abort};
        bool ok = true, drawn_last = false;
        for (int k = 0;; ++k) {
            const long long id = next_item(a, k);
            const bool live = id < a.n_items;
            drawn_last = !live;
            if (k >= 2) ok = wait_warp_sleep(&ctrl->item_empty[k & 1], ((k >> 1) - 1) & 1, w_item, 1000);
            if (!ok) break;
            Item* dst = items + (k & 1);
            if (live) {
                int qtile = 0;
                Item it = decode_item<MODE>(a, static_cast<int>(id), qtile);
                if (is_sparse(MODE)) {
                    SparseSlot* sl = slots + (k & 1);
                    const int n_pre = MODE == kSparseFull ? a.prefix / BM : 0;
                    int ca = -1, cb = -1;
                    if (qtile >= n_pre) {   // a pair of query cubes (ca, cb), not necessarily adjacent
                        const int p = qtile - n_pre;
                        ca = 2 * p;
                        cb = 2 * p + 1 < a.n_cubes ? 2 * p + 1 : -1;
                        if (a.pairs) {
                            const int n_pairs = (a.n_cubes + 1) / 2;
                            const int x = a.pairs[(static_cast<long long>(it.bh) * n_pairs + p) * 2];
                            const int y = a.pairs[(static_cast<long long>(it.bh) * n_pairs + p) * 2 + 1];
                            if (x >= 0 && x < a.n_cubes && y >= -1 && y < a.n_cubes && x != y) {
                                ca = x;
                                cb = y;
                            } else if (lane == 0) {
                                atomicOr(a.status, kDevBadIndex);
                            }
                        }
                        const int kb = MODE == kSparseFull ? a.prefix : 0;
                        it.rbase0 = kb + 64 * ca;
                        it.rbase1 = cb >= 0 ? kb + 64 * cb : -1;
                        it.q_row0 = it.rbase0;
                    }
                    const int nt = build_sparse_tiles<MODE == kSparseFull>(scratch, sl, a, it.bh, qtile, ca, cb);
                    __syncwarp();
                    const bool counts = MODE == kSparseFull && a.cube_valid;
                    if (counts && qtile >= n_pre)   // real keys of every tile half (boundary cubes)
                        for (int t = lane; t < nt; t += 32) {
                            scratch->kv0[t] = static_cast<uint8_t>(cube_count(a, (sl->key0[t] - a.prefix) >> 6));
                            scratch->kv1[t] = static_cast<uint8_t>(cube_count(a, (sl->key1[t] - a.prefix) >> 6));
                        }
                    __syncwarp();
                    for (int t = lane; t < nt; t += 32)
                        sl->info[t] = scratch->mask[t] |
                                      (static_cast<uint32_t>(counts ? scratch->kv0[t] : 64) << 8) |
                                      (static_cast<uint32_t>(counts ? scratch->kv1[t] : 64) << 16);
                    it.n_tiles = nt;
                }
                if (lane == 0) *dst = it;
            } else if (lane == 0) {
                dst->valid = 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->item_full[k & 1]);
            if (!live) break;
        }
        // after an abort: draw on to this CTA's last draw (the counter resets itself)
        if (a.sched)
            while (!drawn_last) drawn_last = next_item(a, 0) >= a.n_items;
    } else if (warp == 0) {
        // ================= TMA producer (whole warp; one elected lane issues)
        int last_it[C::NS];                  // last ring position issued into each slot
#pragma unroll
        for (int s = 0; s < C::NS; ++s) last_it[s] = -1;
        int last_q[2] = {-1, -1};            // last use issued into each query buffer
        int ring = 0, qu = 0;
        bool ok = true;
        // paged: lane j holds the cache row of box j (page_box tokens) of the
        // item after the one being issued; boxes cover the item's 128 keys.
        const int n_box = MODE == kCausalPaged ? BN / a.page_box : 0;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            if (!cur.valid) break;
            const SparseSlot* sl = slots + (k & 1);
            const int n = cur.n_tiles;
            const int qb = cur.bh / a.hq, qh = cur.bh - qb * a.hq;
            const int kvb = cur.kv_bh / a.hkv, kvh = cur.kv_bh - kvb * a.hkv;
            if (n > 0) {
                const int qbuf = qu % C::QB;
                if (qu >= C::QB) ok = wait_warp(&ctrl->q_empty[qbuf], ((qu / C::QB) - 1) & 1, w);
                if (!ok) break;
                if (load_q) {
                    uint8_t* dq = sQ + qbuf * C::Q_BYTES;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&ctrl->q_full[qbuf], C::Q_BYTES);
                        if (is_sparse(MODE)) {   // two 64-row halves; tmM has 64-row boxes
                            const int r1 = cur.rbase1 >= 0 ? cur.rbase1 : cur.rbase0;
#pragma unroll
                            for (int c = 0; c < C::KCH; ++c) {
                                tma_load_4d(dq + c * C::CHUNK, &tmM, &ctrl->q_full[qbuf], c * 64, cur.rbase0, qh, qb);
                                tma_load_4d(dq + c * C::CHUNK + C::HALF, &tmM, &ctrl->q_full[qbuf], c * 64, r1, qh, qb);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < C::KCH; ++c)
                                tma_load_4d(dq + c * C::CHUNK, &tmQ, &ctrl->q_full[qbuf], c * 64, cur.q_row0, qh, qb);
                        }
                    }
                    __syncwarp();
                    last_q[qbuf] = qu;
                }
                ++qu;
                auto page_row = [&](int item) -> int {
                    if (MODE != kCausalPaged || lane >= n_box || item >= 2 * n) return 0;
                    int t, k0, k1;
                    bool iv;
                    ring_item(item, n, C::NSB, t, iv);
                    tile_keys(cur, sl, t, k0, k1);
                    const int tok = k0 + lane * a.page_box;
                    const int b = cur.kv_bh / a.hkv;
                    int page = tok < a.seq_k ? a.page_table[static_cast<long long>(b) * a.max_pages +
                                                            tok / a.page_size]
                                             : 0;
                    if (page < 0 || page >= a.num_phys) {
                        atomicOr(a.status, kDevBadPage);
                        page = 0;
                    }
                    return page * a.page_size + tok % a.page_size;
                };
                int prow_next = page_row(0);
                for (int it = 0; it < 2 * n; ++it) {
                    const int gi = ring + it;
                    if (a.fault == 2 && gi >= 2 * C::NS) {   // test hook: stop mid-stream, drain, leave
                        ok = false;
                        break;
                    }
                    const int slot = slot_of<C::NS>(gi);
                    const int prow_cur = prow_next;
                    if (MODE == kCausalPaged) prow_next = page_row(it + 1);
                    if (!wait_warp(&ctrl->empty[slot], phase_of<C::NS>(gi) ^ 1u, w)) { ok = false; break; }
                    int t;
                    bool is_v;
                    ring_item(it, n, C::NSB, t, is_v);
                    int k0, k1;
                    tile_keys(cur, sl, t, k0, k1);
                    const CUtensorMap* m = is_v ? &tmV : &tmK;
                    uint8_t* dst = sKV + slot * C::SLOT_BYTES;
                    if (MODE == kCausalPaged) {
                        // E4M3 rows of the ring item (128 keys x D bytes) into the slot's upper
                        // half, laid out [key half][column half][64 rows][128 bytes], 128-byte swizzle.
                        uint8_t* stage = dst + C::SLOT_BYTES / 2;
                        const int hk = cur.kv_bh % a.hkv;
                        const int rows_per_box = a.page_box;
                        int rows[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) rows[j] = __shfl_sync(0xffffffffu, prow_cur, j);
                        if (elect_one()) {
                            mbar_arrive_expect_tx(&ctrl->raw_full[slot], BN * D);
                            for (int j = 0; j < n_box; ++j) {
                                const int key = j * rows_per_box;   // 0..127 within the ring item
                                const int kh = key >> 6, r = key & 63;
#pragma unroll
                                for (int ch = 0; ch < D / 128; ++ch)
                                    tma_load_3d(stage + (kh * (D / 128) + ch) * 8192 + r * 128, m,
                                                &ctrl->raw_full[slot], 128 * ch, hk, rows[j]);
                            }
                        }
                        __syncwarp();
                        last_it[slot] = gi;
                        continue;
                    }
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&ctrl->full[slot], C::SLOT_BYTES);
#pragma unroll
                        for (int c = 0; c < C::KCH; ++c) {
                            tma_load_4d(dst + c * C::CHUNK, m, &ctrl->full[slot], c * 64, k0, kvh, kvb);
                            tma_load_4d(dst + c * C::CHUNK + C::HALF, m, &ctrl->full[slot], c * 64, k1,
                                        kvh, kvb);
                        }
                    }
                    __syncwarp();
                    last_it[slot] = gi;
                }
                ring += 2 * n;
            }
            if (!ok) break;
            item_release(k);
        }
        if (!ok && lane == 0) {   // let copies in flight land before the CTA exits
            for (int b = 0; b < C::QB; ++b)
                if (last_q[b] >= 0) drain_wait(&ctrl->q_full[b], (last_q[b] / C::QB) & 1);
            for (int s = 0; s < C::NS; ++s)
                if (last_it[s] >= 0)
                    drain_wait(MODE == kCausalPaged ? &ctrl->raw_full[s] : &ctrl->full[s],
                               phase_of<C::NS>(last_it[s]));
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (whole warp waits; one elected lane issues
        // each group of MMAs and its commits)
        int tb = 0, qu = 0, o_uses = 0;
        Cursor<C::NSB> sb;   // S buffer and phase of tile tb + t (QK order = PV order)
        bool ok = true;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            const int valid = cur.valid, n = cur.n_tiles;
            item_release(k);
            if (!valid) break;
            if (n == 0) continue;
            const int qbuf = qu % C::QB;
            ok = wait_warp(&ctrl->q_full[qbuf], (qu / C::QB) & 1, w);
            ++qu;
            if (!ok) break;
            if (dual_issue(MODE)) {
                // QK only (warp 10 issues PV).  QK_g overwrites the S buffer that
                // PV_{g-NSB} read P_{g-NSB} from, so it waits for that PV to finish.
                // A parity wait on a slot is unambiguous only if the slot's previous
                // ring item is known to have landed: here it is either an earlier K
                // (this warp waited for it) or a V_i that precedes K_g in the ring,
                // so i <= g-NSB (within an item K_t follows V_{t-NSB}; the first
                // NSB K of an item follow every V of the items before) and PV_i
                // finished with PV_{g-NSB}.
                for (int t = 0; t < n; ++t) {
                    const int g = tb + t;
                    const int pos = 2 * tb + pos_k(t);
                    const int slot = slot_of<C::NS>(pos);
                    const int buf = sb.idx;
                    // PV_{g-NSB}: same buffer, previous phase
                    if (g >= C::NSB) ok = wait_warp(&ctrl->pv_done[buf], sb.phase ^ 1u, w);
                    ok = ok && wait_warp(&ctrl->full[slot], phase_of<C::NS>(pos), w);
                    sb.step();
                    if (!ok) break;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_qk(qbuf, slot, buf);
                        mma_commit(&ctrl->s_full[buf]);
                        mma_commit(&ctrl->empty[slot]);
                        if (t == n - 1) mma_commit(&ctrl->q_empty[qbuf]);
                    }
                    __syncwarp();
                }
            } else {
                int it = 2 * tb;
                // S_0 .. S_{L-1} of the item up front (into buffers whose previous
                // PV this thread issued earlier: in order on the tensor pipe), then
                // per tile: PV_j, and QK_{j+L} into the buffer P_j has just been
                // read from.
                for (int t = 0; ok && t < min(n, C::NSB); ++t) {
                    const int slot = slot_of<C::NS>(it);
                    ok = wait_warp(&ctrl->full[slot], phase_of<C::NS>(it), w);
                    if (!ok) break;
                    const int buf = (sb.idx + t) % C::NSB;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_qk(qbuf, slot, buf);
                        mma_commit(&ctrl->s_full[buf]);
                        mma_commit(&ctrl->empty[slot]);
                        if (t == n - 1) mma_commit(&ctrl->q_empty[qbuf]);
                    }
                    __syncwarp();
                    ++it;
                }
                for (int j = 0; ok && j < n; ++j) {
                    const int buf = sb.idx;
                    const int vslot = slot_of<C::NS>(it);
                    ok = wait_warp(&ctrl->p_full[buf], sb.phase, w) &&
                         wait_warp(&ctrl->full[vslot], phase_of<C::NS>(it), w);
                    sb.step();
                    // the item's first PV overwrites O: the previous item's O must be read
                    if (ok && j == 0 && o_uses > 0) ok = wait_warp(&ctrl->o_free, (o_uses - 1) & 1, w);
                    if (!ok) break;
                    ++it;
                    tc_fence_after();
                    if (elect_one()) {
                        issue_pv(vslot, buf, j > 0);
                        mma_commit(&ctrl->empty[vslot]);
                        mma_commit(&ctrl->pv_done[buf]);
                    }
                    __syncwarp();
                    if (j + C::NSB < n) {
                        const int kslot = slot_of<C::NS>(it);
                        ok = wait_warp(&ctrl->full[kslot], phase_of<C::NS>(it), w);
                        if (!ok) break;
                        ++it;
                        tc_fence_after();
                        if (elect_one()) {
                            issue_qk(qbuf, kslot, buf);
                            mma_commit(&ctrl->s_full[buf]);
                            mma_commit(&ctrl->empty[kslot]);
                            if (j + C::NSB == n - 1) mma_commit(&ctrl->q_empty[qbuf]);
                        }
                        __syncwarp();
                    }
                }
                ++o_uses;
            }
            tb += n;
        }
        if (!ok) {   // wait for issued MMAs before tensor memory is freed
            if (elect_one()) mma_commit(&ctrl->drain);
            __syncwarp();
            if (lane == 0) drain_wait(&ctrl->drain, 0);
        }
    } else if (dual_issue(MODE) && warp == kPvWarp) {
        // ================= PV issuer (D=128 modes; whole warp waits, one elected
        // lane issues).  PV_g waits for P_g (the softmax is done with S_g, so
        // every QK up to g has finished) and for V_g in the ring.  A parity wait
        // on a slot is unambiguous only if the slot's previous ring item is known
        // to have landed: an earlier V (this warp waited for it), a K_t with
        // t <= g, or a K of an earlier item is; a K_t of the same item with t > j
        // (a 3-slot ring: t = j+1) is first awaited through its QK.  That QK wait
        // is itself unambiguous: K_t precedes V_j in the ring, so t <= j+NSB-1
        // and QK_{t-NSB} finished before S_j was read.
        int tb = 0, o_uses = 0;
        Cursor<C::NSB> sb;   // S buffer and phase of tile tb + j
        bool ok = true;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            const int valid = cur.valid, n = cur.n_tiles;
            item_release(k);
            if (!valid) break;
            if (n == 0) continue;
            // the item's first PV overwrites O: the previous item's O must be read
            if (o_uses > 0) ok = wait_warp(&ctrl->o_free, (o_uses - 1) & 1, w);
            ++o_uses;
            for (int j = 0; ok && j < n; ++j) {
                const int rpos = pos_v(j, n);
                const int pos = 2 * tb + rpos;
                const int slot = slot_of<C::NS>(pos);
                const int buf = sb.idx;
                ok = wait_warp(&ctrl->p_full[buf], sb.phase, w);
                sb.step();
                if (ok && rpos >= C::NS) {
                    int pt;
                    bool pv;
                    ring_item(rpos - C::NS, n, C::NSB, pt, pv);
                    if (!pv && pt > j)
                        ok = wait_warp(&ctrl->s_full[(tb + pt) % C::NSB], ((tb + pt) / C::NSB) & 1, w);
                }
                ok = ok && wait_warp(&ctrl->full[slot], phase_of<C::NS>(pos), w);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    issue_pv(slot, buf, j > 0);
                    mma_commit(&ctrl->empty[slot]);
                    mma_commit(&ctrl->pv_done[buf]);
                }
                __syncwarp();
            }
            tb += n;
        }
        if (!ok) {   // wait for issued MMAs before tensor memory is freed
            if (elect_one()) mma_commit(&ctrl->drain_pv);
            __syncwarp();
            if (lane == 0) drain_wait(&ctrl->drain_pv, 0);
        }
    } else if (MODE == kCausalPaged && warp >= 10) {
        // ================= E4M3 -> FP16 converters (warps 10..13, paged mode)
        // Thread ct owns key row ct of every ring item: it reads the row's D E4M3
        // bytes from the slot's upper half into registers, waits for the other
        // converters (the FP16 tile overwrites that half), then writes the FP16
        // row into the 128-byte-swizzled K-major layout TMA would have produced.
        const int ct = threadIdx.x - 320;
        const int kh = ct >> 6, rr = ct & 63;
        bool ok = true;
        int ring = 0;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            if (!cur.valid) break;
            const int n = cur.n_tiles;
            for (int it = 0; it < 2 * n; ++it) {
                const int gi = ring + it;
                const int slot = slot_of<C::NS>(gi);
                ok = wait_warp(&ctrl->raw_full[slot], phase_of<C::NS>(gi), w);
                if (!ok) break;
                int t;
                bool is_v;
                ring_item(it, n, C::NSB, t, is_v);
                uint8_t* dst = sKV + slot * C::SLOT_BYTES;
                const uint8_t* stage = dst + C::SLOT_BYTES / 2;
                uint4 raw[D / 16];
#pragma unroll
                for (int ch = 0; ch < D / 128; ++ch)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        raw[ch * 8 + u] = *reinterpret_cast<const uint4*>(
                            stage + (kh * (D / 128) + ch) * 8192 + rr * 128 + ((u ^ (rr & 7)) << 4));
                // all converters must hold their bytes before any FP16 lands on the bytes
                // (a time-bounded barrier wait, like every other wait of the kernel)
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->conv_read[slot]);
                ok = wait_warp(&ctrl->conv_read[slot], phase_of<C::NS>(gi), w);
                if (!ok) break;
                const float sc = is_v ? a.vs : a.ks;
                const __half2 sc2 = is_v ? a.vs2 : a.ks2;
                const int k0 = (cur.tile0 + t) * BN;
                const bool live_key = k0 + ct < a.seq_k;   // rows past the cache end become zeros
#pragma unroll
                for (int q = 0; q < D / 16; ++q) {   // 16 E4M3 bytes -> 16 halves (2 units)
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                    if (live_key) {
                        if (a.scale_mode == 2) {
                            convert16<false>(raw[q], sc2, sc, lo, hi);
                        } else if (a.scale_mode == 1) {
                            convert16<true>(raw[q], sc2, sc, lo, hi);
                        } else {   // power-of-two scale: applied to the scores and outputs instead
                            const uint32_t w4[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
                            uint32_t h[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                h[2 * i] = e4m3x2_to_f16x2(w4[i] & 0xFFFFu);
                                h[2 * i + 1] = e4m3x2_to_f16x2(w4[i] >> 16);
                            }
                            lo = make_uint4(h[0], h[1], h[2], h[3]);
                            hi = make_uint4(h[4], h[5], h[6], h[7]);
                        }
                    }
                    const int d0 = q * 16;            // head-width position of the 16 values
                    const int c = d0 >> 6, u0 = (d0 & 63) >> 3;
                    uint8_t* row = dst + c * C::CHUNK + kh * C::HALF + rr * 128;
                    *reinterpret_cast<uint4*>(row + ((u0 ^ (rr & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(row + (((u0 + 1) ^ (rr & 7)) << 4)) = hi;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the MMAs
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->full[slot]);
            }
            if (!ok) break;
            ring += 2 * n;
            item_release(k);
        }
    } else if (MODE == kMasked && warp == kMaskWarp) {
        // ================= mask loader (masked mode): tile g's mask rows into slot
        // g % 2 once every softmax warp has read tile g - 2 from it
        bool ok = true;
        int tb = 0, issued = 0;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            if (!cur.valid) break;
            const int mb_b = cur.bh / a.hq, mb_h = cur.bh - mb_b * a.hq;
            for (int t = 0; t < cur.n_tiles; ++t) {
                const int g = tb + t;
                if (g >= 2 && !wait_warp(&mbar[2 + (g & 1)], ((g >> 1) - 1) & 1, w)) {
                    ok = false;
                    break;
                }
                int f0, f1;
                tile_keys(cur, nullptr, t, f0, f1);
                if (elect_one()) {
                    uint8_t* dst = sMask + (g & 1) * kMaskSlotBytes;
                    mbar_arrive_expect_tx(&mbar[g & 1], kMaskSlotBytes);
                    tma_load_4d(dst, &tmM, &mbar[g & 1], f0, cur.q_row0, a.mask_sh ? mb_h : 0,
                                a.mask_sb ? mb_b : 0);
                    tma_load_4d(dst + kMaskSlotBytes / 2, &tmM, &mbar[g & 1], f1, cur.q_row0,
                                a.mask_sh ? mb_h : 0, a.mask_sb ? mb_b : 0);
                }
                __syncwarp();
                issued = g + 1;
            }
            if (!ok) break;
            tb += cur.n_tiles;
            item_release(k);
        }
        if (!ok && lane == 0)   // copies in flight must land before the CTA exits
            for (int g = max(0, issued - 2); g < issued; ++g) drain_wait(&mbar[g & 1], (g >> 1) & 1);
        __syncwarp();
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
        const int row_half = row >> 6;
        uint64_t* xbar = &ctrl->xchg[quarter];
        // Exponent factor: scores arrive raw (scale*log2e applies), or in masked
        // mode as y = scale*s + mask (log2e applies).
        const float sl2 = MODE == kMasked ? 1.4426950408889634f : a.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t xphase = 0;
        Cursor<C::NSB> sc;   // S buffer and phase of the CTA's tile g
        Cursor<2> gp;        // g & 1 and (g >> 1) & 1 (exchange buffer, mask slot)
        int prev_buf = 0;    // S buffer and phase of tile g - 1
        uint32_t prev_phase = 0;
        bool ok = true;
        for (int k = 0; ok && (kPersist || k < 1); ++k) {
            Item cur;
            ok = get_item(k, cur);
            if (!ok) break;
            if (!cur.valid) break;
            const SparseSlot* sl = slots + (k & 1);
            const int n_tiles = cur.n_tiles;
            // token row of this thread's query row (a missing second cube: past the end)
            const int rb = row < 64 ? cur.rbase0 : cur.rbase1;
            const long long row_g =
                rb < 0 ? static_cast<long long>(a.seq_q) : static_cast<long long>(rb) + (row & 63);
            bool pad_row = false;   // a padding query slot of a boundary cube, read before the loop
            if (MODE == kSparseFull && a.cube_valid && row_g >= a.prefix && row_g < a.seq_q) {
                const int vr = static_cast<int>(row_g - a.prefix);
                pad_row = (vr & 63) >= cube_count(a, vr >> 6);
            }
            int lim = a.seq_k;   // keys >= lim are invisible to this row
            if (is_causal(MODE))
                lim = static_cast<int>(min(static_cast<long long>(a.seq_k), a.kv_prefix + row_g + 1));
            const int lim0 = is_causal(MODE)
                                 ? static_cast<int>(min(static_cast<long long>(a.seq_k),
                                                        static_cast<long long>(a.kv_prefix) + cur.q_row0 + 1))
                                 : a.seq_k;
            float m_run = -INFINITY, l = 0.0f;
            // Masked mode: tile g's mask arrives in slot g % 2, this thread's row of
            // its half at [half][row][128 bytes] (staged by the mask warp).
            for (int j = 0; j < n_tiles; ++j) {
                // (one item per CTA: the running tile count is j, and the plain
                // j-based form measured 1-1.5% faster than the cursors in dense)
                const int buf = kPersist ? sc.idx : j % C::NSB;
                const uint32_t sphase = kPersist ? sc.phase : (j / C::NSB) & 1;
                const int gb = kPersist ? gp.idx : j & 1;                 // g & 1
                const uint32_t gph = kPersist ? gp.phase : (j >> 1) & 1;  // (g >> 1) & 1
                const uint32_t sbuf = tl + buf * 128;
                // Sparse modes: this half's visible-column limit (a hidden quadrant 0, a
                // boundary cube its real-key count), read before S arrives so that its
                // shared-memory latency stays off the path from S to P.
                int lim_c = 64;
                if (is_sparse(MODE)) {
                    const uint32_t ti = sl->info[j];
                    const bool vis = (ti >> (row_half * 2 + half)) & 1u;
                    // plain VSA: all 64 keys or none (a limit the compiler can see)
                    lim_c = !vis ? 0 : MODE == kSparseFull ? static_cast<int>((ti >> (8 + 8 * half)) & 0xFFu) : 64;
                }
                ok = wait_warp(&ctrl->s_full[buf], sphase, w);
                if (!ok) break;
                tc_fence_after();
                uint32_t s[64];
                tmem_ld32(sbuf + half * 64, s);
                tmem_ld32(sbuf + half * 64 + 32, s + 32);
                tmem_ld_wait();

                int k0, k1;
                tile_keys(cur, sl, j, k0, k1);
                if (MODE == kMasked) {
                    // y = scale * s + mask, then hidden keys -> -inf.
                    ok = wait_warp(&mbar[gb], gph, w);
                    if (!ok) break;
                    const uint64_t sc2 = f2_pack(a.scale, a.scale);
                    const uint8_t* mrow =
                        sMask + gb * kMaskSlotBytes + half * (kMaskSlotBytes / 2) + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 mv = *reinterpret_cast<const uint4*>(mrow + ((c ^ (lane & 7)) << 4));
                        const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 4 * c + e;   // key pair 2i, 2i+1
                            const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mw[e]));
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                             sc2, f2_pack(mf.x, mf.y)),
                                      x0, x1);
                            s[2 * i] = __float_as_uint(x0);
                            s[2 * i + 1] = __float_as_uint(x1);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&mbar[2 + gb]);   // this warp is done with the slot
                    // keys past the end and rows past the end hidden through one column limit
                    const int kh = half ? k1 : k0;
                    const int lim_m = row_g >= a.seq_q ? 0 : a.seq_k - kh;
                    if (lim_m < 64) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (c >= lim_m) s[c] = __float_as_uint(-INFINITY);
                    }
                } else if (is_sparse(MODE)) {
                    // One column limit per tile half (read above): a quadrant hidden from
                    // this row's cube hides all 64 keys, a boundary cube its padding keys.
                    // (Two separate masking loops here had cost the full-layout kernel 45
                    // registers and a quarter of its speed.)
                    if (lim_c < 64) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (c >= lim_c) s[c] = __float_as_uint(-INFINITY);
                    }
                } else {
                    const int kh = half ? k1 : k0;
                    if (kh + 64 > lim0) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (kh + c >= lim) s[c] = __float_as_uint(-INFINITY);
                    }
                }
                // row max of the 64 values with four independent chains (short latency):
                // s[0..3] start the chains, s[4..59] in seven steps of eight, s[60..63] last
                float m4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) m4[q] = __uint_as_float(s[q]);
#pragma unroll
                for (int c = 4; c < 60; c += 8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        m4[q] = max3f(m4[q], __uint_as_float(s[c + q]), __uint_as_float(s[c + 4 + q]));
                }
                m4[0] = max3f(m4[0], __uint_as_float(s[60]), __uint_as_float(s[61]));
                m4[1] = max3f(m4[1], __uint_as_float(s[62]), __uint_as_float(s[63]));
                const float pm = fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
                ex->mx[gb][half][row] = pm;
                tc_fence_before();   // our S loads are ordered before the partner's P stores
                mbar_arrive(xbar);
                ok = wait_warp(xbar, xphase, w);
                xphase ^= 1u;
                if (!ok) break;
                tc_fence_after();
                const float mx = fmaxf(pm, ex->mx[gb][half ^ 1][row]);
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
                for (int q = 0; q < 4; ++q) rs[q] = f2_pack(0.0f, 0.0f);
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
                    if (PS) {   // keep p for its low half
                        s[2 * i] = __float_as_uint(p0);
                        s[2 * i + 1] = __float_as_uint(p1);
                    }
                }
                float r0, r1, r2, r3, r4, r5, r6, r7;
                f2_unpack(rs[0], r0, r1);
                f2_unpack(rs[1], r2, r3);
                f2_unpack(rs[2], r4, r5);
                f2_unpack(rs[3], r6, r7);
                l = l * alpha + (((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7)));
                // P_g over the first 64 columns of its S buffer; both threads of the
                // row have loaded their S halves (they passed the exchange above).
                tmem_st32(sbuf + half * 32, p2);
                if (PS) {   // lo = RNE(p - hi); p - hi is exact in FP32
                    uint32_t lo2[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&p2[i]));
                        lo2[i] = pack_half2(__uint_as_float(s[2 * i]) - h.x, __uint_as_float(s[2 * i + 1]) - h.y);
                    }
                    tmem_st32(sbuf + 64 + half * 32, lo2);
                }
                tmem_st_wait();
                if (warp_need && j > 0) {   // rescale this thread's half of O after PV_{g-1}
                    ok = wait_warp(&ctrl->pv_done[kPersist ? prev_buf : (j - 1) % C::NSB],
                                   kPersist ? prev_phase : ((j - 1) / C::NSB) & 1, w);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                    for (int cc = 0; cc < D / 64; ++cc) {
                        const uint32_t col = tl + C::T_O + half * (D / 2) + cc * 32;
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
                if (kPersist) {
                    prev_buf = buf;
                    prev_phase = sphase;
                    sc.step();
                    gp.step();
                }
            }
            if (!ok) break;
            if (n_tiles > 0) {   // PV of the item's last tile
                ok = wait_warp(&ctrl->pv_done[kPersist ? prev_buf : (n_tiles - 1) % C::NSB],
                               kPersist ? prev_phase : ((n_tiles - 1) / C::NSB) & 1, w);
                tc_fence_after();
            }
            if (!ok) break;
            // combine the two partial row sums
            ex->l[half][row] = l;
            mbar_arrive(xbar);
            ok = wait_warp(xbar, xphase, w);
            xphase ^= 1u;
            if (!ok) break;
            l += ex->l[half ^ 1][row];
            // O out of tensor memory 32 columns at a time; once the last chunk is in
            // registers the next item's first PV may overwrite O.
            item_release(k);
            const bool row_ok = row_g < a.seq_q;
            const bool zero_row = (is_causal(MODE) && row_g >= a.q_real) || pad_row;
            const float inv_l = (l > 0.0f && !zero_row) ? (MODE == kCausalPaged ? a.out_mul : 1.0f) / l : 0.0f;
            const float lse2 = (l > 0.0f && !zero_row) ? m_run + __log2f(l) : -INFINITY;
            const bool partial = is_causal(MODE) && a.n_chunks > 1;
            const int qb = cur.bh / a.hq, qh = cur.bh - qb * a.hq;
            const long long orow = static_cast<long long>(cur.bh) * a.seq_q + row_g;
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t o[32];
                if (n_tiles > 0) {
                    tmem_ld32(tl + C::T_O + half * (D / 2) + cc * 32, o);
                    tmem_ld_wait();
                    if (kPersist && cc == D / 64 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctrl->o_free);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (!row_ok) continue;
                {
                    const int c0 = half * (D / 2) + cc * 32;   // first output column of this chunk
                    const uint32_t* oc32 = o;
                    if (partial) {
                        float4* dst = reinterpret_cast<float4*>(
                            a.part_o + ((static_cast<long long>(cur.chunk) * a.heads_q * a.seq_q + orow) * D + c0));
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(oc32[4 * e]) * inv_l,
                                                 __uint_as_float(oc32[4 * e + 1]) * inv_l,
                                                 __uint_as_float(oc32[4 * e + 2]) * inv_l,
                                                 __uint_as_float(oc32[4 * e + 3]) * inv_l);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(a.o + qb * a.o_sb + qh * a.o_sh +
                                                              row_g * a.o_sr + c0);
                        float y[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) y[e] = __uint_as_float(oc32[e]) * inv_l;
                        if (is_sparse(MODE) && a.coarse && row_g >= a.prefix && !pad_row) {
                            // coarse branch: o += gate * o_coarse[cube of the row]
                            const int cube = static_cast<int>((row_g - a.prefix) >> 6);
                            const float4* ocv = reinterpret_cast<const float4*>(
                                a.coarse + (static_cast<long long>(cur.bh) * a.n_cubes + cube) * D + c0);
                            const uint4* gt = reinterpret_cast<const uint4*>(
                                a.gate + (static_cast<long long>(cur.bh) * a.seq_q + row_g) * D + c0);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint4 gw = gt[e];
                                const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
                                const float4 c0v = ocv[2 * e], c1v = ocv[2 * e + 1];
                                const float cv[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1v.x, c1v.y, c1v.z, c1v.w};
#pragma unroll
                                for (int f = 0; f < 4; ++f) {
                                    const float2 g2 = __half22float2(*reinterpret_cast<const __half2*>(&gv[f]));
                                    y[8 * e + 2 * f] = fmaf(g2.x, cv[2 * f], y[8 * e + 2 * f]);
                                    y[8 * e + 2 * f + 1] = fmaf(g2.y, cv[2 * f + 1], y[8 * e + 2 * f + 1]);
                                }
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t hw[4];
#pragma unroll
                            for (int f = 0; f < 4; ++f) hw[f] = pack_half2(y[8 * e + 2 * f], y[8 * e + 2 * f + 1]);
                            dst[e] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        }
                    }
                }
            }
            if (row_ok && half == 0) {
                if (partial)
                    a.part_lse[static_cast<long long>(cur.chunk) * a.heads_q * a.seq_q + orow] = lse2;
                else if (a.lse)
                    a.lse[orow] = lse2 * 0.69314718055994531f;
            }
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

// Combine the per-chunk FP32 partials of the causal prefill (the final merge of
// the FP32 prefix/tail states): with L_c = log2-sum-exp2 of chunk c,
// L = log2(sum_c 2^L_c) and O = sum_c 2^(L_c - L) O_c.  One warp per row.
// Six CTAs per SM (at most 40 registers): the merge streams the FP32 partials,
// and full occupancy with 60 registers (four CTAs) left DRAM idle (82 against
// 72 us for the 7-chunk, 131,072-key prefill; eight CTAs at 32 registers spill).
template <int D>
__global__ void __launch_bounds__(256, 6) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_lse,
                                                         int n_chunks, long long rows, int seq_q,
                                                         int q_real, int hq, Strides os,
                                                         __half* __restrict__ o,
                                                         float* __restrict__ lse) {
    const long long row = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = static_cast<int>(row % seq_q);
    constexpr int PER = D / 32;   // elements per lane (contiguous)
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
    float total = -INFINITY;
    if (i < q_real) {
        float mx = -INFINITY;
        for (int c = 0; c < n_chunks; ++c) mx = fmaxf(mx, part_lse[c * rows + row]);
        if (mx != -INFINITY) {
            float wsum = 0.0f;
            for (int c = 0; c < n_chunks; ++c) wsum += exp2f(part_lse[c * rows + row] - mx);
            total = mx + log2f(wsum);
            for (int c = 0; c < n_chunks; ++c) {
                const float wc = exp2f(part_lse[c * rows + row] - total);
                if (wc == 0.0f) continue;
                const float4* src =
                    reinterpret_cast<const float4*>(part_o + (c * rows + row) * D + lane * PER);
#pragma unroll
                for (int e = 0; e < PER / 4; ++e) {
                    const float4 v = src[e];
                    acc[4 * e] += wc * v.x;
                    acc[4 * e + 1] += wc * v.y;
                    acc[4 * e + 2] += wc * v.z;
                    acc[4 * e + 3] += wc * v.w;
                }
            }
        }
    }
    const long long bh = row / seq_q;
    const long long ob = bh / hq, oh = bh - ob * hq;
    uint32_t* dst = reinterpret_cast<uint32_t*>(o + ob * os.b + oh * os.h + i * os.r + lane * PER);
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) dst[e] = pack_half2(acc[2 * e], acc[2 * e + 1]);
    if (lse && lane == 0) lse[row] = total * 0.69314718055994531f;
}

template <int D, int MODE, bool PS = false>
int set_smem_attr() {
    static std::once_flag once[64];
    static int rc[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBATTN_ERR_CUDA;
    std::call_once(once[dev], [&] {
        rc[dev] = cudaFuncSetAttribute(attn_fwd_kernel<D, MODE, PS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes<D, MODE>()) == cudaSuccess
                      ? GBATTN_OK
                      : GBATTN_ERR_CUDA;
    });
    return rc[dev];
}

template <int D, int MODE, bool PS = false>
int launch_attn(const void* q, const void* k, const void* v, int seq_q, int seq_k, int heads_q,
                const Strides& qs, const Strides& kvs, long long n_items, int items_x,
                AttnArgs args, cudaStream_t stream, const CUtensorMap* mask_map = nullptr,
                const CUtensorMap* kv_maps = nullptr) {
    // Persistent modes: one CTA per SM (never more than items); otherwise one CTA
    // per item.  Item numbers and the counter's draws stay in int.
    if (n_items <= 0 || n_items > 0x7FFFFFFFLL - args.nsm) return GBATTN_ERR_SHAPE;
    args.n_items = static_cast<int>(n_items);
    args.items_x = items_x;
    // One CTA per item: a 2-D grid (items of a row x rows), in the item order; on
    // GB300 this ran dense attention 1-2% faster than the same order as a 1-D grid.
    const dim3 grid = persistent(MODE)
                          ? dim3(static_cast<unsigned>(std::min<long long>(n_items, args.nsm)))
                          : dim3(static_cast<unsigned>(items_x), static_cast<unsigned>(n_items / items_x));
    // 4-D maps (D, S, heads, batch) with the callers' strides; boxes past a head's
    // last row read zeros and never cross into another head
    const int batch = heads_q / args.hq;
    CUtensorMap tq, tk, tv;
    if (encode_tmap_f16_4d(&tq, q, D, seq_q, args.hq, batch, qs.r, qs.h, qs.b, 64, BM) != GBATTN_OK)
        return GBATTN_ERR_CUDA;
    if (kv_maps) {   // paged E4M3 K and V
        tk = kv_maps[0];
        tv = kv_maps[1];
    } else if (encode_tmap_f16_4d(&tk, k, D, seq_k, args.hkv, batch, kvs.r, kvs.h, kvs.b, 64, 64) !=
                   GBATTN_OK ||
               encode_tmap_f16_4d(&tv, v, D, seq_k, args.hkv, batch, kvs.r, kvs.h, kvs.b, 64, 64) !=
                   GBATTN_OK) {
        return GBATTN_ERR_CUDA;
    }
    CUtensorMap tq64;   // sparse modes: query cubes load as two 64-row boxes
    if (is_sparse(MODE) &&
        encode_tmap_f16_4d(&tq64, q, D, seq_q, args.hq, batch, qs.r, qs.h, qs.b, 64, 64) != GBATTN_OK)
        return GBATTN_ERR_CUDA;
    int rc = set_smem_attr<D, MODE, PS>();
    if (rc != GBATTN_OK) return rc;
    attn_fwd_kernel<D, MODE, PS><<<grid, threads_for(MODE), smem_bytes<D, MODE>(), stream>>>(
        tq, tk, tv, mask_map ? *mask_map : (is_sparse(MODE) ? tq64 : tq), args);
    count_launches(1);
    return launch_status();
}


AttnArgs base_args(const DeviceState& dev, float scale) {
    AttnArgs a{};
    a.fault = fault_mode();
    a.scale_log2 = scale * 1.4426950408889634f;
    a.scale = scale;
    a.status = dev.status;
    a.nsm = dev.num_sms > 0 ? dev.num_sms : 148;
    a.wait_limit = wait_limit_ns();
    a.group = 1;
    return a;
}

void set_out_strides(AttnArgs& a, const Strides& os) {
    a.o_sb = os.b;
    a.o_sh = os.h;
    a.o_sr = os.r;
}

Strides dense_strides(int H, int S, int D) {
    Strides t;
    make_strides(nullptr, 2, H, S, D, false, &t);   // B=2 keeps the dense batch stride
    return t;
}

// Key-range chunks per causal query tile: minimise (waves of CTAs) / chunks
// plus a small charge per chunk for the merge traffic, keeping at least two
// key tiles per chunk.  The rule depends only on the padded query count, so
// the workspace query and the call agree; real queries fewer than Q_pad only
// lengthen the key ranges.
int choose_chunks(int B, int Hq, int Q_pad, int KV, int nsm) {
    const long long nqt = (Q_pad + BM - 1) / BM;
    const long long units = static_cast<long long>(B) * Hq * nqt;
    const long long q_real_max = std::min(Q_pad, KV);
    const long long kend0 = std::min<long long>(KV, KV - q_real_max + BM);
    const long long tmin = (kend0 + BN - 1) / BN;
    int best = 1;
    double best_cost = 1e30;
    for (int c = 1; c <= 8; ++c) {
        if (c > 1 && tmin < 2LL * c) break;
        const long long waves = (units * c + nsm - 1) / nsm;
        const double cost = static_cast<double>(waves) / c + 0.01 * c;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

size_t causal_workspace(int chunks, int B, int Hq, int Q_pad, int D) {
    if (chunks <= 1) return 0;
    return static_cast<size_t>(chunks) * B * Hq * Q_pad * (static_cast<size_t>(D) + 1) *
           sizeof(float);
}

int sm_count_or_default() {
    DeviceState d;
    return current_device(&d) == GBATTN_OK ? d.num_sms : 148;
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;



extern "C" int attn_dense_mask_fwd(const void* q, const void* k, const void* v, const void* mask,
                                   long long mask_stride_b, long long mask_stride_h, void* o,
                                   float* lse, int B, int H, int Sq, int Skv, int D, float scale,
                                   void* stream) {
    CallRange nvtx_range("attn_dense_mask_fwd");
    if (!q || !k || !v || !mask || !o) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || Sq <= 0 || Skv <= 0) return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    const long long slice = static_cast<long long>(Sq) * Skv;
    if (mask_stride_b < 0 || mask_stride_h < 0 || Skv % 8 != 0 || mask_stride_b % 8 != 0 ||
        mask_stride_h % 8 != 0 || (mask_stride_h != 0 && mask_stride_h < slice) ||
        (mask_stride_b != 0 && mask_stride_b < slice))
        return GBATTN_ERR_SHAPE;
    if (D != 128) return GBATTN_ERR_UNSUPPORTED;
    if (!finite_positive(scale)) return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(mask) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t qb = static_cast<size_t>(B) * H * Sq * D * 2;
    const size_t kb = static_cast<size_t>(B) * H * Skv * D * 2;
    const size_t lb = static_cast<size_t>(B) * H * Sq * 4;
    const size_t mb = (static_cast<size_t>(B - 1) * mask_stride_b +
                       static_cast<size_t>(H - 1) * mask_stride_h +
                       static_cast<size_t>(Sq) * Skv) * 2;
    if (overlaps(o, qb, q, qb) || overlaps(o, qb, k, kb) || overlaps(o, qb, v, kb) ||
        overlaps(o, qb, mask, mb) || overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) ||
        overlaps(lse, lb, v, kb) || overlaps(lse, lb, mask, mb) || overlaps(lse, lb, o, qb))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    AttnArgs a = base_args(dev, scale);
    a.seq_q = Sq;
    a.seq_k = Skv;
    a.heads_q = B * H;
    a.hq = H;
    a.hkv = H;
    a.n_chunks = 1;
    a.o = static_cast<__half*>(o);
    a.lse = lse;
    a.mask = static_cast<const __half*>(mask);
    a.mask_sb = mask_stride_b;
    a.mask_sh = mask_stride_h;
    // Mask map [b][h][Sq][Skv]; a shared dimension has extent 1 (its stride is
    // then only a placeholder the encoder accepts).
    const uint64_t hm = mask_stride_h ? H : 1, bm = mask_stride_b ? B : 1;
    const uint64_t sh = mask_stride_h ? mask_stride_h : slice;
    const uint64_t sb = mask_stride_b ? mask_stride_b : sh * hm;
    CUtensorMap tm;
    if (encode_tmap_f16_mask(&tm, mask, Skv, Sq, hm, bm, sh, sb) != GBATTN_OK)
        return GBATTN_ERR_CUDA;
    set_out_strides(a, dense_strides(H, Sq, D));
    return launch_attn<128, kMasked>(q, k, v, Sq, Skv, B * H, dense_strides(H, Sq, D),
                                     dense_strides(H, Skv, D),
                                     static_cast<long long>((Sq + BM - 1) / BM) * B * H, B * H, a,
                                     static_cast<cudaStream_t>(stream), &tm);
}

extern "C" size_t attn_causal_prefill_workspace_size(int B, int Hq, int Q_pad, int KV, int D) {
    if (B <= 0 || Hq <= 0 || Q_pad <= 0 || KV <= 0 || D <= 0) return 0;
    return causal_workspace(choose_chunks(B, Hq, Q_pad, KV, sm_count_or_default()), B, Hq, Q_pad,
                            D);
}

extern "C" int attn_causal_prefill_fwd(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int Hq, int Hkv, int Q_pad, int Q_real,
                                       int KV, int D, const int64_t* q_strides,
                                       const int64_t* kv_strides, const int64_t* o_strides,
                                       float scale, int flags, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    CallRange nvtx_range("attn_causal_prefill_fwd");
    if (!q || !k || !v || !o) return GBATTN_ERR_NULL;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Q_pad <= 0 || KV <= 0) return GBATTN_ERR_SHAPE;
    if (Hq % Hkv != 0 || Q_pad % 64 != 0 || Q_real < 1 || Q_real > Q_pad || Q_real > KV ||
        KV % 32 != 0)
        return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq > 65535) return GBATTN_ERR_SHAPE;
    if (flags & ~GBATTN_PROB_SPLIT) return GBATTN_ERR_SHAPE;
    if (D != 256) return GBATTN_ERR_UNSUPPORTED;
    Strides qs, kvs, os;
    if (!make_strides(q_strides, B, Hq, Q_pad, D, false, &qs) ||
        !make_strides(kv_strides, B, Hkv, KV, D, false, &kvs) ||
        !make_strides(o_strides, B, Hq, Q_pad, D, true, &os))
        return GBATTN_ERR_SHAPE;
    if (!finite_positive(scale)) return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t qb = strided_bytes(qs, B, Hq, Q_pad, D);
    const size_t kb = strided_bytes(kvs, B, Hkv, KV, D);
    const size_t ob = strided_bytes(os, B, Hq, Q_pad, D);
    const size_t lb = static_cast<size_t>(B) * Hq * Q_pad * 4;
    if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, kb) ||
        overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
        overlaps(lse, lb, o, ob))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    int chunks = choose_chunks(B, Hq, Q_pad, KV, dev.num_sms);
    while (chunks > 1 && (!workspace || workspace_bytes < causal_workspace(chunks, B, Hq, Q_pad, D)))
        --chunks;
    const size_t wb = causal_workspace(chunks, B, Hq, Q_pad, D);
    if (wb > 0 && (overlaps(workspace, wb, q, qb) || overlaps(workspace, wb, k, kb) ||
                   overlaps(workspace, wb, v, kb) || overlaps(workspace, wb, o, ob) ||
                   overlaps(workspace, wb, lse, lb)))
        return GBATTN_ERR_ALIAS;
    AttnArgs a = base_args(dev, scale);
    a.seq_q = Q_pad;
    a.seq_k = KV;
    a.heads_q = B * Hq;
    a.hq = Hq;
    a.hkv = Hkv;
    a.group = Hq / Hkv;
    a.q_real = Q_real;
    a.kv_prefix = KV - Q_real;
    a.n_chunks = chunks;
    a.o = static_cast<__half*>(o);
    set_out_strides(a, os);
    a.lse = lse;
    const long long rows = static_cast<long long>(B) * Hq * Q_pad;
    if (chunks > 1) {
        a.part_o = static_cast<float*>(workspace);
        a.part_lse = a.part_o + static_cast<size_t>(chunks) * rows * D;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ix = ((Q_pad + BM - 1) / BM) * chunks;
    const long long ni = static_cast<long long>(ix) * B * Hq;
    rc = (flags & GBATTN_PROB_SPLIT)
             ? launch_attn<256, kCausal, true>(q, k, v, Q_pad, KV, B * Hq, qs, kvs, ni, ix, a, s)
             : launch_attn<256, kCausal>(q, k, v, Q_pad, KV, B * Hq, qs, kvs, ni, ix, a, s);
    if (rc != GBATTN_OK || chunks == 1) return rc;
    const long long threads = rows * 32;
    attn_merge_kernel<256><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(
        a.part_o, a.part_lse, chunks, rows, Q_pad, Q_real, Hq, os, a.o, lse);
    count_launches(1);
    return launch_status();
}

extern "C" int attn_causal_prefill_paged_fwd(const void* q, const uint8_t* k_pages,
                                             const uint8_t* v_pages, const int32_t* page_table,
                                             void* o, float* lse, int B, int Hq, int Hkv,
                                             int Q_pad, int Q_real, int KV, int D,
                                             int num_phys_pages, int page_size, int max_pages,
                                             float k_scale, float v_scale, float scale,
                                             int flags, void* workspace, size_t workspace_bytes,
                                             void* stream) {
    CallRange nvtx_range("attn_causal_prefill_paged_fwd");
    if (!q || !k_pages || !v_pages || !page_table || !o) return GBATTN_ERR_NULL;
    if (flags & ~GBATTN_PROB_SPLIT) return GBATTN_ERR_SHAPE;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Q_pad <= 0 || KV <= 0 || num_phys_pages <= 0 ||
        page_size <= 0 || max_pages <= 0)
        return GBATTN_ERR_SHAPE;
    if (Hq % Hkv != 0 || Q_pad % 64 != 0 || Q_real < 1 || Q_real > Q_pad || Q_real > KV ||
        KV % 32 != 0 || static_cast<long long>(KV) > static_cast<long long>(max_pages) * page_size)
        return GBATTN_ERR_SHAPE;
    if (static_cast<long long>(B) * Hq > 65535) return GBATTN_ERR_SHAPE;
    if (D != 256) return GBATTN_ERR_UNSUPPORTED;
    if (page_size < 16 || (page_size & (page_size - 1)) != 0 ||
        static_cast<long long>(num_phys_pages) * page_size > 0x7FFFFFFFLL)
        return GBATTN_ERR_UNSUPPORTED;
    if (!finite_positive(scale) || !finite_positive(k_scale) || !finite_positive(v_scale))
        return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    const size_t qb = static_cast<size_t>(B) * Hq * Q_pad * D * 2;
    const size_t pb = static_cast<size_t>(num_phys_pages) * page_size * Hkv * D;
    const size_t tb = static_cast<size_t>(B) * max_pages * 4;
    const size_t lb = static_cast<size_t>(B) * Hq * Q_pad * 4;
    if (overlaps(o, qb, q, qb) || overlaps(o, qb, k_pages, pb) || overlaps(o, qb, v_pages, pb) ||
        overlaps(o, qb, page_table, tb) || overlaps(lse, lb, q, qb) ||
        overlaps(lse, lb, k_pages, pb) || overlaps(lse, lb, v_pages, pb) ||
        overlaps(lse, lb, page_table, tb) || overlaps(lse, lb, o, qb))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    int chunks = choose_chunks(B, Hq, Q_pad, KV, dev.num_sms);
    while (chunks > 1 && (!workspace || workspace_bytes < causal_workspace(chunks, B, Hq, Q_pad, D)))
        --chunks;
    const size_t wb = causal_workspace(chunks, B, Hq, Q_pad, D);
    if (wb > 0 && (overlaps(workspace, wb, q, qb) || overlaps(workspace, wb, k_pages, pb) ||
                   overlaps(workspace, wb, v_pages, pb) || overlaps(workspace, wb, o, qb) ||
                   overlaps(workspace, wb, page_table, tb) || overlaps(workspace, wb, lse, lb)))
        return GBATTN_ERR_ALIAS;
    const int box = page_size < 64 ? page_size : 64;
    CUtensorMap kv[2];
    const uint64_t total_rows = static_cast<uint64_t>(num_phys_pages) * page_size;
    if (encode_tmap_u8_pages(&kv[0], k_pages, D, Hkv, total_rows, box) != GBATTN_OK ||
        encode_tmap_u8_pages(&kv[1], v_pages, D, Hkv, total_rows, box) != GBATTN_OK)
        return GBATTN_ERR_CUDA;
    // exact scaled values: a power of two in [2^-15, 2^7] folds into the score
    // scale and the output; an FP16-valued scale uses one FP16 multiply; any
    // other scale the round-to-odd product (the bridge's rule)
    auto pow2_in = [](float sv) {
        int e = 0;
        const float m = frexpf(sv, &e);
        return m == 0.5f && e - 1 >= -15 && e - 1 <= 7;
    };
    const int mode = pow2_in(k_scale) && pow2_in(v_scale) ? 0
                     : (is_fp16_value(k_scale) && is_fp16_value(v_scale)) ? 1 : 2;
    AttnArgs a = base_args(dev, scale * (mode == 0 ? k_scale : 1.0f));
    a.seq_q = Q_pad;
    a.seq_k = KV;
    a.heads_q = B * Hq;
    a.hq = Hq;
    a.hkv = Hkv;
    a.group = Hq / Hkv;
    a.q_real = Q_real;
    a.kv_prefix = KV - Q_real;
    a.n_chunks = chunks;
    a.o = static_cast<__half*>(o);
    a.lse = lse;
    a.page_table = page_table;
    a.num_phys = num_phys_pages;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.page_box = box;
    a.scale_mode = mode;
    a.ks = k_scale;
    a.vs = v_scale;
    a.ks2 = __float2half2_rn(k_scale);
    a.vs2 = __float2half2_rn(v_scale);
    a.out_mul = mode == 0 ? v_scale : 1.0f;
    const Strides qs = dense_strides(Hq, Q_pad, D);
    set_out_strides(a, qs);
    const long long rows = static_cast<long long>(B) * Hq * Q_pad;
    if (chunks > 1) {
        a.part_o = static_cast<float*>(workspace);
        a.part_lse = a.part_o + static_cast<size_t>(chunks) * rows * D;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ix = ((Q_pad + BM - 1) / BM) * chunks;
    const long long ni = static_cast<long long>(ix) * B * Hq;
    rc = (flags & GBATTN_PROB_SPLIT)
             ? launch_attn<256, kCausalPaged, true>(q, nullptr, nullptr, Q_pad, KV, B * Hq, qs, qs,
                                                    ni, ix, a, s, nullptr, kv)
             : launch_attn<256, kCausalPaged>(q, nullptr, nullptr, Q_pad, KV, B * Hq, qs, qs, ni,
                                              ix, a, s, nullptr, kv);
    if (rc != GBATTN_OK || chunks == 1) return rc;
    const long long threads = rows * 32;
    attn_merge_kernel<256><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(
        a.part_o, a.part_lse, chunks, rows, Q_pad, Q_real, Hq, qs, a.o, lse);
    count_launches(1);
    return launch_status();
}


extern "C" int vsa_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                              const int32_t* pairs, int prefix, const int32_t* cube_valid,
                              const float* o_coarse, const void* gate, void* o, float* lse, int B,
                              int H, int S, int D, int block, int topk, float scale,
                              void* workspace, size_t workspace_bytes, void* stream) {
    CallRange nvtx_range("vsa_sparse_fwd");
    if (!q || !k || !v || !idx || !o || (!o_coarse) != (!gate)) return GBATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || S <= 0 || topk <= 0 || prefix < 0 || prefix >= S)
        return GBATTN_ERR_SHAPE;
    if (D != 128 || block != 64) return GBATTN_ERR_UNSUPPORTED;
    if ((S - prefix) % block != 0 || prefix % BM != 0) return GBATTN_ERR_SHAPE;
    const int nc = (S - prefix) / block;
    if (topk > nc || topk > kMaxTopk) return GBATTN_ERR_SHAPE;
    if (prefix / BM + (nc + 1) / 2 > kMaxSparseTiles) return GBATTN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(cube_valid) & 3u) || (reinterpret_cast<uintptr_t>(pairs) & 3u) ||
        !aligned16(o_coarse) || !aligned16(gate))
        return GBATTN_ERR_ALIGN;
    if (static_cast<long long>(B) * H > 65535) return GBATTN_ERR_SHAPE;
    if (!finite_positive(scale)) return GBATTN_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return GBATTN_ERR_ALIGN;
    if (workspace && workspace_bytes < kSparseWorkspaceBytes) return GBATTN_ERR_WORKSPACE;
    const size_t xb = static_cast<size_t>(B) * H * S * D * 2;
    const size_t ib = static_cast<size_t>(B) * H * nc * topk * 4;
    const size_t lb = static_cast<size_t>(B) * H * S * 4;
    const size_t cb = static_cast<size_t>(B) * H * nc * D * 4;
    if (overlaps(o, xb, q, xb) || overlaps(o, xb, k, xb) || overlaps(o, xb, v, xb) ||
        overlaps(o, xb, idx, ib) || overlaps(lse, lb, q, xb) || overlaps(lse, lb, k, xb) ||
        overlaps(lse, lb, v, xb) || overlaps(lse, lb, idx, ib) || overlaps(lse, lb, o, xb) ||
        overlaps(o, xb, o_coarse, cb) || overlaps(o, xb, gate, xb) || overlaps(lse, lb, o_coarse, cb) ||
        overlaps(lse, lb, gate, xb))
        return GBATTN_ERR_ALIAS;
    const size_t wb = kSparseWorkspaceBytes, pb = static_cast<size_t>(B) * H * ((nc + 1) / 2) * 8;
    const size_t vb = static_cast<size_t>(nc) * 4;   // cube_valid: one count per cube
    if (workspace && (overlaps(workspace, wb, q, xb) || overlaps(workspace, wb, k, xb) ||
                      overlaps(workspace, wb, v, xb) || overlaps(workspace, wb, o, xb) ||
                      overlaps(workspace, wb, idx, ib) || overlaps(workspace, wb, lse, lb) ||
                      overlaps(workspace, wb, pairs, pb) || overlaps(workspace, wb, cube_valid, vb) ||
                      overlaps(workspace, wb, o_coarse, cb) || overlaps(workspace, wb, gate, xb)))
        return GBATTN_ERR_ALIAS;
    DeviceState dev;
    int rc = current_device(&dev);
    if (rc != GBATTN_OK) return rc;
    AttnArgs a = base_args(dev, scale);
    a.sched = static_cast<int*>(workspace);
    a.seq_q = S;
    a.seq_k = S;
    a.heads_q = B * H;
    a.hq = H;
    a.hkv = H;
    a.n_chunks = 1;
    a.n_cubes = nc;
    a.topk = topk;
    a.idx = idx;
    a.prefix = prefix;
    a.cube_valid = cube_valid;
    a.coarse = o_coarse;
    a.gate = static_cast<const __half*>(gate);
    a.pairs = pairs;
    a.o = static_cast<__half*>(o);
    a.lse = lse;
    const int ix = prefix / BM + (nc + 1) / 2;
    const long long ni = static_cast<long long>(ix) * B * H;
    const Strides ds = dense_strides(H, S, D);
    set_out_strides(a, ds);
    if (prefix > 0 || cube_valid)
        return launch_attn<128, kSparseFull>(q, k, v, S, S, B * H, ds, ds, ni, ix, a,
                                             static_cast<cudaStream_t>(stream));
    return launch_attn<128, kSparse>(q, k, v, S, S, B * H, ds, ds, ni, ix, a,
                                     static_cast<cudaStream_t>(stream));
}

extern "C" size_t vsa_sparse_workspace_size(void) {
    return kSparseWorkspaceBytes;
}
