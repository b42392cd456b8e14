/*
 * gbattn — fused FP16 attention for one NVIDIA GB300 (sm_103a), C ABI.
 *
 * The library computes O = softmax(scale * Q K^T + mask) V with FP16 storage,
 * FP32 accumulation of Q K^T and P V, an FP32 online-softmax state and FP16
 * probabilities ("Integrate FP32 v37 prefill and exact E4M3 bridge",
 * Implementation: FP32 QK/PV accumulation and prefix/tail state, probabilities
 * and final output stored as FP16), in these variants:
 *   - dense non-causal heads of width 128 (the video-DiT attention of "Share
 *     SM70 projection, attention and row reduction paths", Purpose), also with
 *     an additive FP16 mask (the mask term of the formula);
 *   - causal long prefill with shared-KV heads at width 256, the query block
 *     appended after a key prefix, optionally fed from a paged E4M3 cache
 *     through an exact E4M3 -> FP16 bridge, or reading the pages directly
 *     ("Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation);
 *   - decode over a paged E4M3 cache: the newest tokens of ragged sequences
 *     against their whole caches (same page, Validation: the E4M3 decode wave
 *     kernels and the 256000-input decode);
 *   - VSA block-sparse attention: 64-token cubes, mean-pooled cube scores pick
 *     the top-k key cubes of every query cube, then attention runs over only
 *     those cubes, optionally with dense prefix tokens and padded boundary
 *     cubes ("Integrate H3 SM70 execution, metrics and VSA diagnostics",
 *     Purpose: top-k = 64, prefix-dense queries, boundary handling).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates no memory; scratch space is passed in as
 *     `workspace`, sized by the matching *_workspace_size() query.
 *   - Tensors are row-major in the layout each call states, with 16-byte
 *     aligned base addresses.  They are dense, except where a call takes
 *     strides: a `*_strides` argument is NULL (dense) or a host array of three
 *     int64 element strides {batch, head, row} of a [B][H][S][D] view whose D
 *     elements are contiguous.  Strides are positive multiples of 8 elements
 *     below 2^38, the row stride is at least D; a dimension of extent 1 may
 *     carry any stride.  So a packed QKV tensor [B][S][3][H][D] passes its
 *     three slices without a copy (row stride 3*H*D, head stride D, batch
 *     stride 3*S*H*D).  An output's strides must not map two elements to one
 *     address.  Overlap checks use each tensor's whole address span, so an
 *     output interleaved between an input's rows is rejected too.
 *   - `stream` is a cudaStream_t passed as void*; all GPU work is queued on it
 *     and the call returns without waiting.  Inputs must stay unchanged and
 *     outputs unread until that work completes.
 *   - Every call returns a status (enum gbattn_status).  Arguments are
 *     validated before anything is queued; on a validation error nothing is
 *     written.  An output range that overlaps an input range is rejected.
 *   - Errors found by a kernel while it runs (a pipeline wait that passed its
 *     time limit, a page-table entry or a cube index out of range) are
 *     recorded as bits in a per-device status word, read and cleared with
 *     gbattn_device_status().
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum gbattn_status {
    GBATTN_OK = 0,
    GBATTN_ERR_NULL = 1,        /* a required pointer is NULL */
    GBATTN_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
    GBATTN_ERR_UNSUPPORTED = 3, /* a valid but unsupported configuration (e.g. head width) */
    GBATTN_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    GBATTN_ERR_ALIAS = 5,       /* an output overlaps an input */
    GBATTN_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required */
    GBATTN_ERR_CUDA = 7,        /* a CUDA runtime call failed (no device, launch error) */
    GBATTN_ERR_SCALE = 8        /* a scale is not a finite positive number */
};

/* Bits of the per-device status word written by running kernels. */
enum gbattn_device_flag {
    GBATTN_DEV_WAIT_TIMEOUT = 1u, /* an in-kernel pipeline wait exceeded its limit; the
                                     kernel stopped early and its output is invalid */
    GBATTN_DEV_BAD_PAGE = 2u,     /* a page-table entry was outside [0, num_phys_pages);
                                     that page's tokens were written as zeros */
    GBATTN_DEV_BAD_INDEX = 4u,    /* a VSA cube list was not strictly ascending or held an
                                     index outside [0, S/block); the entry was skipped */
    GBATTN_DEV_BAD_LENGTH = 8u    /* a decode sequence length was outside [nq, max_kv_len];
                                     that sequence's rows were written as O = 0, lse = -inf */
};

/* Flags of the causal prefill calls. */
enum gbattn_flag {
    GBATTN_PROB_SPLIT = 1 /* probabilities enter the P V product as two FP16 halves, hi = RNE(p)
                             and lo = RNE(p - hi) (about 22 bits of p, one more group of
                             tensor-core MMAs per key tile), instead of the pages' single FP16
                             value; the output error then no longer carries the FP16 rounding of
                             P, which for large |V| (the E4M3 cache's values reach 448 * scale)
                             can exceed a few 1e-3 where a row's output cancels */
};

/* Library version (major*10000 + minor*100 + patch). */
int gbattn_version(void);

/* Human-readable text for a gbattn_status value; never NULL. */
const char* gbattn_status_string(int status);

/* Reads and clears the status word of the current device.  Waits for all work
 * queued on `stream` first.  *flags_out receives the OR of gbattn_device_flag
 * bits seen since the previous read.  Returns GBATTN_OK or GBATTN_ERR_CUDA. */
int gbattn_device_status(void* stream, uint32_t* flags_out);

/* Upper bound, in nanoseconds, of every in-kernel wait of the attention kernels
 * (default 2e9).  A wait that passes it sets GBATTN_DEV_WAIT_TIMEOUT and the kernel
 * returns instead of hanging.  Affects launches made after the call. */
int gbattn_set_wait_limit_ns(uint64_t limit_ns);

/* Number of kernels this library has launched since it was loaded (all devices). */
uint64_t gbattn_launch_count(void);

/* Test hook for the failure path of the bounded waits (the pages ask for
 * exception-safe operator lifetimes and explicit rollback: "Integrate FP32 v37
 * prefill and exact E4M3 bridge", Purpose).  mode 1 makes every later
 * attention launch skip its query-tile load, so its first pipeline wait runs
 * out after gbattn_set_wait_limit_ns(); mode 2 makes the load warp stop after
 * the first two rounds of its K/V ring (waiting for the copies it issued), so
 * the waits run out mid-stream with tensor-core work in flight (in the fused
 * paged prefill, the E4M3 converter warps' waits run out too).  In the paged
 * decode, mode 1 makes every warp load no stage and mode 2 stop after two
 * rounds of its own ring.  Either way the kernel records
 * GBATTN_DEV_WAIT_TIMEOUT, lets its copies and MMAs finish, frees its tensor
 * memory and returns (outputs are then undefined).  mode 0 (default) restores
 * normal operation.  Returns GBATTN_OK or GBATTN_ERR_SHAPE. */
int gbattn_test_inject_fault(int mode);

/*
 * Dense non-causal attention, head width D == 128.
 * Cites: "Share SM70 projection, attention and row reduction paths", Purpose
 * (D128 attention interfaces); FastVideo compare view, minimax_h3_prefix.cu
 * (BHSD operands with a contiguous 128-wide last dimension, strided rows
 * allowed, LSE output).
 *   q, o : [B][H][Sq][D]  FP16     k, v : [B][H][Skv][D] FP16 (k and v share kv_strides)
 *   q_strides, kv_strides, o_strides: {batch, head, row} element strides or NULL (dense)
 *   lse  : optional dense [B][H][Sq] FP32, natural-log sum of exp of the scaled scores
 *   scale: finite, > 0 (typically 1/sqrt(D))
 * Sizes: B, H, Sq, Skv >= 1; B*H <= 65535; Sq, Skv < 2^31.
 */
int attn_dense_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int Sq, int Skv, int D, const int64_t* q_strides,
                   const int64_t* kv_strides, const int64_t* o_strides, float scale, void* stream);

/*
 * Causal prefill with shared-KV heads, head width D == 256.
 * Cites: "Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation
 * (causal D256 Hq6/Hkv1, queries in multiples of 64, Q < KV, KV a multiple of
 * 32, real-query causal offsets kept when queries are padded, FP32 prefix/tail
 * state and final merge, bounded workspace).
 *   q, o : [B][Hq][Q_pad][D] FP16   k, v : [B][Hkv][KV][D] FP16   lse: optional [B][Hq][Q_pad]
 *   q_strides, kv_strides, o_strides: {batch, head, row} element strides or NULL (dense)
 *   flags: 0 or GBATTN_PROB_SPLIT.
 *   Query head h reads KV head h / (Hq/Hkv).  Query i < Q_real sits at absolute
 *   position KV - Q_real + i and sees keys j <= that position.  Rows i >= Q_real
 *   are written as zeros (lse = -inf).
 *   Q_pad % 64 == 0, 1 <= Q_real <= Q_pad, Q_real <= KV, KV % 32 == 0, Hq % Hkv == 0.
 *   The key range of every query tile is split into chunks processed by
 *   separate CTAs; their FP32 partial outputs and log-sum-exps go to
 *   `workspace` and a merge kernel combines them.  A workspace smaller than
 *   attn_causal_prefill_workspace_size() makes the call use fewer chunks
 *   (down to one, which needs no workspace); NULL with 0 bytes is allowed.
 */
size_t attn_causal_prefill_workspace_size(int B, int Hq, int Q_pad, int KV, int D);
int attn_causal_prefill_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Q_pad, int Q_real, int KV, int D,
                            const int64_t* q_strides, const int64_t* kv_strides,
                            const int64_t* o_strides, float scale, int flags, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Causal prefill reading K and V straight from paged E4M3 caches (the bridge fused into the
 * attention).
 * Cites: "Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation (exact E4M3 paged
 * -> FP16 bridge with unit and non-unit scales, FP32 prefill).
 *   q, o : [B][Hq][Q_pad][D] FP16; k_pages, v_pages : [num_phys_pages][page_size][Hkv][D]
 *   bytes; page_table : int32 [B][max_pages]; lse optional FP32 [B][Hq][Q_pad].
 *   Computes exactly what e4m3_paged_to_fp16 followed by attn_causal_prefill_fwd computes: the
 *   keys and values are RNE_fp16(decode(byte) * scale), formed in shared memory from the
 *   cached bytes.  Same query positions, padding and split-KV workspace rules as
 *   attn_causal_prefill_fwd (attn_causal_prefill_workspace_size applies).  flags: 0 or
 *   GBATTN_PROB_SPLIT.
 *   D == 256; page_size a power of two >= 16; KV <= max_pages * page_size, KV % 32 == 0;
 *   num_phys_pages * page_size < 2^31.  A page-table entry outside [0, num_phys_pages) sets
 *   GBATTN_DEV_BAD_PAGE (that page reads physical page 0).
 */
int attn_causal_prefill_paged_fwd(const void* q, const uint8_t* k_pages, const uint8_t* v_pages,
                                  const int32_t* page_table, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Q_pad, int Q_real, int KV, int D,
                                  int num_phys_pages, int page_size, int max_pages, float k_scale,
                                  float v_scale, float scale, int flags, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Paged FP8 E4M3 ("fn" flavour) -> FP16 bridge.
 * Cites: "Integrate FP32 v37 prefill and exact E4M3 bridge", Purpose and
 * Implementation (exact E4M3 byte conversion, unit and non-unit scales, live
 * length); FastVideo compare view, minimax_h3_swiglu_quant.cuh scale_float
 * (exact E4M3 bit construction).
 *   k_pages, v_pages : [num_phys_pages][page_size][Hkv][D] bytes
 *   page_table       : int32 [ceil(kv_len / page_size)], logical page -> physical page
 *   k_out, v_out     : [Hkv][kv_len][D] FP16 (the K/V input of attn_causal_prefill_fwd, B = 1)
 *   out = FP16 nearest to decode(byte) * scale, ties to even (one rounding).
 *   Only tokens t < kv_len are read and written.  D % 16 == 0.  Scales finite, > 0.
 *   An out-of-range page-table entry sets GBATTN_DEV_BAD_PAGE and writes that
 *   page's tokens as zeros.
 */
int e4m3_paged_to_fp16(const uint8_t* k_pages, const uint8_t* v_pages, const int32_t* page_table,
                       int num_phys_pages, int page_size, int kv_len, int Hkv, int D,
                       float k_scale, float v_scale, void* k_out, void* v_out, void* stream);

/*
 * Dense attention with an additive mask: O = softmax(scale * Q K^T + mask) V.
 * Cites: the mask term of the attention formula; FastVideo compare view,
 * minimax_h3_fusions/block_lists.py (H3's mask builder: square masks over the
 * score matrix per batch entry and head).
 *   q, o : [B][H][Sq][D] FP16; k, v : [B][H][Skv][D] FP16; lse optional FP32 [B][H][Sq].
 *   mask : FP16; the slice of (b, h) starts at mask + b*mask_stride_b + h*mask_stride_h
 *          (element strides; 0 shares one slice) and is [Sq][Skv] row-major.  -inf hides a
 *          key; a row whose keys are all hidden gets O = 0, lse = -inf.
 *   D == 128; Skv and both strides multiples of 8 (16-byte rows); mask 16-byte aligned.
 *   Mask bytes are read once per query tile per (b, h) slice use: 2*Sq*Skv per head.
 */
int attn_dense_mask_fwd(const void* q, const void* k, const void* v, const void* mask,
                        long long mask_stride_b, long long mask_stride_h, void* o, float* lse,
                        int B, int H, int Sq, int Skv, int D, float scale, void* stream);

/*
 * Decode attention over a paged FP8 E4M3 KV cache.
 * Cites: "Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation (the
 * exact E4M3 paged -> FP16 bridge and its page table) and Validation (the E4M3
 * decode wave kernels, the 256000-input decode with shared-KV heads).
 *   q          : [B][Hq][nq][D] FP16, the nq newest tokens of every sequence
 *   k_pages,
 *   v_pages    : [num_phys_pages][page_size][Hkv][D] E4M3 bytes (the bridge's layout)
 *   page_table : int32 [B][max_pages], row b maps logical page p of sequence b to a
 *                physical page (entries past ceil(kv_lens[b] / page_size) are not read)
 *   kv_lens    : int32 [B] on the device, cached tokens per sequence, the new ones included
 *   o          : [B][Hq][nq][D] FP16; lse optional FP32 [B][Hq][nq] (natural log)
 *   Query i of sequence b sits at position kv_lens[b] - nq + i and sees the cached
 *   tokens t <= that position; query head h reads KV head h / (Hq / Hkv).  K and V
 *   are exactly the bridge's values RNE_fp16(decode(byte) * scale); scores, softmax
 *   and accumulation are FP32 (probabilities enter the PV product as FP16 hi + lo
 *   halves), O is rounded to FP16 once.
 *   D is 128 or 256; page_size a power of two >= 16; Hq % Hkv == 0; B <= 4096;
 *   nq <= max_kv_len <= max_pages * page_size; num_phys_pages * page_size < 2^31.
 *   max_kv_len bounds every kv_lens[b]; a length outside [nq, max_kv_len] sets
 *   GBATTN_DEV_BAD_LENGTH and yields O = 0, lse = -inf for that sequence.  An
 *   out-of-range page-table entry sets GBATTN_DEV_BAD_PAGE (that page reads
 *   physical page 0).
 *   The work (16-token tiles of every sequence, KV head and group of <= 8 query rows)
 *   is split evenly over the warps of a persistent grid whatever the lengths; each
 *   warp writes FP32 partial records to `workspace` and a merge kernel combines them.
 *   The workspace (required) holds one record per warp plus one per (sequence, KV
 *   head, row group); attn_paged_decode_workspace_size() gives the full-speed size,
 *   a smaller one runs fewer warps, and below one CTA's worth the call returns
 *   GBATTN_ERR_WORKSPACE.
 */
size_t attn_paged_decode_workspace_size(int B, int Hq, int Hkv, int nq, int max_kv_len, int D);
int attn_paged_decode_fwd(const void* q, const uint8_t* k_pages, const uint8_t* v_pages,
                          const int32_t* page_table, const int32_t* kv_lens, void* o, float* lse,
                          int B, int Hq, int Hkv, int nq, int D, int num_phys_pages,
                          int page_size, int max_pages, int max_kv_len, float k_scale,
                          float v_scale, float scale, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * VSA key-cube selection.
 * Cites: "Integrate H3 SM70 execution, metrics and VSA diagnostics", Purpose
 * (top-k = 64); FastVideo compare view, minimax_h3_fusions/query_pool.py and
 * key_quant.py (FP32 tile means: FP32 sum divided by the count, 64-token tiles),
 * block_lists.py (per-query-block key-block lists).
 *   q, k : [B][H][S][D] FP16.  Tokens [0, prefix) are prefix tokens (text or audio) that take
 *          no part; tokens [prefix, S) are the video tokens in cube-major order (cube c =
 *          slots prefix + c*block .. + block-1).
 *   cube_valid : int32 [(S-prefix)/block] real tokens per cube (1..block; a boundary cube of a
 *          grid the cube size does not divide holds its real tokens in its first slots and
 *          padding after them), or NULL when every cube is full.  Out-of-range counts set
 *          GBATTN_DEV_BAD_INDEX and are clamped to [1, block].
 *   idx  : int32 [B][H][(S-prefix)/block][topk], for every query cube the topk key cubes with
 *          the largest score, ties to the lower cube index, in ascending cube order.
 *   Pooled vector = FP32 sum over the cube's real tokens in token order / their count
 *   (FP32, RN); padding contents are never read.
 *   Score = the exact dot product of the two FP32 pooled vectors (no rounding): FP32
 *   scores with a rigorous error bound decide almost every key, and the keys whose
 *   FP32 score lies within that bound of the k-th value are ranked by exact integer
 *   scores.  (Inputs holding Inf or NaN give an unspecified but valid selection.)
 *   block == 64, D == 128, (S - prefix) % block == 0, 1 <= topk <= (S-prefix)/block <= 1024.
 *   Workspace: vsa_select_workspace_size() bytes for rows = B*H*(S/block) query cubes:
 *   the FP32 means of Q and K (rows*D*4 each), their norms and one int32 flag per row
 *   (rows*4 each), and the FP32 scores (rows * (S/block rounded up to 128) * 4), each
 *   part rounded up to 256 bytes.
 */
size_t vsa_select_workspace_size(int B, int H, int S, int D, int block);
int vsa_select_blocks(const void* q, const void* k, int B, int H, int S, int D, int block,
                      int topk, int prefix, const int32_t* cube_valid, int32_t* idx,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * The selection plus the coarse ("compression") branch of VSA.
 * Cites: "Integrate H3 SM70 execution, metrics and VSA diagnostics", Purpose (VSA with
 * learned compression); FastVideo compare view, minimax_h3_fusions/kv_pool.py (the values
 * pooled per tile like the keys: FP32 sum / count).  The pages do not print the attention
 * that consumes the pooled values; this is the cube-level attention of the VSA design:
 *   v     : [B][H][S][D] FP16, pooled like q and k (same prefix, cubes and counts)
 *   o_coarse: FP32 [B][H][(S-prefix)/block][D]: for query cube i,
 *           o_coarse[i] = sum_j softmax_j(scale * qm_i . km_j) vm_j over ALL key cubes j
 *           (qm, km, vm the FP32 cube means; FP32 scores, softmax and accumulation).
 *   idx and every other argument as for vsa_select_blocks; scale finite, > 0.
 *   Workspace: vsa_select_coarse_workspace_size() (vsa_select_blocks' plus the pooled values).
 * The gate that mixes o_coarse into the fine output is the caller's (see vsa_sparse_fwd).
 */
size_t vsa_select_coarse_workspace_size(int B, int H, int S, int D, int block);
int vsa_select_blocks_coarse(const void* q, const void* k, const void* v, int B, int H, int S,
                             int D, int block, int topk, int prefix, const int32_t* cube_valid,
                             float scale, int32_t* idx, float* o_coarse, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * vsa_select_blocks for callers that cannot allocate device memory.  The pages
 * have no counterpart; this entry point exists for callers such as a plugin
 * whose host program fixed its memory at start-up and forbids later
 * allocations, code whose device memory is owned by a pool it cannot reach, or
 * a latency-critical loop where a cudaMalloc (which may synchronise the
 * device) is not acceptable.  It computes exactly what vsa_select_blocks
 * computes, with the scratch (vsa_select_workspace_size() bytes: the FP32
 * pooled cube means, their norms, one flag per query cube and the FP32 cube
 * scores) taken from a fixed array of GBATTN_NOALLOC_SCRATCH_BYTES (48 MiB +
 * 192 KiB) inside the library, which every GPU that loads the library keeps
 * until the process exits.
 *   - Sizes whose vsa_select_workspace_size() exceeds that array are rejected
 *     with GBATTN_ERR_WORKSPACE before anything is queued.  At D=128, block=64
 *     and S = 32768 (512 cubes per head) the limit is B*H <= 32, i.e.
 *     B*H*S <= 1,048,576 tokens x heads.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - The library allocates nothing here, and the caller does not allocate
 *     either: only inputs and outputs are passed.
 *   - All calls share the one array, which keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls whose GPU work overlaps in
 *     time on one device (for example on two streams) race on it: order them
 *     on one stream or synchronise between them.
 */
#define GBATTN_NOALLOC_SCRATCH_BYTES ((48u << 20) + (192u << 10))
int vsa_select_blocks_noalloc(const void* q, const void* k, int B, int H, int S, int D, int block,
                              int topk, int prefix, const int32_t* cube_valid, int32_t* idx,
                              void* stream);

/*
 * VSA block-sparse attention over the selected key cubes (the full VSA layout).
 * Cites: "Integrate H3 SM70 execution, metrics and VSA diagnostics", Purpose (top-k = 64,
 * prefix-dense queries, per-query video blocks, boundary handling); FastVideo compare view,
 * block_lists.py (two 64-token query halves against two 64-token key halves per 128x128
 * block, with a 4-bit quadrant mask, and per-tile valid counts).
 *   q, k, v, o : [B][H][S][D] FP16; tokens [0, prefix) are prefix tokens, tokens
 *   [prefix, S) the cube-major video tokens; idx: int32 [B][H][(S-prefix)/block][topk]
 *   strictly ascending per row; pairs: the query cubes each CTA takes two at a time
 *   (vsa_pair_query_cubes), or NULL for cubes 2p and 2p+1; cube_valid as for
 *   vsa_select_blocks (NULL: full cubes); lse optional [B][H][S].
 *   A prefix query attends densely to every prefix token and every real video token; a real
 *   video query in cube c attends exactly the real tokens of cubes idx[b][h][c][*]; a padding
 *   query slot gets O = 0, lse = -inf.  Padding slots of V must hold finite values (their
 *   weight is exactly zero).
 *   o_coarse, gate: both NULL, or the coarse branch ("learned compression" of the same VSA
 *   page): o_coarse FP32 [B][H][(S-prefix)/block][D] from vsa_select_blocks_coarse and gate
 *   FP16 [B][H][S][D] (the caller's learned gate); every real video token then gets
 *   O = O_fine + gate * o_coarse[its cube], elementwise, before the FP16 rounding (lse stays
 *   the fine branch's).  Prefix tokens and padding slots are unchanged.
 *   block == 64, D == 128, prefix % 128 == 0, (S - prefix) % block == 0,
 *   1 <= topk <= min((S-prefix)/block, 512), prefix/128 + ceil(cubes/2) <= 512.
 *   workspace: NULL, or vsa_sparse_workspace_size() bytes of device memory, 16-byte aligned,
 *   overlapping no other argument, that hold zeros before the first call using them.  The
 *   work items (query-cube pairs, prefix query tiles) are then handed to the GPU's persistent
 *   CTAs by a counter in it, whichever CTA is free first, and every call leaves it at zero
 *   again, an aborted one (GBATTN_DEV_WAIT_TIMEOUT) included.  Calls that may run at the
 *   same time (two streams, concurrent graph launches) need separate workspaces.  NULL:
 *   CTA c of the G persistent CTAs takes items c, c + G, c + 2G, ... (slower when the
 *   items' key lists differ in length).  Too small: GBATTN_ERR_WORKSPACE.
 */
int vsa_sparse_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                   const int32_t* pairs, int prefix, const int32_t* cube_valid,
                   const float* o_coarse, const void* gate, void* o, float* lse, int B, int H,
                   int S, int D, int block, int topk, float scale, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Bytes of vsa_sparse_fwd's optional workspace (16). */
size_t vsa_sparse_workspace_size(void);

/*
 * Pairs the video query cubes of every head for vsa_sparse_fwd, which runs two query cubes per
 * CTA over the union of their selections: cubes whose selections overlap more waste less.
 * Cites: FastVideo compare view, block_lists.py (two 64-token query halves per 128-row block).
 * Not a step of the method: the attention result does not depend on the pairing (up to the
 * summation order); it only changes how much work the union tiles carry.
 *   idx   : int32 [B][H][n_cubes][topk] from vsa_select_blocks.
 *   pairs : int32 [B][H][ceil(n_cubes/2)][2], every cube exactly once; the second entry of a
 *           pair is -1 for the one unpaired cube of an odd count.
 *   workspace: vsa_pair_workspace_size(B, H, n_cubes) bytes of device memory, 16-byte aligned,
 *           overlapping neither idx nor pairs (each cube's selection as a bitset and its 32 best
 *           partners); its contents need no initial value.  NULL or smaller: GBATTN_ERR_WORKSPACE.
 *   Each head is paired greedily: the two cubes whose selections share the most key cubes first
 *   (ties: the lower cube indices), then the most overlapping two of the cubes left, and so on;
 *   a lone cube of an odd count stays alone.  The pairs are listed longest union first (ties:
 *   the lower first cube), the order in which the sparse kernel hands out its items.
 *   n_cubes <= 1024, B * H <= 65535.  Three kernel launches.
 */
size_t vsa_pair_workspace_size(int B, int H, int n_cubes);
int vsa_pair_query_cubes(const int32_t* idx, int B, int H, int n_cubes, int topk, int32_t* pairs,
                         void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
