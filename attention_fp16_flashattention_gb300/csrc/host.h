// Host-side helpers shared by the entry points: per-device state, argument
// checks, TMA descriptor encoding and launch accounting.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#ifndef GBATTN_NVTX
#define GBATTN_NVTX 1
#endif
#if GBATTN_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#include "../../include/gbattn.h"

namespace gbattn {

struct DeviceState {
    int device = -1;
    int num_sms = 0;
    uint32_t* status = nullptr;   // device address of the status word
};

// State of the current device (SM count, status-word address), set up on
// first use.  Returns GBATTN_OK or GBATTN_ERR_CUDA.
int current_device(DeviceState* out);

uint64_t wait_limit_ns();
// Test hook of the bounded waits (gbattn_test_inject_fault): 0 normal, 1 nothing
// loaded, 2 loads stop mid-stream.
int fault_mode();
void count_launches(int n);

// Encode a 4-D FP16 tensor map over [B][H][S][D] heads with element strides
// (row, head, batch; D contiguous) and a box of box0 x box1 x 1 x 1 elements,
// 128-byte swizzle.  Returns GBATTN_OK or GBATTN_ERR_CUDA.
int encode_tmap_f16_4d(CUtensorMap* map, const void* base, uint64_t D, uint64_t S, uint64_t H,
                       uint64_t B, uint64_t row_stride, uint64_t head_stride, uint64_t batch_stride,
                       uint32_t box0, uint32_t box1);

// Element strides of a [B][H][S][D] tensor (D contiguous).
struct Strides {
    long long b, h, r;
};

// Strides from a caller's {batch, head, row} array (NULL: dense).  Rows must be
// at least D elements apart, every stride a multiple of 8 elements (16-byte
// rows) and below 2^38; a dimension of extent 1 may carry any stride (it is
// replaced by the row stride, never used to address).  `out_injective` asks
// for no two elements of the tensor to share an address (an output).
inline bool make_strides(const int64_t* s, int B, int H, int S, int D, bool out_injective,
                         Strides* out) {
    Strides t;
    if (!s) {
        t.r = D;
        t.h = static_cast<long long>(S) * D;
        t.b = static_cast<long long>(H) * S * D;
    } else {
        t.b = s[0];
        t.h = s[1];
        t.r = s[2];
    }
    if (S == 1) t.r = D;
    if (H == 1) t.h = t.r;
    if (B == 1) t.b = t.r;
    const long long lim = 1LL << 38;
    for (long long v : {t.b, t.h, t.r})
        if (v <= 0 || v % 8 != 0 || v >= lim) return false;
    if (t.r < D) return false;
    if (out_injective) {
        // sorted by stride, every stride must clear the span of the smaller ones
        struct Dim { long long n, st; } d[3] = {{S, t.r}, {H, t.h}, {B, t.b}};
        for (int i = 0; i < 3; ++i)
            for (int j = i + 1; j < 3; ++j)
                if (d[j].st < d[i].st) {
                    const Dim x = d[i];
                    d[i] = d[j];
                    d[j] = x;
                }
        long long span = D;
        for (int i = 0; i < 3; ++i) {
            if (d[i].n <= 1) continue;
            if (d[i].st < span) return false;
            span += d[i].st * (d[i].n - 1);
        }
    }
    *out = t;
    return true;
}

// Bytes from the first to one past the last element of a strided tensor.
inline size_t strided_bytes(const Strides& t, int B, int H, int S, int D) {
    return static_cast<size_t>((B - 1) * t.b + (H - 1) * t.h + (static_cast<long long>(S) - 1) * t.r + D) * 2;
}

// Encode a 4-D FP16 tensor map over additive-mask slices [batch][heads][sq][skv]
// (element strides stride_h, stride_b between slices; size-1 dimensions are
// shared) with a box of 64 keys x 32 rows and the 128-byte swizzle.  Returns
// GBATTN_OK or GBATTN_ERR_CUDA.
int encode_tmap_f16_mask(CUtensorMap* map, const void* base, uint64_t skv, uint64_t sq,
                         uint64_t heads, uint64_t batch, uint64_t stride_h, uint64_t stride_b);

// Encode a 3-D byte tensor map over paged rows [rows][hkv][D] (D bytes per
// row and head) with a box of 128 bytes x 1 head x box_rows rows and the
// 128-byte swizzle.  Returns GBATTN_OK or GBATTN_ERR_CUDA.
int encode_tmap_u8_pages(CUtensorMap* map, const void* base, uint64_t D, uint64_t hkv,
                         uint64_t rows, uint32_t box_rows);

// One NVTX range per C-ABI call (its name is the entry point's), so profiler
// timelines show which call queued which kernels.  NVTX v3 is header-only and
// costs a branch when no tool is attached; builds with GBATTN_NVTX=0 drop it.
struct CallRange {
#if GBATTN_NVTX
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
#else
    explicit CallRange(const char*) {}
#endif
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline bool finite_positive(float s) { return s > 0.0f && s <= 3.402823466e38f; }

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

}  // namespace gbattn
