// Host-side helpers shared by the entry points: per-device state, argument
// checks, TMA descriptor encoding and launch accounting.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

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
void count_launches(int n);

// Encode a 3-D FP16 tensor map over a dense [d2][d1][d0] array with a box of
// box0 x box1 x 1 elements and the 128-byte swizzle.  Returns GBATTN_OK or
// GBATTN_ERR_CUDA.
int encode_tmap_f16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint32_t box0, uint32_t box1);

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
