// Library-wide entry points (version, status text, device status word, wait
// limit, launch counter) and the host helpers declared in host.h.
#include <atomic>
#include <mutex>

#include "host.h"

namespace gbattn {

// One status word per device; kernels OR gbattn_device_flag bits into it.
static __device__ uint32_t g_device_status;

namespace {
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit{2000000000ull};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
}  // namespace

int current_device(DeviceState* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GBATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (s.device < 0) {
        int sms = 0;
        void* addr = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return GBATTN_ERR_CUDA;
        }
        s.num_sms = sms;
        s.status = static_cast<uint32_t*>(addr);
        s.device = dev;
    }
    *out = s;
    return GBATTN_OK;
}

uint64_t wait_limit_ns() { return g_wait_limit.load(); }

namespace {
std::atomic<int> g_fault_mode{0};   // test hook, see gbattn_test_inject_fault
}
int fault_mode() { return g_fault_mode.load(); }
void count_launches(int n) { g_launches += static_cast<uint64_t>(n); }

namespace {
int load_encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return GBATTN_ERR_CUDA;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return GBATTN_OK;
}
}  // namespace

int encode_tmap_f16_4d(CUtensorMap* map, const void* base, uint64_t D, uint64_t S, uint64_t H,
                       uint64_t B, uint64_t row_stride, uint64_t head_stride, uint64_t batch_stride,
                       uint32_t box0, uint32_t box1) {
    if (load_encoder() != GBATTN_OK) return GBATTN_ERR_CUDA;
    cuuint64_t dims[4] = {D, S, H, B};
    cuuint64_t strides[3] = {row_stride * 2, head_stride * 2, batch_stride * 2};   // bytes
    cuuint32_t box[4] = {box0, box1, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int encode_tmap_f16_mask(CUtensorMap* map, const void* base, uint64_t skv, uint64_t sq,
                         uint64_t heads, uint64_t batch, uint64_t stride_h, uint64_t stride_b) {
    if (load_encoder() != GBATTN_OK) return GBATTN_ERR_CUDA;
    cuuint64_t dims[4] = {skv, sq, heads, batch};
    cuuint64_t strides[3] = {skv * 2, stride_h * 2, stride_b * 2};   // bytes, dims 1..3
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int encode_tmap_u8_pages(CUtensorMap* map, const void* base, uint64_t D, uint64_t hkv,
                         uint64_t rows, uint32_t box_rows) {
    if (load_encoder() != GBATTN_OK) return GBATTN_ERR_CUDA;
    cuuint64_t dims[3] = {D, hkv, rows};
    cuuint64_t strides[2] = {D, D * hkv};   // bytes, dims 1 and 2
    cuuint32_t box[3] = {128, 1, box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GBATTN_OK : GBATTN_ERR_CUDA;
}

}  // namespace gbattn

using namespace gbattn;

extern "C" int gbattn_version(void) { return 100; }   // 0.1.0

extern "C" const char* gbattn_status_string(int status) {
    switch (status) {
        case GBATTN_OK: return "ok";
        case GBATTN_ERR_NULL: return "a required pointer is NULL";
        case GBATTN_ERR_SHAPE: return "a size is out of range or inconsistent";
        case GBATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case GBATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case GBATTN_ERR_ALIAS: return "an output overlaps an input";
        case GBATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case GBATTN_ERR_CUDA: return "CUDA runtime error";
        case GBATTN_ERR_SCALE: return "scale must be finite and positive";
        default: return "unknown status";
    }
}

extern "C" int gbattn_device_status(void* stream, uint32_t* flags_out) {
    if (!flags_out) return GBATTN_ERR_NULL;
    DeviceState d;
    int rc = current_device(&d);
    if (rc != GBATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, d.status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemsetAsync(d.status, 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return GBATTN_ERR_CUDA;
    }
    *flags_out = host;
    return GBATTN_OK;
}

extern "C" int gbattn_set_wait_limit_ns(uint64_t limit_ns) {
    if (limit_ns == 0) return GBATTN_ERR_SHAPE;
    g_wait_limit = limit_ns;
    return GBATTN_OK;
}

extern "C" uint64_t gbattn_launch_count(void) { return g_launches.load(); }

extern "C" int gbattn_test_inject_fault(int mode) {
    if (mode < 0 || mode > 2) return GBATTN_ERR_SHAPE;
    g_fault_mode = mode;
    return GBATTN_OK;
}
