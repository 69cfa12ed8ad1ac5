// Host-side pieces shared by the library's entry points: per-device state,
// status bookkeeping, argument checks and TMA descriptors.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/exact_attn.h"
#include "api_common.h"

namespace elsattn {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return ATTN_ERR_CUDA;
}

namespace {
std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

int resolve_tensor_map_encoder() {
    static std::mutex m;
    std::lock_guard<std::mutex> lock(m);
    if (g_encode) return ATTN_OK;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return ATTN_OK;
}

int device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return ATTN_ERR_NO_DEVICE;
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (s.cc_major != 10 || s.cc_minor != 3) return ATTN_ERR_UNSUPPORTED;  // built for sm_103a only
        const int st = resolve_tensor_map_encoder();
        if (st != ATTN_OK) return st;
        void* w = nullptr;
        if ((e = cudaMalloc(&w, 256)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemset(w, 0, 256)) != cudaSuccess) {
            cudaFree(w);
            return cuda_fail(e);
        }
        s.error_word = static_cast<uint32_t*>(w);
        s.ready = true;
    }
    *out = &s;
    return ATTN_OK;
}

int encode_rows_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return ATTN_OK;
}

int encode_f32_rows_map(CUtensorMap* map, void* base, int BH, int N, int d, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return ATTN_OK;
}

int encode_u8_map(CUtensorMap* map, const void* base, uint64_t e0, uint64_t e1, uint64_t e2, uint64_t s1,
                  uint64_t s2, uint32_t b0, uint32_t b1) {
    cuuint64_t dims[3] = {e0, e1, e2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_args(const void* Q, const void* K, const void* V, const void* O, const void* LSE, int B, int H, int N,
               int d, float scale) {
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * N >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return ATTN_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

}  // namespace elsattn
