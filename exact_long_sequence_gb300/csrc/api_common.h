// Host-side pieces shared by the library's entry points (forward, backward):
// per-device state, status bookkeeping, argument checks and TMA descriptors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/exact_attn.h"

namespace elsattn {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s for any single wait

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t* error_word = nullptr;  // 256-byte device block, first word = error code
    bool smem_configured[2][2][2] = {};                                   // forward <d == 128><causal><dynamic schedule>
    bool bwd_smem_configured[2][2] = {{false, false}, {false, false}};  // backward <d == 128><causal>
    bool fp8_smem_configured[2][2][2] = {};  // FP8 forward <causal><dynamic schedule><K/V segments>
};

// The cudaError_t of this thread's most recent ATTN_ERR_CUDA.
extern thread_local int g_last_cuda_error;

// Records `e` as this thread's last CUDA error and returns ATTN_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Looks up the driver's cuTensorMapEncodeTiled once per process.
int resolve_tensor_map_encoder();

// The current device's state, set up on first use (checks for sm_103,
// resolves the tensor-map encoder, allocates the error word).
int device_state(DeviceState** out);

// A bf16 tensor viewed as [BH][N][d] (d innermost), read by TMA in boxes of
// 64 columns x box_rows rows with the 128-byte swizzle the tcgen05
// descriptors expect.  Rows past N read as zero.
int encode_rows_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// An fp32 tensor viewed as [BH][N][d], written by TMA (reduce-add) in boxes of
// d columns x box_rows rows, unswizzled.  Rows past N are dropped.
int encode_f32_rows_map(CUtensorMap* map, void* base, int BH, int N, int d, int box_rows);

// A 3-D byte tensor (E4M3 codes) with extents {e0, e1, e2} (e0 innermost) and
// byte strides s1, s2 (multiples of 16), read by TMA in boxes of b0 x b1 with
// the 128-byte swizzle (b0 = 128).  Elements past an extent read as zero.
int encode_u8_map(CUtensorMap* map, const void* base, uint64_t e0, uint64_t e1, uint64_t e2, uint64_t s1,
                  uint64_t s2, uint32_t b0, uint32_t b1);

bool aligned16(const void* p);

// Shared argument checks of the forward and backward entry points.
int check_args(const void* Q, const void* K, const void* V, const void* O, const void* LSE, int B, int H, int N,
               int d, float scale);

}  // namespace elsattn
