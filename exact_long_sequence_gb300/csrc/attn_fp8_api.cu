// C ABI of the FP8 (E4M3) exact-attention forward: argument checks, the
// transposed copy of V, TMA descriptors and the launch of the FP8
// instantiation of the forward kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/exact_attn.h"
#include "api_common.h"
#include "attn_fwd_fp8_kernel.cuh"
#include "attn_fwd_kernel.cuh"
#include "plan.h"
#include "split_policy.h"

extern "C" int attn_plan_impl(int B, int H, int N, int d, int causal, int num_sms, attn_plan_t* out);

namespace elsattn {
namespace {

constexpr int kFp8D = 128;  // the E4M3 tiles are one 128-byte swizzle row wide

// Row pitch (bytes) of the transposed V: a multiple of 16, as TMA strides must be.
size_t vt_pitch(int N) { return (static_cast<size_t>(N) + 15) / 16 * 16; }

// Vt[bh][c][j] = V[bh][j][c] for one (batch, head) and one tile of 128 keys,
// through a padded shared-memory tile.  Keys past N are written as zero up to
// the padded pitch.
__global__ void __launch_bounds__(256) transpose_v_e4m3(const uint8_t* V, uint8_t* Vt, int N, size_t pitch) {
    __shared__ __align__(16) uint8_t tile[128][kFp8D + 4];
    const int bh = blockIdx.y;
    const int j0 = blockIdx.x * 128;
    const uint8_t* src = V + static_cast<size_t>(bh) * N * kFp8D;
    for (int i = threadIdx.x; i < 128 * (kFp8D / 16); i += blockDim.x) {
        const int r = i / (kFp8D / 16), c16 = (i % (kFp8D / 16)) * 16;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j0 + r < N) v = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(j0 + r) * kFp8D + c16);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&tile[r][c16]);
        dst[0] = v.x;
        dst[1] = v.y;
        dst[2] = v.z;
        dst[3] = v.w;
    }
    __syncthreads();
    uint8_t* out = Vt + static_cast<size_t>(bh) * kFp8D * pitch;
    for (int i = threadIdx.x; i < kFp8D * 8; i += blockDim.x) {
        const int c = i / 8, k16 = (i % 8) * 16;
        if (j0 + k16 >= N) continue;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = static_cast<uint32_t>(tile[k16 + 4 * q][c]) | (static_cast<uint32_t>(tile[k16 + 4 * q + 1][c]) << 8) |
                   (static_cast<uint32_t>(tile[k16 + 4 * q + 2][c]) << 16) |
                   (static_cast<uint32_t>(tile[k16 + 4 * q + 3][c]) << 24);
        *reinterpret_cast<uint4*>(out + static_cast<size_t>(c) * pitch + j0 + k16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <bool CAUSAL, bool DYN = false, bool SPLIT = false>
int launch_fp8(DeviceState& dev, const attn_plan_t& plan, const CUtensorMap& tq, const CUtensorMap& tk,
               const CUtensorMap& tvt, const FwdParams& p, cudaStream_t stream) {
    if constexpr (!SPLIT) {
        // split launches take the instantiation with K/V segments
        if (p.kv_split > 1) return launch_fp8<CAUSAL, DYN, true>(dev, plan, tq, tk, tvt, p, stream);
    }
    if constexpr (CAUSAL && !DYN) {
        // causal launches with a schedule counter take the dynamic instantiation
        if (p.sched_counter != nullptr) return launch_fp8<CAUSAL, true, SPLIT>(dev, plan, tq, tk, tvt, p, stream);
    }
    auto kernel = attn_fwd_fp8_kernel<CAUSAL, DYN, SPLIT>;
    constexpr int smem = Fp8Layout::kSmem;
    bool& configured = dev.fp8_smem_configured[CAUSAL][DYN][SPLIT];
    cudaError_t e;
    if (!configured) {
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail(e);
        configured = true;
    }
    // every CTA starts with item blockIdx.x: the grid never exceeds the items
    const int grid = p.num_items < dev.num_sms ? p.num_items : dev.num_sms;
    if constexpr (DYN) {
        // a programmatic dependent of the counter's zeroing kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(static_cast<unsigned>(plan.threads));
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tvt, p)) != cudaSuccess) return cuda_fail(e);
    } else {
        kernel<<<grid, plan.threads, smem, stream>>>(tq, tk, tvt, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    }
    if (p.kv_split > 1) {
        // the segments' merge, as a programmatic dependent launch (see attn_api.cu)
        const int rows = p.split_units * 2 * kBr;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((rows + kCombineRowsPerCta - 1) / kCombineRowsPerCta));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        auto combine = p.kv_split == 2 ? attn_fwd_combine_kernel<kFp8D, CAUSAL, 2>
                       : p.kv_split == 3 ? attn_fwd_combine_kernel<kFp8D, CAUSAL, 3> : attn_fwd_combine_kernel<kFp8D, CAUSAL, 4>;
        if ((e = cudaLaunchKernelEx(&cfg, combine, p)) != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
}

bool positive_finite(float x) { return std::isfinite(x) && x > 0.f; }

}  // namespace
}  // namespace elsattn

using namespace elsattn;

// Workspace: the transposed V codes, a 256-byte block for the schedule
// counter, then the split units' partial O and LSE, each part 256-aligned.
size_t vt_bytes(int B, int H, int N, int d) {
    const size_t b = static_cast<size_t>(B) * H * d * vt_pitch(N);
    return (b + 255) & ~static_cast<size_t>(255);
}

namespace {

// The work schedule on the current device; no split without a usable device.
KvSplit fp8_schedule(int B, int H, int N, int d, int causal) {
    DeviceState* dev = nullptr;
    attn_plan_t plan;
    if (device_state(&dev) != ATTN_OK || attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan) != ATTN_OK)
        return KvSplit{1, 0, 0, false};
    return choose_kv_split(plan, dev->num_sms, B * H, N, causal);
}

}  // namespace

extern "C" size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    size_t b = vt_bytes(B, H, N, d) + kCounterBlock;
    if (d == kFp8D && static_cast<long long>(B) * H * N < (1ll << 31)) {
        // the larger of the two masks' splits, so one size serves both
        for (int causal = 0; causal < 2; ++causal) {
            const KvSplit s = fp8_schedule(B, H, N, d, causal);
            const size_t parts = split_part_o_bytes(s, d) + split_part_lse_bytes(s);
            if (vt_bytes(B, H, N, d) + kCounterBlock + parts > b) b = vt_bytes(B, H, N, d) + kCounterBlock + parts;
        }
    }
    return b;
}

extern "C" int attn_fwd_fp8(const void* Q8, const void* K8, const void* V8, void* O, float* LSE, int B, int H, int N,
                            int d, int causal, float scale, float q_scale, float k_scale, float v_scale,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int st = check_args(Q8, K8, V8, O, LSE, B, H, N, d, scale);
    if (st != ATTN_OK) return st;
    // The FP8 kernel tracks the row maximum of the scaled scores assuming a positive factor.
    if (!positive_finite(scale) || !positive_finite(q_scale) || !positive_finite(k_scale) || !positive_finite(v_scale))
        return ATTN_ERR_INVALID_ARG;
    if (d != kFp8D) return ATTN_ERR_UNSUPPORTED;
    if (!workspace) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
    if (workspace_bytes < attn_fwd_fp8_workspace_bytes(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    attn_plan_t plan;
    if ((st = attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan)) != ATTN_OK) return st;

    const int BH = B * H;
    const size_t pitch = vt_pitch(N);
    uint8_t* vt = static_cast<uint8_t*>(workspace);
    {
        const dim3 grid((N + 127) / 128, BH);
        transpose_v_e4m3<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(V8), vt, N, pitch);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    CUtensorMap tq, tk, tvt;
    const uint64_t rows = static_cast<uint64_t>(N), bh = static_cast<uint64_t>(BH);
    if ((st = encode_u8_map(&tq, Q8, kFp8D, rows, bh, kFp8D, rows * kFp8D, kFp8D, kBr)) != ATTN_OK ||
        (st = encode_u8_map(&tk, K8, kFp8D, rows, bh, kFp8D, rows * kFp8D, kFp8D, kBc)) != ATTN_OK ||
        (st = encode_u8_map(&tvt, vt, rows, kFp8D, bh, pitch, pitch * kFp8D, kBc, kFp8D)) != ATTN_OK)
        return st;

    FwdParams p;
    p.O = static_cast<__nv_bfloat16*>(O);
    p.LSE = LSE;
    p.error_word = dev->error_word;
    p.timeout_ns = kDefaultTimeoutNs;
    p.N = N;
    p.BH = BH;
    p.num_q_tiles = (N + kBr - 1) / kBr;
    p.num_kv_tiles = (N + kBc - 1) / kBc;
    p.num_pairs = (p.num_q_tiles + 1) / 2;
    p.num_units = plan.num_units;
    p.heads_per_group = plan.heads_per_group;
    p.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
    p.out_scale = v_scale;
    // The bf16 forward's work schedule: K/V segments for launches with fewer
    // units than SMs or a partial last wave, dynamic claiming for causal ones.
    const KvSplit split = choose_kv_split(plan, dev->num_sms, BH, N, causal);
    uint8_t* counter_block = vt + vt_bytes(B, H, N, d);
    p.kv_split = split.segs;
    p.split_first = split.first;
    p.split_units = split.units;
    p.num_items = plan.num_units + split.units * (split.segs - 1);
    p.part_o = split.segs > 1 ? reinterpret_cast<float*>(counter_block + kCounterBlock) : nullptr;
    p.part_lse =
        split.segs > 1 ? reinterpret_cast<float*>(counter_block + kCounterBlock + split_part_o_bytes(split, d)) : nullptr;
    p.sched_counter = nullptr;
    if (split.dynamic) {
        // CTAs claim items, heaviest first, from a counter zeroed on the stream by a
        // kernel the attention launch depends on programmatically (see attn_api.cu)
        int* counter = reinterpret_cast<int*>(counter_block);
        zero_sched_counter_kernel<<<1, 1, 0, stream>>>(counter);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        p.sched_counter = counter;
    }
    return causal ? launch_fp8<true>(*dev, plan, tq, tk, tvt, p, stream)
                  : launch_fp8<false>(*dev, plan, tq, tk, tvt, p, stream);
}
