// C ABI of the standalone streaming row operations (row softmax, layer
// normalisation): argument checks, the choice of chunks per thread, launches.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/exact_attn.h"
#include "api_common.h"
#include "rowwise_kernels.cuh"

namespace elsattn {
namespace {

// Chunks per thread and threads per CTA for a row of `nvec` 16-byte chunks:
// about four chunks (64 bytes) per thread keep enough loads in flight per SM;
// longer rows use up to kRowMaxChunks chunks on kRowThreadsMax threads.
void row_shape(int nvec, int* chunks, int* threads) {
    int t = (nvec + 3) / 4;
    t = (t + 31) / 32 * 32;
    if (t < 32) t = 32;
    if (t > kRowThreadsMax) t = kRowThreadsMax;
    int c = 1;
    while (c < kRowMaxChunks && c * t < nvec) c *= 2;
    *chunks = c;
    *threads = t;
}

#define ELS_DISPATCH_CHUNKS(chunks, LAUNCH) \
    switch (chunks) {                        \
        case 1: LAUNCH(1); break;            \
        case 2: LAUNCH(2); break;            \
        case 4: LAUNCH(4); break;            \
        case 8: LAUNCH(8); break;            \
        default: LAUNCH(16); break;          \
    }

int row_args(const void* X, const void* Y, int64_t R, int N) {
    if (!X || !Y || R < 1 || N < 1 || R >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
    if (N % kRowChunkElems != 0) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(Y)) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

// The current device must be the sm_103 the kernels are built for.
int row_device() {
    DeviceState* dev = nullptr;
    return device_state(&dev);
}

int launched() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Rows of nseg <= kClusterMax segments of kFusedRowMax elements as one cluster of
// nseg CTAs per row.  Sets *used = false (and launches nothing) when the device
// cannot hold such a cluster.
int launch_softmax_cluster(const __nv_bfloat16* x, __nv_bfloat16* y, int64_t R, int N, int nseg, cudaStream_t stream,
                           bool* used) {
    auto kernel = softmax_rows_cluster<kRowMaxChunks>;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(R * nseg));
    cfg.blockDim = dim3(kRowThreadsMax);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(nseg);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg)) != cudaSuccess) return cuda_fail(e);
    *used = clusters > 0;
    if (!*used) return ATTN_OK;
    if ((e = cudaLaunchKernelEx(&cfg, kernel, x, y, N, nseg)) != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

}  // namespace
}  // namespace elsattn

using namespace elsattn;

extern "C" size_t attn_softmax_rows_workspace_bytes(int64_t R, int N) {
    if (R < 1 || N <= kFusedRowMax) return 0;
    const int64_t nseg = (N + kSoftmaxSegment - 1) / kSoftmaxSegment;
    return static_cast<size_t>(R * nseg) * sizeof(SoftmaxStat);
}

extern "C" int attn_softmax_rows(const void* X, void* Y, int64_t R, int N, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    int st = row_args(X, Y, R, N);
    if (st != ATTN_OK) return st;
    const int64_t nseg = (N + kSoftmaxSegment - 1) / kSoftmaxSegment;
    if (N > kFusedRowMax) {
        if (!workspace || workspace_bytes < attn_softmax_rows_workspace_bytes(R, N)) return ATTN_ERR_INVALID_ARG;
        if (R * nseg >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return ATTN_ERR_MISALIGNED;
    }
    if ((st = row_device()) != ATTN_OK) return st;
    const auto* x = static_cast<const __nv_bfloat16*>(X);
    auto* y = static_cast<__nv_bfloat16*>(Y);
    const int64_t nclu = (N + kFusedRowMax - 1) / kFusedRowMax;
    if (N > kFusedRowMax && nclu <= kClusterMax && R * nclu < (1LL << 31)) {
        bool used = false;
        if ((st = launch_softmax_cluster(x, y, R, N, static_cast<int>(nclu), stream, &used)) != ATTN_OK)
            return st;
        if (used) return ATTN_OK;
    }
    if (N <= kFusedRowMax) {
        int chunks, threads;
        row_shape(N / kRowChunkElems, &chunks, &threads);
#define ELS_LAUNCH(C) softmax_rows_fused<C><<<static_cast<unsigned>(R), threads, 0, stream>>>(x, y, N)
        ELS_DISPATCH_CHUNKS(chunks, ELS_LAUNCH)
#undef ELS_LAUNCH
        return launched();
    }
    auto* stats = static_cast<SoftmaxStat*>(workspace);
    int chunks, threads;
    row_shape(kSoftmaxSegment / kRowChunkElems, &chunks, &threads);
    const unsigned grid = static_cast<unsigned>(R * nseg);
#define ELS_LAUNCH(C) softmax_rows_seg_stats<C><<<grid, threads, 0, stream>>>(x, N, static_cast<int>(nseg), stats)
    ELS_DISPATCH_CHUNKS(chunks, ELS_LAUNCH)
#undef ELS_LAUNCH
    if ((st = launched()) != ATTN_OK) return st;
#define ELS_LAUNCH(C) softmax_rows_seg_write<C><<<grid, threads, 0, stream>>>(x, y, N, static_cast<int>(nseg), stats)
    ELS_DISPATCH_CHUNKS(chunks, ELS_LAUNCH)
#undef ELS_LAUNCH
    return launched();
}

extern "C" int attn_layernorm_rows(const void* X, const void* gamma, const void* beta, void* Y, int64_t R, int N,
                                   float eps, cudaStream_t stream) {
    int st = row_args(X, Y, R, N);
    if (st != ATTN_OK) return st;
    if (!gamma || !beta || !(std::isfinite(eps) && eps >= 0.f)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(gamma) || !aligned16(beta)) return ATTN_ERR_MISALIGNED;
    if (N > kFusedRowMax) return ATTN_ERR_UNSUPPORTED;
    if ((st = row_device()) != ATTN_OK) return st;
    int chunks, threads;
    row_shape(N / kRowChunkElems, &chunks, &threads);
    const auto* x = static_cast<const __nv_bfloat16*>(X);
    const auto* g = static_cast<const __nv_bfloat16*>(gamma);
    const auto* b = static_cast<const __nv_bfloat16*>(beta);
    auto* y = static_cast<__nv_bfloat16*>(Y);
#define ELS_LAUNCH(C) layernorm_rows_fused<C><<<static_cast<unsigned>(R), threads, 0, stream>>>(x, g, b, y, N, eps)
    ELS_DISPATCH_CHUNKS(chunks, ELS_LAUNCH)
#undef ELS_LAUNCH
    return launched();
}
