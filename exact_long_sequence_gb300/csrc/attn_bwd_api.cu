// C ABI of the exact-attention backward: argument checks, workspace layout,
// TMA descriptors and the three launches (statistics, gradients, dQ to bf16).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/exact_attn.h"
#include "api_common.h"
#include "attn_bwd_kernel.cuh"
#include "plan.h"

namespace elsattn {
namespace {

template <int D, bool CAUSAL>
int launch_bwd(DeviceState& dev, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p, int BH, cudaStream_t stream) {
    auto kernel = attn_bwd_kernel<D, CAUSAL>;
    bool& configured = dev.bwd_smem_configured[D == 128][CAUSAL];
    cudaError_t e;
    if (!configured) {
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdLayout<D>::kSmem)) !=
            cudaSuccess)
            return cuda_fail(e);
        configured = true;
    }
    kernel<<<BH * p.num_k_tiles, kBwdThreads, BwdLayout<D>::kSmem, stream>>>(tq, tk, tv, tdo, tdq, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace elsattn

using namespace elsattn;

extern "C" size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t padded = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + kBc - 1) / kBc * kBc);
    return align256(rows * d * 4) + 2 * align256(padded * 4);
}

extern "C" int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                        void* dQ, void* dK, void* dV, int B, int H, int N, int d, int causal, float scale,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
    if (st != ATTN_OK) return st;
    if (!dO || !dQ || !dK || !dV || !workspace) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(dO) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) || !aligned16(workspace))
        return ATTN_ERR_MISALIGNED;
    if (workspace_bytes < attn_bwd_workspace_bytes(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;

    const int BH = B * H;
    const size_t rows = static_cast<size_t>(BH) * N;
    const int nkt = (N + kBc - 1) / kBc;
    const int Np = nkt * kBc;
    const size_t padded = static_cast<size_t>(BH) * Np;
    float* dqacc = static_cast<float*>(workspace);
    float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * d * 4));
    float* lse2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dvec) + align256(padded * 4));
    CUtensorMap tq, tk, tv, tdo, tdq;
    if ((st = encode_rows_map(&tq, Q, BH, N, d, kBq)) != ATTN_OK ||
        (st = encode_rows_map(&tk, K, BH, N, d, kBc)) != ATTN_OK ||
        (st = encode_rows_map(&tv, V, BH, N, d, kBc)) != ATTN_OK ||
        (st = encode_rows_map(&tdo, dO, BH, N, d, kBq)) != ATTN_OK ||
        (st = encode_f32_rows_map(&tdq, dqacc, BH, N, d, kBq / 2)) != ATTN_OK)
        return st;

    // D_i = sum_c dO_ic O_ic and LSE_i * log2(e) on tile-padded rows; the dQ accumulator zeroed
    {
        const size_t threads = padded * (d / 8);
        const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
        const auto* o = static_cast<const __nv_bfloat16*>(O);
        const auto* g = static_cast<const __nv_bfloat16*>(dO);
        if (d == 64)
            attn_bwd_prep_kernel<64><<<blocks, 256, 0, stream>>>(o, g, LSE, dvec, lse2, dqacc, N, Np, padded, scale);
        else
            attn_bwd_prep_kernel<128><<<blocks, 256, 0, stream>>>(o, g, LSE, dvec, lse2, dqacc, N, Np, padded, scale);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    BwdParams p;
    p.dQacc = dqacc;
    p.lse2 = lse2;
    p.Dvec = dvec;
    p.dK = static_cast<__nv_bfloat16*>(dK);
    p.dV = static_cast<__nv_bfloat16*>(dV);
    p.error_word = dev->error_word;
    p.timeout_ns = kDefaultTimeoutNs;
    p.N = N;
    p.num_k_tiles = nkt;
    p.num_q_blocks = (N + kBq - 1) / kBq;
    p.Np = Np;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale = scale;
    if (d == 64)
        st = causal ? launch_bwd<64, true>(*dev, tq, tk, tv, tdo, tdq, p, BH, stream)
                    : launch_bwd<64, false>(*dev, tq, tk, tv, tdo, tdq, p, BH, stream);
    else
        st = causal ? launch_bwd<128, true>(*dev, tq, tk, tv, tdo, tdq, p, BH, stream)
                    : launch_bwd<128, false>(*dev, tq, tk, tv, tdo, tdq, p, BH, stream);
    if (st != ATTN_OK) return st;
    // dQ = bf16(accumulator)
    const size_t n4 = rows * d / 4;
    attn_bwd_post_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(
        dqacc, static_cast<__nv_bfloat16*>(dQ), n4);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
