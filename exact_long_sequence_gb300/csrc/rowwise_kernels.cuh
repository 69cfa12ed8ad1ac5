// Standalone streaming row operations for sm_103a: row softmax and layer
// normalisation of bf16 rows, the "Softmax streaming" and "LayerNorm
// streaming" that the outlook of "From Attention Graph to FlashAttention - A
// Memory-Centric Compilation Approach in AICF" (section 8) proposes as the next
// uses of the memory-centric transformation.
//
// Both are HBM-bound: the target is one read and one write of every element.
// A CTA owns a row (or, for long softmax rows, a segment of one).  Each thread
// loads all of its 16-byte chunks up front (the whole row is in flight), keeps
// them in registers, and folds them into running statistics in one pass:
//   softmax:   (m, l) = running maximum and sum of exp(x - m), with the sum
//              rescaled by exp(m_old - m_new) when the maximum grows (the
//              online-softmax recurrence of the "IO-Aware Algorithms" page);
//   LayerNorm: (n, mean, M2) merged chunk by chunk with the pairwise update of
//              the running mean and sum of squared deviations.
// The per-thread statistics are merged across the CTA with the same rules, and
// the row is written once from registers.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace elsattn {

constexpr int kRowThreadsMax = 512;
constexpr int kRowChunkElems = 8;                     // one 16-byte chunk of bf16
constexpr int kRowMaxChunks = 16;                     // chunks per thread in registers
constexpr int kFusedRowMax = kRowThreadsMax * kRowChunkElems * kRowMaxChunks;  // 65536 elements
constexpr int kSoftmaxSegment = 16384;                // segment of a long softmax row
constexpr float kLog2e = 1.4426950408889634f;

struct SoftmaxStat {
    float m;  // running maximum (log2 units: x * log2 e)
    float l;  // sum of 2^(x * log2 e - m)
};

__device__ __forceinline__ SoftmaxStat merge_softmax(SoftmaxStat a, SoftmaxStat b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.f};
    return {m, a.l * ex2_approx(a.m - m) + b.l * ex2_approx(b.m - m)};
}

struct MeanStat {
    float n;     // count
    float mean;  // running mean
    float m2;    // sum of squared deviations from the mean
};

__device__ __forceinline__ MeanStat merge_mean(MeanStat a, MeanStat b) {
    const float n = a.n + b.n;
    if (n == 0.f) return {0.f, 0.f, 0.f};
    const float delta = b.mean - a.mean;
    const float wb = b.n / n;
    return {n, fmaf(delta, wb, a.mean), a.m2 + b.m2 + delta * delta * a.n * wb};
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Merge one statistic per thread into a CTA-wide one, returned to every thread.
template <class Stat, class Merge>
__device__ __forceinline__ Stat block_merge(Stat s, Merge merge, Stat* smem) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Stat o;
        float* of = reinterpret_cast<float*>(&o);
        const float* sf = reinterpret_cast<const float*>(&s);
#pragma unroll
        for (int k = 0; k < static_cast<int>(sizeof(Stat) / 4); ++k) of[k] = __shfl_xor_sync(0xffffffffu, sf[k], off);
        s = merge(s, o);
    }
    if (lane == 0) smem[warp] = s;
    __syncthreads();
    if (warp == 0) {
        Stat t = smem[lane < nwarps ? lane : 0];
        if (lane >= nwarps) {  // identity elements for the missing warps
            float* tf = reinterpret_cast<float*>(&t);
            if constexpr (sizeof(Stat) == sizeof(SoftmaxStat)) {
                tf[0] = -INFINITY;
                tf[1] = 0.f;
            } else {
                tf[0] = tf[1] = tf[2] = 0.f;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Stat o;
            float* of = reinterpret_cast<float*>(&o);
            const float* tf = reinterpret_cast<const float*>(&t);
#pragma unroll
            for (int k = 0; k < static_cast<int>(sizeof(Stat) / 4); ++k) of[k] = __shfl_xor_sync(0xffffffffu, tf[k], off);
            t = merge(t, o);
        }
        if (lane == 0) smem[32] = t;
    }
    __syncthreads();
    return smem[32];
}

// Softmax statistics of a thread's chunks (chunk c covers elements 8 (tid + c T) ..
// +7 of the range; chunks at or past nvec are absent).
template <int CHUNKS>
__device__ __forceinline__ SoftmaxStat thread_softmax_stat(const uint4 (&v)[CHUNKS], int nvec) {
    SoftmaxStat s{-INFINITY, 0.f};
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        if (static_cast<int>(threadIdx.x) + c * static_cast<int>(blockDim.x) >= nvec) break;
        float f[8];
        bf16x8_to_float(v[c], f);
        float mc = f[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) mc = fmaxf(mc, f[k]);
        mc *= kLog2e;
        if (mc > s.m) {  // the maximum grew: rescale the running sum
            s.l = (s.m == -INFINITY) ? 0.f : s.l * ex2_approx(s.m - mc);
            s.m = mc;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) s.l += ex2_approx(fmaf(f[k], kLog2e, -s.m));
    }
    return s;
}

// Fused row softmax: one CTA per row of N (multiple of 8, at most kFusedRowMax) elements.
template <int CHUNKS>
__global__ void __launch_bounds__(kRowThreadsMax) softmax_rows_fused(const __nv_bfloat16* X, __nv_bfloat16* Y,
                                                                     int N) {
    __shared__ SoftmaxStat red[33];
    const size_t row = blockIdx.x;
    const int nvec = N / kRowChunkElems;
    const uint4* x = reinterpret_cast<const uint4*>(X + row * N);
    uint4 v[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx < nvec) v[c] = ld_stream(x + idx);
    }
    const SoftmaxStat s = block_merge(thread_softmax_stat<CHUNKS>(v, nvec), merge_softmax, red);
    const float inv_l = 1.f / s.l;
    uint4* y = reinterpret_cast<uint4*>(Y + row * N);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx >= nvec) break;
        float f[8];
        bf16x8_to_float(v[c], f);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16x2(ex2_approx(fmaf(f[2 * k], kLog2e, -s.m)) * inv_l,
                               ex2_approx(fmaf(f[2 * k + 1], kLog2e, -s.m)) * inv_l);
        st_stream(y + idx, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Long rows, pass 1: statistics of one segment; CTA b covers segment b % nseg of
// row b / nseg.
template <int CHUNKS>
__global__ void __launch_bounds__(kRowThreadsMax) softmax_rows_seg_stats(const __nv_bfloat16* X, int N, int nseg,
                                                                         SoftmaxStat* stats) {
    __shared__ SoftmaxStat red[33];
    const size_t row = blockIdx.x / nseg;
    const int seg = blockIdx.x % nseg;
    const int seg0 = seg * kSoftmaxSegment;
    const int nvec = min(kSoftmaxSegment, N - seg0) / kRowChunkElems;
    const uint4* x = reinterpret_cast<const uint4*>(X + row * N + seg0);
    uint4 v[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx < nvec) v[c] = ld_stream(x + idx);
    }
    const SoftmaxStat s = block_merge(thread_softmax_stat<CHUNKS>(v, nvec), merge_softmax, red);
    if (threadIdx.x == 0) stats[row * nseg + seg] = s;
}

// Long rows, pass 2: merge the row's segment statistics and write one segment
// (the same CTA numbering as pass 1).
template <int CHUNKS>
__global__ void __launch_bounds__(kRowThreadsMax) softmax_rows_seg_write(const __nv_bfloat16* X, __nv_bfloat16* Y,
                                                                         int N, int nseg, const SoftmaxStat* stats) {
    __shared__ SoftmaxStat red[33];
    const size_t row = blockIdx.x / nseg;
    const int seg0 = (blockIdx.x % nseg) * kSoftmaxSegment;
    const int nvec = min(kSoftmaxSegment, N - seg0) / kRowChunkElems;
    const uint4* x = reinterpret_cast<const uint4*>(X + row * N + seg0);
    uint4 v[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx < nvec) v[c] = ld_stream(x + idx);
    }
    SoftmaxStat s{-INFINITY, 0.f};
    for (int k = threadIdx.x; k < nseg; k += blockDim.x) s = merge_softmax(s, stats[row * nseg + k]);
    s = block_merge(s, merge_softmax, red);
    const float inv_l = 1.f / s.l;
    uint4* y = reinterpret_cast<uint4*>(Y + row * N + seg0);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx >= nvec) break;
        float f[8];
        bf16x8_to_float(v[c], f);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16x2(ex2_approx(fmaf(f[2 * k], kLog2e, -s.m)) * inv_l,
                               ex2_approx(fmaf(f[2 * k + 1], kLog2e, -s.m)) * inv_l);
        st_stream(y + idx, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Cluster primitives (thread-block clusters on sm_90 and later).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The (m, l) that CTA `rank` of the cluster keeps at the same shared-memory offset as `local`.
__device__ __forceinline__ SoftmaxStat ld_peer_stat(const SoftmaxStat* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    SoftmaxStat s;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(s.m), "=f"(s.l) : "r"(remote) : "memory");
    return s;
}

// Rows of up to kClusterMax segments of kFusedRowMax elements: a cluster of
// nseg CTAs per row (CTA b holds segment b % nseg of row b / nseg in registers).
// Each CTA publishes its segment's (m, l) in shared memory, the cluster
// synchronises, every CTA merges the nseg statistics read through distributed
// shared memory, and writes its segment: one read and one write per element.
// Measured on GB300, clusters beyond 4 CTAs (one CTA per SM each) lose to the
// two-pass segment path: the gang-scheduled SMs sit idle between rows.
constexpr int kClusterMax = 4;
template <int CHUNKS>
__global__ void __launch_bounds__(kRowThreadsMax) softmax_rows_cluster(const __nv_bfloat16* X, __nv_bfloat16* Y,
                                                                       int N, int nseg) {
    __shared__ SoftmaxStat red[33];
    __shared__ SoftmaxStat mine;
    const uint32_t rank = cluster_ctarank();
    const size_t row = blockIdx.x / nseg;
    const int seg0 = static_cast<int>(rank) * kFusedRowMax;
    const int nvec = min(kFusedRowMax, N - seg0) / kRowChunkElems;
    const uint4* x = reinterpret_cast<const uint4*>(X + row * N + seg0);
    uint4 v[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx < nvec) v[c] = ld_stream(x + idx);
    }
    const SoftmaxStat local = block_merge(thread_softmax_stat<CHUNKS>(v, nvec), merge_softmax, red);
    if (threadIdx.x == 0) mine = local;
    cluster_sync_all();  // every CTA's statistic is published
    SoftmaxStat s{-INFINITY, 0.f};
    if (threadIdx.x < 32) {
        if (threadIdx.x < static_cast<unsigned>(nseg)) s = ld_peer_stat(&mine, threadIdx.x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            SoftmaxStat o;
            o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
            o.l = __shfl_xor_sync(0xffffffffu, s.l, off);
            s = merge_softmax(s, o);
        }
        if (threadIdx.x == 0) red[32] = s;
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its statistic
    s = red[32];
    const float inv_l = 1.f / s.l;
    uint4* y = reinterpret_cast<uint4*>(Y + row * N + seg0);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx >= nvec) break;
        float f[8];
        bf16x8_to_float(v[c], f);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16x2(ex2_approx(fmaf(f[2 * k], kLog2e, -s.m)) * inv_l,
                               ex2_approx(fmaf(f[2 * k + 1], kLog2e, -s.m)) * inv_l);
        st_stream(y + idx, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Fused layer normalisation: one CTA per row of N (multiple of 8, at most
// kFusedRowMax) elements; gamma, beta bf16 [N] (read through L2, where every
// row's CTA finds them).
template <int CHUNKS>
__global__ void __launch_bounds__(kRowThreadsMax) layernorm_rows_fused(const __nv_bfloat16* X,
                                                                       const __nv_bfloat16* gamma,
                                                                       const __nv_bfloat16* beta,
                                                                       __nv_bfloat16* Y, int N, float eps) {
    __shared__ MeanStat red[33];
    const size_t row = blockIdx.x;
    const int nvec = N / kRowChunkElems;
    const uint4* x = reinterpret_cast<const uint4*>(X + row * N);
    uint4 v[CHUNKS];
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx < nvec) v[c] = ld_stream(x + idx);
    }
    MeanStat s{0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        if (static_cast<int>(threadIdx.x) + c * static_cast<int>(blockDim.x) >= nvec) break;
        float f[8];
        bf16x8_to_float(v[c], f);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) sum += f[k];
        const float mc = sum * 0.125f;
        float m2 = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) m2 = fmaf(f[k] - mc, f[k] - mc, m2);
        s = merge_mean(s, MeanStat{8.f, mc, m2});
    }
    s = block_merge(s, merge_mean, red);
    const float rstd = rsqrtf(s.m2 / static_cast<float>(N) + eps);
    const uint4* g = reinterpret_cast<const uint4*>(gamma);
    const uint4* b = reinterpret_cast<const uint4*>(beta);
    uint4* y = reinterpret_cast<uint4*>(Y + row * N);
#pragma unroll
    for (int c = 0; c < CHUNKS; ++c) {
        const int idx = threadIdx.x + c * blockDim.x;
        if (idx >= nvec) break;
        float f[8], gf[8], bf[8];
        bf16x8_to_float(v[c], f);
        bf16x8_to_float(__ldg(g + idx), gf);
        bf16x8_to_float(__ldg(b + idx), bf);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16x2(fmaf((f[2 * k] - s.mean) * rstd, gf[2 * k], bf[2 * k]),
                               fmaf((f[2 * k + 1] - s.mean) * rstd, gf[2 * k + 1], bf[2 * k + 1]));
        st_stream(y + idx, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

}  // namespace elsattn
