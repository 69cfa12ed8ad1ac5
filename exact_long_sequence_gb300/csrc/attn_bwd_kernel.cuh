// Exact-attention backward for sm_103a: gradients dQ, dK, dV of
// O = softmax(scale * Q K^T + mask) V for an upstream gradient dO.
//
// The "IO-Aware Algorithms" page notes that FlashAttention recomputes its
// activations in the backward pass instead of storing them; this kernel does
// the same: it never stores P.  With the forward's per-row log-sum-exp it
// recomputes P = exp(scale * q.k - LSE) tile by tile and applies
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  (D_i = sum_c dO_ic O_ic),
//     dQ = scale * dS K,  dK = scale * dS^T Q.
//
// One CTA owns one (batch, head) and one tile of 128 keys; K_j and V_j stay in
// shared memory while the query tiles Q_i, dO_i stream through a TMA ring.
// Per query tile the MMA warp issues, all on tcgen05 with fp32 accumulators in
// TMEM (the key index is the MMA's M dimension, one TMEM lane per key):
//     S^T  = K_j Q_i^T           (A = K_j, B = Q_i, both from shared memory)
//     dP^T = V_j dO_i^T          (A = V_j, B = dO_i)
//     dV  += P^T dO_i            (A = P^T bf16 in TMEM, B = dO_i)
//     dK  += dS^T Q_i            (A = dS^T bf16 in TMEM, B = Q_i)
//     dQ_i = dS K_j              (A = dS bf16 in shared memory, M = queries)
// The compute warpgroup (thread r = key row r) turns S^T into P^T and dP^T
// into dS^T (scale folded in), writes dS^T to TMEM and dS to shared memory,
// and adds the partial dQ_i into an fp32 accumulator in global memory.
//
// TMEM columns: [0,128) S^T, then P^T (first 64), then the dQ_i partial |
// [128,256) dP^T, then dS^T (first 64) | [256,256+d) dV | [256+d,256+2d) dK.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "plan.h"
#include "sm103_ptx.cuh"

namespace elsattn {

constexpr int kBwdThreads = 256;  // warp 0 TMA, warp 1 MMA, warps 4-7 compute
constexpr int kBwdStages = 2;     // Q_i + dO_i ring depth

struct BwdParams {
    float* dQacc;          // [BH, N, d] fp32, zeroed; receives scale * dS K
    const float* lse2;     // [BH, Np] LSE * log2(e) of the forward; +inf on the padding rows
    const float* Dvec;     // [BH, Np] D_i = sum_c dO_ic O_ic; 0 on the padding rows
    __nv_bfloat16* dK;     // [BH, N, d]
    __nv_bfloat16* dV;     // [BH, N, d]
    uint32_t* error_word;
    uint64_t timeout_ns;
    int N;
    int num_q_tiles;       // ceil(N / 128)
    int Np;                // num_q_tiles * 128: row stride of lse2 and Dvec
    float scale_log2;      // scale * log2(e)
    float scale;
};

template <int D>
struct BwdLayout {
    static constexpr int kTile = tile_bytes(D);          // one [128 x d] bf16 tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kTile;
    static constexpr int kRingOff = 2 * kTile;            // stage s: Q_i at +0, dO_i at +kTile
    static constexpr int kDsOff = kRingOff + kBwdStages * 2 * kTile;  // dS, [2 query blocks][128 keys][64]
    static constexpr int kDsBytes = 2 * 128 * 128;
    static constexpr int kBarOff = kDsOff + kDsBytes;
    // barriers
    static constexpr int kKvFull = 0;
    static constexpr int kQFull = 1;                      // [kBwdStages]
    static constexpr int kQEmpty = kQFull + kBwdStages;   // [kBwdStages]
    static constexpr int kSpFull = kQEmpty + kBwdStages;  // S^T and dP^T complete
    static constexpr int kPFull = kSpFull + 1;            // P^T in TMEM (4 warp arrivals)
    static constexpr int kDsFull = kPFull + 1;            // dS^T in TMEM, dS in shared memory (4)
    static constexpr int kDsEmpty = kDsFull + 1;          // dQ_i MMA done reading dS
    static constexpr int kDqFull = kDsEmpty + 1;          // dQ_i partial complete
    static constexpr int kStFree = kDqFull + 1;           // dQ_i partial read out (4)
    static constexpr int kKvDone = kStFree + 1;           // dK, dV accumulation complete
    static constexpr int kDrain = kKvDone + 1;
    static constexpr int kNumBars = kDrain + 1;
    static constexpr int kFlagsOff = kBarOff + kNumBars * 8;
    static constexpr int kBytes = kFlagsOff + 16;
    static constexpr int kSmem = kBytes + kSmemAlign;
    static_assert(kSmem <= kSmemLimit, "backward shared memory");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                const BwdParams p) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + L::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kFlagsOff);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kFlagsOff + 4);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtx ctx{abort_flag, p.error_word, p.timeout_ns};

    const int bh = blockIdx.x / p.num_q_tiles;     // key tiles per head == query tiles per head
    const int kt = blockIdx.x - bh * p.num_q_tiles;
    const int i_first = CAUSAL ? kt : 0;           // query tiles before the key tile see none of its keys
    const int n_iter = p.num_q_tiles - i_first;

    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        mbar_init(bar(L::kKvFull), 1);
        for (int s = 0; s < kBwdStages; ++s) {
            mbar_init(bar(L::kQFull + s), 1);
            mbar_init(bar(L::kQEmpty + s), 1);
        }
        mbar_init(bar(L::kSpFull), 1);
        mbar_init(bar(L::kPFull), 4);
        mbar_init(bar(L::kDsFull), 4);
        mbar_init(bar(L::kDsEmpty), 1);
        mbar_init(bar(L::kDqFull), 1);
        mbar_init(bar(L::kStFree), 4);
        mbar_init(bar(L::kKvDone), 1);
        mbar_init(bar(L::kDrain), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        bool ok = true;
        mbar_arrive_expect_tx(bar(L::kKvFull), 2 * L::kTile);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
            tma_load_3d(s_base + L::kKOff + b * 16384, &tmap_k, bar(L::kKvFull), b * 64, kt * kBc, bh);
            tma_load_3d(s_base + L::kVOff + b * 16384, &tmap_v, bar(L::kKvFull), b * 64, kt * kBc, bh);
        }
        int issued = 0;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int s = it % kBwdStages;
            ok = mbar_wait(bar(L::kQEmpty + s), ((it / kBwdStages) & 1) ^ 1, ctx);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(L::kQFull + s), 2 * L::kTile);
            const uint32_t dst = s_base + L::kRingOff + s * 2 * L::kTile;
            const int row = (i_first + it) * kBr;
#pragma unroll
            for (int b = 0; b < D / 64; ++b) {
                tma_load_3d(dst + b * 16384, &tmap_q, bar(L::kQFull + s), b * 64, row, bh);
                tma_load_3d(dst + L::kTile + b * 16384, &tmap_do, bar(L::kQFull + s), b * 64, row, bh);
            }
            issued = it + 1;
        }
        // Every issued copy lands before the CTA ends (bounded wait; also on abort).
        mbar_wait_drain(bar(L::kKvFull), 0, 50000000ull);
        for (int it = issued > kBwdStages ? issued - kBwdStages : 0; it < issued; ++it)
            mbar_wait_drain(bar(L::kQFull + it % kBwdStages), (it / kBwdStages) & 1, 50000000ull);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_nt = make_idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t id_tn = make_idesc_bf16_f32(128, D, false, true);      // dV, dK (A in TMEM)
        constexpr uint32_t id_mn = make_idesc_bf16_f32(128, D, true, true);       // dQ (A MN-major)
        const uint32_t t_st = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + D;
        const uint64_t dk_k = make_smem_desc_sw128(s_base + L::kKOff, 16, 1024);      // K_j, K-major
        const uint64_t dv_k = make_smem_desc_sw128(s_base + L::kVOff, 16, 1024);      // V_j, K-major
        const uint64_t dk_mn = make_smem_desc_sw128(s_base + L::kKOff, 16384, 1024);  // K_j, MN-major
        const uint64_t dds_mn = make_smem_desc_sw128(s_base + L::kDsOff, 16384, 1024);  // dS, MN-major
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvFull), 0, ctx));
        for (int it = 0; it < n_iter && ok; ++it) {
            const int s = it % kBwdStages;
            const uint32_t ph = it & 1;
            const uint32_t qbase = s_base + L::kRingOff + s * 2 * L::kTile;
            const uint64_t dq_k = make_smem_desc_sw128(qbase, 16, 1024);                     // Q_i, K-major
            const uint64_t ddo_k = make_smem_desc_sw128(qbase + L::kTile, 16, 1024);         // dO_i, K-major
            const uint64_t dq_mn = make_smem_desc_sw128(qbase, 16384, 1024);                 // Q_i, MN-major
            const uint64_t ddo_mn = make_smem_desc_sw128(qbase + L::kTile, 16384, 1024);     // dO_i, MN-major
            bool w = mbar_wait(bar(L::kQFull + s), (it / kBwdStages) & 1, ctx);
            w = w && mbar_wait(bar(L::kStFree), ph ^ 1u, ctx);  // previous dQ_i partial read out
            if (!(ok = __all_sync(0xffffffffu, w))) break;
            tc_fence_after_sync();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_ss(t_st, dk_k + off, dq_k + off, id_nt, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_ss(t_dp, dv_k + off, ddo_k + off, id_nt, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kSpFull));
            }
            __syncwarp();
            // dV += P^T dO_i once P^T is in TMEM
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kPFull), ph, ctx)))) break;
            tc_fence_after_sync();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(t_dv, t_st + kk * 8, ddo_mn + static_cast<uint64_t>((kk * 2048) >> 4), id_tn,
                           (it > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
            // dK += dS^T Q_i and dQ_i = dS K_j once dS is ready
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDsFull), ph, ctx)))) break;
            tc_fence_after_sync();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(t_dk, t_dp + kk * 8, dq_mn + static_cast<uint64_t>((kk * 2048) >> 4), id_tn,
                           (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(t_st, dds_mn + static_cast<uint64_t>((kk * 2048) >> 4),
                           dk_mn + static_cast<uint64_t>((kk * 2048) >> 4), id_mn, kk > 0 ? 1u : 0u);
                mma_commit(bar(L::kDqFull));
                mma_commit(bar(L::kDsEmpty));
                mma_commit(bar(L::kQEmpty + s));
                if (it == n_iter - 1) mma_commit(bar(L::kKvDone));
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(bar(L::kDrain));
        __syncwarp();
        mbar_wait_drain(bar(L::kDrain), 0, 1000000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute warpgroup
        // Every tcgen05.ld/st below is warp-aligned: all 32 lanes execute it,
        // whatever their row; only global stores and atomics are per-lane.
        // The warps never wait on one another, only on mbarriers.
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                 // key row in the tile (TMEM lane)
        const int key = kt * kBc + r;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t t_st = tmem + lane_addr, t_dp = tmem + lane_addr + 128;
        uint8_t* ds_s = smem + L::kDsOff;
        const float sl2 = p.scale_log2;
        const size_t head = static_cast<size_t>(bh) * p.N;
        const size_t stat_head = static_cast<size_t>(bh) * p.Np;
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int qt = i_first + it;
            const uint32_t ph = it & 1;
            const float* lse2 = p.lse2 + stat_head + static_cast<size_t>(qt) * kBr;   // this query tile's
            const float* dvec = p.Dvec + stat_head + static_cast<size_t>(qt) * kBr;   // statistics
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kSpFull), ph, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            // P^T = exp2(S^T * scale * log2e - LSE * log2e), masked, -> bf16 over S^T's first 64 columns
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t sv[32];
                tmem_ld32(t_st + c0, sv);
                float l[32];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(lse2 + c0 + c));
                    l[c] = t.x, l[c + 1] = t.y, l[c + 2] = t.z, l[c + 3] = t.w;
                }
                tmem_wait_ld(sv);
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const int q0 = qt * kBr + c0 + c;
                    float a = ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, -l[c]));
                    float b = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), sl2, -l[c + 1]));
                    if (key >= p.N || (CAUSAL && key > q0)) a = 0.f;
                    if (key >= p.N || (CAUSAL && key > q0 + 1)) b = 0.f;
                    pk[c / 2] = pack_bf16x2(a, b);
                }
                tmem_st16(t_st + c0 / 2, pk);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kPFull));
            __syncwarp();
            // dS = scale * P * (dP - D): dS^T -> TMEM (dP^T's first 64 columns),
            // dS -> shared memory (MN-major, 128-byte swizzled) for dQ_i = dS K_j.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDsEmpty), ph ^ 1u, ctx));
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t dv[32], pv[16];
                tmem_ld32(t_dp + c0, dv);
                tmem_ld16(t_st + c0 / 2, pv);
                float dd[32];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(dvec + c0 + c));
                    dd[c] = t.x, dd[c + 1] = t.y, dd[c + 2] = t.z, dd[c + 3] = t.w;
                }
                tmem_wait_ld(dv);
                tmem_wait_ld16(pv);
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float pa = __uint_as_float(pv[c / 2] << 16), pb = __uint_as_float(pv[c / 2] & 0xffff0000u);
                    const float a = p.scale * pa * (__uint_as_float(dv[c]) - dd[c]);
                    const float b = p.scale * pb * (__uint_as_float(dv[c + 1]) - dd[c + 1]);
                    pk[c / 2] = pack_bf16x2(a, b);
                }
                tmem_st16(t_dp + c0 / 2, pk);
                // queries c0..c0+31 of key row r: four 16-byte chunks of block c0/64
                uint8_t* rowp = ds_s + (c0 >> 6) * 16384 + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = ((c0 & 63) >> 3) + q;
                    *reinterpret_cast<uint4*>(rowp + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();  // dS written by threads, read by the tensor core
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kDsFull));
            __syncwarp();
            // dQ_i partial (TMEM lane = query row) -> fp32 atomics into the accumulator
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDqFull), ph, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            const int qrow = qt * kBr + r;
            const bool row_ok = qrow < p.N;
            float* dqrow = p.dQacc + (head + (row_ok ? qrow : 0)) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(t_st + c0, v);
                tmem_wait_ld(v);
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        atomicAdd(reinterpret_cast<float4*>(dqrow + c0 + c),
                                  make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                              __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])));
                }
                __syncwarp();
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kStFree));
            __syncwarp();
        }
        // dK, dV of this key tile -> bf16 (all lanes read TMEM; rows past N store nothing)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvDone), 0, ctx));
        if (ok) {
            tc_fence_after_sync();
            const bool key_ok = key < p.N;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const uint32_t src = tmem + lane_addr + 256 + (g == 0 ? D : 0);  // dK, then dV
                uint4* dst = reinterpret_cast<uint4*>((g == 0 ? p.dK : p.dV) + (head + (key_ok ? key : 0)) * D);
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(src + c0, v);
                    tmem_wait_ld(v);
                    uint32_t wv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) wv[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    if (key_ok) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[c0 / 8 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                    }
                    __syncwarp();
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Per-row statistics of the backward, on rows padded to whole query tiles
// (Np = ceil(N / 128) * 128 per (batch, head)):
//     D_i = sum_c dO_ic O_ic (fp32), lse2_i = LSE_i * log2(e);
// padding rows get D = 0 and lse2 = +inf (so that exp2(. - lse2) = 0 there).
// Also zeroes the dQ accumulator.  D/8 threads per padded row, 8 elements each.
template <int D>
__global__ void attn_bwd_prep_kernel(const __nv_bfloat16* O, const __nv_bfloat16* dO, const float* LSE,
                                     float* Dvec, float* lse2, float* dQacc, int N, int Np, size_t padded_rows) {
    constexpr int kTpr = D / 8;
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t prow = tid / kTpr;
    const int part = static_cast<int>(tid % kTpr);
    const size_t bh = prow / static_cast<size_t>(Np);
    const int n = static_cast<int>(prow - bh * static_cast<size_t>(Np));
    const bool live = prow < padded_rows && n < N;
    const size_t row = bh * static_cast<size_t>(N) + n;
    float acc = 0.f;
    if (live) {
        const uint4 o = reinterpret_cast<const uint4*>(O + row * D)[part];
        const uint4 g = reinterpret_cast<const uint4*>(dO + row * D)[part];
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc = fmaf(__uint_as_float(ow[k] << 16), __uint_as_float(gw[k] << 16), acc);
            acc = fmaf(__uint_as_float(ow[k] & 0xffff0000u), __uint_as_float(gw[k] & 0xffff0000u), acc);
        }
        reinterpret_cast<float4*>(dQacc + row * D)[2 * part] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(dQacc + row * D)[2 * part + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (prow < padded_rows && part == 0) {
        Dvec[prow] = acc;
        lse2[prow] = live ? LSE[row] * 1.4426950408889634f : INFINITY;
    }
}

// dQ = bf16(dQ accumulator)
__global__ void attn_bwd_post_kernel(const float* dQacc, __nv_bfloat16* dQ, size_t n4) {
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n4) {
        const float4 v = reinterpret_cast<const float4*>(dQacc)[i];
        reinterpret_cast<uint2*>(dQ)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
}

}  // namespace elsattn
