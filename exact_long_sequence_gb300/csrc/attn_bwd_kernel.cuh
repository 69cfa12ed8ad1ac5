// Exact-attention backward for sm_103a: gradients dQ, dK, dV of
// O = softmax(scale * Q K^T + mask) V for an upstream gradient dO.
//
// The "IO-Aware Algorithms" page notes that FlashAttention recomputes its
// activations in the backward pass instead of storing them; this kernel does
// the same: it never stores P.  With the forward's per-row log-sum-exp it
// recomputes P = exp(scale * q.k - LSE) block by block and applies
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  (D_i = sum_c dO_ic O_ic),
//     dQ = scale * dS K,  dK = scale * dS^T Q.
//
// One CTA owns one (batch, head) and one tile of 128 keys; K_j and V_j stay in
// shared memory while blocks of 64 queries (Q_i, dO_i) stream through a TMA
// ring.  Per query block the MMA warp issues, on tcgen05 with fp32
// accumulators in TMEM:
//     S^T  = K_j Q_i^T     M = 128 keys, N = 64 queries   (A, B in shared memory)
//     dP^T = V_j dO_i^T    M = 128 keys, N = 64 queries
//     dV  += P^T dO_i      M = 128 keys, N = d            (A = P^T bf16 in TMEM)
//     dK  += dS^T Q_i      M = 128 keys, N = d            (A = dS^T bf16 in TMEM)
//     dQ_i^T = K_j^T dS^T  M = d (padded to 128), N = 64  (A = K_j read transposed)
// S^T and dP^T are double-buffered in TMEM, so the tensor core computes the
// scores of block i+2 while the compute warps still work on block i.  dQ is
// produced transposed (TMEM lane = head-dim column); the readout warps copy it
// to registers, release the TMEM columns, stage it in shared memory as
// [query][d] fp32 and add it to the fp32 accumulator in global memory with one
// TMA bulk reduce per block.  The per-query LSE and D of a block arrive by TMA
// with its Q_i and dO_i.
//
// Warp roles: 0 TMA producer, 1 MMA issuer, 4-7 and 12-15 P and dS (thread =
// key row; each warpgroup takes half of the block's queries), 8-11 dQ readout
// (thread = head-dim column); at the end 4-7 and 12-15 write dV, 8-11 dK.
//
// TMEM columns: [0, d) dV | [d, 2d) dK | buffer b at 2d + 128 b:
//   [0, 64) S^T, then P^T (bf16) of queries 0-31 over [0, 16) and of queries
//   32-63 over [32, 48);  [64, 128) dP^T, then dS^T likewise, then dQ^T of the
//   block (fp32).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "plan.h"
#include "sm103_bulk.cuh"
#include "sm103_ptx.cuh"

namespace elsattn {

constexpr int kBwdThreads = 512;  // warps 0 TMA, 1 MMA, 4-7 and 12-15 P/dS, 8-11 dQ readout
constexpr int kBq = 64;           // queries per block
// Q_i + dO_i ring depth: three blocks are in flight (i, i+1 and the i+2 whose
// scores are computed ahead), so three stages suffice.
constexpr int bwd_stages(int d) { return d == 128 ? 3 : 4; }

struct BwdParams {
    float* dQacc;          // [BH, N, d] fp32, zeroed; receives scale * dS K
    const float* lse2;     // [BH, Np] -LSE * log2(e) of the forward; -inf on the padding rows
    const float* Dvec;     // [BH, Np] -scale * D_i, D_i = sum_c dO_ic O_ic; 0 on the padding rows
    __nv_bfloat16* dK;     // [BH, N, d]
    __nv_bfloat16* dV;     // [BH, N, d]
    uint32_t* error_word;
    uint64_t timeout_ns;
    int N;
    int num_k_tiles;       // ceil(N / 128): CTAs per (batch, head)
    int num_q_blocks;      // ceil(N / 64)
    int Np;                // num_k_tiles * 128: row stride of lse2 and Dvec
    float scale_log2;      // scale * log2(e)
    float scale;
};

template <int D>
struct BwdLayout {
    static constexpr int kBwdStages = bwd_stages(D);
    static constexpr int kKvTile = 128 * D * 2;             // K_j or V_j: [128 keys x d] bf16
    static constexpr int kQTile = kBq * D * 2;              // Q_i or dO_i: [64 queries x d] bf16
    static constexpr int kKvBlock = 128 * 128;              // one 64-column block of a K/V tile
    static constexpr int kQBlock = kBq * 128;               // one 64-column block of a Q/dO tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKvTile;
    static constexpr int kRingOff = 2 * kKvTile;            // stage s: Q_i at +0, dO_i at +kQTile
    static constexpr int kStageBytes = 2 * kQTile;
    static constexpr int kDsOff = kRingOff + kBwdStages * kStageBytes;  // [2][128 keys][64 queries] bf16
    static constexpr int kDsBuf = 128 * kBq * 2;
    static constexpr int kDqOff = kDsOff + 2 * kDsBuf;     // [2 halves][32 queries][d] fp32: dQ_i staged
    static constexpr int kStatOff = kDqOff + kBq * D * 4;  // [stage][lse2 x 64, D x 64] fp32
    static constexpr int kStatBytes = 2 * kBq * 4;
    static constexpr int kBarOff = kStatOff + kBwdStages * kStatBytes;
    // barriers
    static constexpr int kKvFull = 0;
    static constexpr int kQFull = 1;                         // [kBwdStages]
    static constexpr int kQEmpty = kQFull + kBwdStages;      // [kBwdStages]
    static constexpr int kSpFull = kQEmpty + kBwdStages;     // [2] S^T and dP^T of a block complete
    static constexpr int kPFull = kSpFull + 2;               // [2] P^T in TMEM (8 warp arrivals)
    static constexpr int kDsFull = kPFull + 2;               // [2] dS^T in TMEM, dS in shared memory (8)
    static constexpr int kDsEmpty = kDsFull + 2;             // [2] dQ^T MMA done reading dS
    static constexpr int kDqFull = kDsEmpty + 2;             // [2] dQ^T of a block complete
    static constexpr int kDqFree = kDqFull + 2;              // [2] dQ^T read out of TMEM (4)
    static constexpr int kStFull = kDqFree + 2;              // [2] a half of dQ_i staged (4)
    static constexpr int kStEmpty = kStFull + 2;             // [2] the reduce has read that half
    static constexpr int kKvDone = kStEmpty + 2;             // dK, dV accumulation complete
    static constexpr int kDrain = kKvDone + 1;
    static constexpr int kNumBars = kDrain + 1;
    static constexpr int kFlagsOff = kBarOff + kNumBars * 8;
    static constexpr int kBytes = kFlagsOff + 16;
    static constexpr int kSmem = kBytes + kSmemAlign;
    static_assert(kSmem <= kSmemLimit, "backward shared memory");
    static_assert(2 * kSmem > 233472, "one CTA per SM: each allocates all TMEM columns");
    static_assert(kRingOff % 1024 == 0 && kStageBytes % 1024 == 0 && kQTile % 1024 == 0 && kDsOff % 1024 == 0,
                  "swizzle atoms are 1024-byte aligned");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                const __grid_constant__ CUtensorMap tmap_dq, const BwdParams p) {
    using L = BwdLayout<D>;
    constexpr int kBwdStages = L::kBwdStages;
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

    const int bh = blockIdx.x / p.num_k_tiles;
    const int kt = blockIdx.x - bh * p.num_k_tiles;
    const int i_first = CAUSAL ? 2 * kt : 0;     // query blocks before the key tile see none of its keys
    const int n_iter = p.num_q_blocks - i_first;  // >= 1: the diagonal block is always visited

    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        mbar_init(bar(L::kKvFull), 1);
        for (int s = 0; s < kBwdStages; ++s) {
            mbar_init(bar(L::kQFull + s), 1);
            mbar_init(bar(L::kQEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::kSpFull + b), 1);
            mbar_init(bar(L::kPFull + b), 8);
            mbar_init(bar(L::kDsFull + b), 8);
            mbar_init(bar(L::kDsEmpty + b), 1);
            mbar_init(bar(L::kDqFull + b), 1);
            mbar_init(bar(L::kDqFree + b), 4);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(L::kStFull + h), 4);
            mbar_init(bar(L::kStEmpty + h), 1);
        }
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
        mbar_arrive_expect_tx(bar(L::kKvFull), 2 * L::kKvTile);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
            tma_load_3d(s_base + L::kKOff + b * L::kKvBlock, &tmap_k, bar(L::kKvFull), b * 64, kt * kBc, bh);
            tma_load_3d(s_base + L::kVOff + b * L::kKvBlock, &tmap_v, bar(L::kKvFull), b * 64, kt * kBc, bh);
        }
        int issued = 0;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int s = it % kBwdStages;
            ok = mbar_wait(bar(L::kQEmpty + s), ((it / kBwdStages) & 1) ^ 1, ctx);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(L::kQFull + s), L::kStageBytes + L::kStatBytes);
            const uint32_t dst = s_base + L::kRingOff + s * L::kStageBytes;
            const int row = (i_first + it) * kBq;
            const size_t stat = static_cast<size_t>(bh) * p.Np + row;
            const uint32_t sdst = s_base + L::kStatOff + s * L::kStatBytes;
            bulk_load(sdst, p.lse2 + stat, kBq * 4, bar(L::kQFull + s));
            bulk_load(sdst + kBq * 4, p.Dvec + stat, kBq * 4, bar(L::kQFull + s));
#pragma unroll
            for (int b = 0; b < D / 64; ++b) {
                tma_load_3d(dst + b * L::kQBlock, &tmap_q, bar(L::kQFull + s), b * 64, row, bh);
                tma_load_3d(dst + L::kQTile + b * L::kQBlock, &tmap_do, bar(L::kQFull + s), b * 64, row, bh);
            }
            issued = it + 1;
        }
        // Every issued copy lands before the CTA ends (bounded wait; also on abort).
        mbar_wait_drain(bar(L::kKvFull), 0, 50000000ull);
        for (int it = issued > kBwdStages ? issued - kBwdStages : 0; it < issued; ++it)
            mbar_wait_drain(bar(L::kQFull + it % kBwdStages), (it / kBwdStages) & 1, 50000000ull);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_s = make_idesc_bf16_f32(128, kBq, false, false);  // S^T, dP^T
        constexpr uint32_t id_acc = make_idesc_bf16_f32(128, D, false, true);   // dV, dK (A in TMEM)
        constexpr uint32_t id_dq = make_idesc_bf16_f32(128, kBq, true, true);   // dQ^T (A, B MN-major)
        const uint32_t t_dv = tmem, t_dk = tmem + D;
        const uint64_t dk_k = make_smem_desc_sw128(s_base + L::kKOff, 16, 1024);            // K_j, K-major
        const uint64_t dv_k = make_smem_desc_sw128(s_base + L::kVOff, 16, 1024);            // V_j, K-major
        // K_j^T as A of dQ^T: d-blocks of 64 are L::kKvBlock apart.  For d = 64 the
        // second block (rows 64..127 of dQ^T) reads V_j: those lanes are never used.
        const uint64_t dkt_mn = make_smem_desc_sw128(s_base + L::kKOff, L::kKvBlock, 1024);
        auto ring = [&](int i) { return s_base + L::kRingOff + static_cast<uint32_t>(i % kBwdStages) * L::kStageBytes; };
        auto kstep_a = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * L::kKvBlock + (kk & 3) * 32) >> 4); };
        auto kstep_b = [](int kk) { return static_cast<uint64_t>(((kk >> 2) * L::kQBlock + (kk & 3) * 32) >> 4); };
        constexpr uint64_t kRows16 = (16 * 128) >> 4;  // 16 rows of an MN-major operand
        // TMEM column of the bf16 A operand (P^T or dS^T) for queries 16 kk .. 16 kk + 15:
        // each compute warpgroup packs its 32 queries over the first 16 of its own 32 columns.
        auto a_col = [](int kk) { return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8); };

        // S^T and dP^T of block i into buffer i & 1.  The S^T half is free: P^T of
        // block i - 2 was read by dV (issued earlier) and by the dS pass (its
        // DsFull was awaited).  The dP^T half holds dQ^T of block i - 2 until the
        // readout warps release it.
        auto issue_sdp = [&](int i) -> bool {
            const int b = i & 1;
            const uint32_t q = ring(i);
            bool w = mbar_wait(bar(L::kQFull + i % kBwdStages), (i / kBwdStages) & 1, ctx);
            if (!__all_sync(0xffffffffu, w)) return false;
            tc_fence_after_sync();
            const uint32_t t_s = tmem + 2 * D + 128 * b;
            const uint64_t dq_k = make_smem_desc_sw128(q, 16, 1024);
            const uint64_t ddo_k = make_smem_desc_sw128(q + L::kQTile, 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(t_s, dk_k + kstep_a(kk), dq_k + kstep_b(kk), id_s, kk > 0 ? 1u : 0u);
            }
            __syncwarp();
            if (i >= 2) {
                w = mbar_wait(bar(L::kDqFree + b), ((i - 2) >> 1) & 1, ctx);
                if (!__all_sync(0xffffffffu, w)) return false;
                tc_fence_after_sync();
            }
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(t_s + 64, dv_k + kstep_a(kk), ddo_k + kstep_b(kk), id_s, kk > 0 ? 1u : 0u);
                mma_commit(bar(L::kSpFull + b));
            }
            __syncwarp();
            return true;
        };

        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvFull), 0, ctx));
        if (ok) ok = issue_sdp(0);
        if (ok && n_iter > 1) ok = issue_sdp(1);
        for (int it = 0; it < n_iter && ok; ++it) {
            const int b = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const uint32_t q = ring(it);
            const uint32_t t_s = tmem + 2 * D + 128 * b;
            const uint64_t dq_mn = make_smem_desc_sw128(q, L::kQBlock, 1024);               // Q_i, MN-major
            const uint64_t ddo_mn = make_smem_desc_sw128(q + L::kQTile, L::kQBlock, 1024);  // dO_i, MN-major
            const uint64_t dds_mn = make_smem_desc_sw128(s_base + L::kDsOff + b * L::kDsBuf, L::kDsBuf, 1024);
            // dV += P^T dO_i once P^T is in TMEM
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kPFull + b), ph, ctx)))) break;
            tc_fence_after_sync();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kBq / 16; ++kk)
                    mma_ts(t_dv, t_s + a_col(kk), ddo_mn + kk * kRows16, id_acc, (it > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
            // dK += dS^T Q_i and dQ_i^T = K_j^T dS^T once dS is ready
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDsFull + b), ph, ctx)))) break;
            tc_fence_after_sync();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kBq / 16; ++kk)
                    mma_ts(t_dk, t_s + 64 + a_col(kk), dq_mn + kk * kRows16, id_acc, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kBc / 16; ++kk)
                    mma_ss(t_s + 64, dkt_mn + kk * kRows16, dds_mn + kk * kRows16, id_dq, kk > 0 ? 1u : 0u);
                mma_commit(bar(L::kDqFull + b));
                mma_commit(bar(L::kDsEmpty + b));
                mma_commit(bar(L::kQEmpty + it % kBwdStages));
                if (it == n_iter - 1) mma_commit(bar(L::kKvDone));
            }
            __syncwarp();
            if (it + 2 < n_iter) ok = issue_sdp(it + 2);
        }
        if (elect_one()) mma_commit(bar(L::kDrain));
        __syncwarp();
        mbar_wait_drain(bar(L::kDrain), 0, 1000000000ull);
    } else if ((warp >= 4 && warp < 8) || warp >= 12) {
        // (x0, x1) = (a0 * b + c0, a1 * b + c1) and (x0, x1) *= (m0, m1) on packed fp32 pairs
        auto ffma2c = [](float& x0, float& x1, float a0, float a1, float b, float c0, float c1) {
            uint64_t rr;
            asm("{\n\t.reg .b64 pa, pb, pc;\n\tmov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %3};\n\t"
                "mov.b64 pc, {%4, %5};\n\tfma.rn.f32x2 %0, pa, pb, pc;\n\t}"
                : "=l"(rr) : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(rr));
        };
        auto fmul2 = [](float& x0, float& x1, float m0, float m1) {
            uint64_t rr;
            asm("{\n\t.reg .b64 pa, pb;\n\tmov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %4};\n\tmul.rn.f32x2 %0, pa, pb;\n\t}"
                : "=l"(rr) : "f"(x0), "f"(x1), "f"(m0), "f"(m1));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(rr));
        };
        // ------------------------------------------------------------ P and dS
        // Thread r = key row r of the tile (TMEM lane r).  Warps 4-7 take the
        // block's queries 0-31, warps 12-15 queries 32-63.  Every tcgen05.ld/st
        // is executed by all 32 lanes of the warp; only stores are per-lane.
        const int quad = warp & 3;
        const int c0 = warp >= 12 ? 32 : 0;  // this warpgroup's query columns
        const int r = quad * 32 + lane;
        const int key = kt * kBc + r;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const float sl2 = p.scale_log2;
        const size_t head = static_cast<size_t>(bh) * p.N;
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int b = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int q0 = (i_first + it) * kBq;
            const uint32_t t_s = tmem + lane_addr + 2 * D + 128 * b, t_dp = t_s + 64;
            const int s = it % kBwdStages;
            const float* lse2 = reinterpret_cast<const float*>(smem + L::kStatOff + s * L::kStatBytes);
            const float* dvec = lse2 + kBq;
            // S^T of the block, and the block's statistics (they land with Q_i)
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kSpFull + b), ph, ctx) &&
                                             mbar_wait(bar(L::kQFull + s), (it / kBwdStages) & 1, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            // P^T = exp2(S^T * scale * log2e - LSE * log2e), masked -> bf16 over S^T's first 32 columns
            // (the statistics hold -LSE * log2e and -scale * D)
            {
                uint32_t sv[32];
                tmem_ld32(t_s + c0, sv);
                float l[32];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(lse2 + c0 + c);
                    l[c] = t.x, l[c + 1] = t.y, l[c + 2] = t.z, l[c + 3] = t.w;
                }
                tmem_wait_ld(sv);
                uint32_t pk[16];
                // masking is needed only in tiles that hold a padding key or cross the diagonal
                const bool need_mask = __any_sync(0xffffffffu, key >= p.N || (CAUSAL && key > q0 + c0));
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const int qa = q0 + c0 + c;
                        float a, bb;
                        ffma2c(a, bb, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sl2, l[c], l[c + 1]);
                        a = ex2_approx(a);
                        bb = ex2_approx(bb);
                        if (key >= p.N || (CAUSAL && key > qa)) a = 0.f;
                        if (key >= p.N || (CAUSAL && key > qa + 1)) bb = 0.f;
                        pk[c / 2] = pack_bf16x2(a, bb);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float a, bb;
                        ffma2c(a, bb, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sl2, l[c], l[c + 1]);
                        pk[c / 2] = pack_bf16x2(ex2_approx(a), ex2_approx(bb));
                    }
                }
                tmem_st16(t_s + c0, pk);  // over this warpgroup's own S^T columns
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kPFull + b));
            __syncwarp();
            // dS = scale * P * (dP - D): dS^T -> TMEM over dP^T's first 32 columns,
            // dS -> shared memory ([key][query], 128-byte swizzled) for dQ^T.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDsEmpty + b), ph ^ 1u, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            uint8_t* ds_row = smem + L::kDsOff + b * L::kDsBuf + r * 128;
            {
                uint32_t dv[32], pv[16];
                tmem_ld32(t_dp + c0, dv);
                tmem_ld16(t_s + c0, pv);
                float dd[32];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(dvec + c0 + c);
                    dd[c] = t.x, dd[c + 1] = t.y, dd[c + 2] = t.z, dd[c + 3] = t.w;
                }
                tmem_wait_ld(dv);
                tmem_wait_ld16(pv);
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float pa = __uint_as_float(pv[c / 2] << 16), pb = __uint_as_float(pv[c / 2] & 0xffff0000u);
                    float a, bb;  // scale * dP - scale * D, then times P
                    ffma2c(a, bb, __uint_as_float(dv[c]), __uint_as_float(dv[c + 1]), p.scale, dd[c], dd[c + 1]);
                    fmul2(a, bb, pa, pb);
                    pk[c / 2] = pack_bf16x2(a, bb);
                }
                tmem_st16(t_dp + c0, pk);  // over this warpgroup's own dP^T columns
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = (c0 >> 3) + q;  // 16-byte chunk of the 128-byte row
                    *reinterpret_cast<uint4*>(ds_row + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();  // dS written by threads, read by the tensor core
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kDsFull + b));
            __syncwarp();
        }
        // dV of this key tile -> bf16, half of its columns per warpgroup (all lanes
        // read TMEM; rows past N store nothing)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvDone), 0, ctx));
        if (ok) {
            tc_fence_after_sync();
            const bool key_ok = key < p.N;
            uint4* dst = reinterpret_cast<uint4*>(p.dV + (head + (key_ok ? key : 0)) * D);
#pragma unroll 1
            for (int cv = (c0 ? D / 2 : 0); cv < (c0 ? D : D / 2); cv += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_addr + cv, v);
                tmem_wait_ld(v);
                uint32_t wv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) wv[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                if (key_ok) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[cv / 8 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                }
                __syncwarp();
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ dQ readout
        // Thread r = head-dim column r of dQ_i^T (TMEM lane r).  The block's dQ_i is
        // staged in shared memory as two halves of [32 queries][d] fp32 (a warp
        // writes 32 consecutive floats of a row per store), and each half is added
        // to the accumulator by one TMA reduce while the other half is staged.
        // Rows past N fall outside the tensor and are dropped.  One thread issues
        // the reduces; it releases a half once the reduce issued before the
        // current one has read its data.
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const size_t head = static_cast<size_t>(bh) * p.N;
        const bool col_ok = r < D;  // warp-uniform: d is a multiple of 32
        const bool issuer = warp == 8 && lane == 0;
        constexpr int kHalf = kBq / 2;
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
            const int b = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int q0 = (i_first + it) * kBq;
            const uint32_t t_dq = tmem + lane_addr + 2 * D + 128 * b + 64;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kDqFull + b), ph, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t v[2][32];
            tmem_ld32(t_dq, v[0]);
            tmem_ld32(t_dq + 32, v[1]);
            tmem_wait_ld(v[0]);
            tmem_wait_ld(v[1]);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kDqFree + b));
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2 && ok; ++h) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kStEmpty + h), (it & 1) ^ 1u, ctx));
                if (!ok) break;
                float* stage = reinterpret_cast<float*>(smem + L::kDqOff + h * kHalf * D * 4);
                if (col_ok) {
#pragma unroll
                    for (int c = 0; c < kHalf; ++c) stage[c * D + r] = __uint_as_float(v[h][c]);
                }
                fence_proxy_async_smem();  // staged by threads, read by the TMA unit
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kStFull + h));
                bool w = true;
                if (issuer) {
                    w = mbar_wait(bar(L::kStFull + h), it & 1, ctx);
                    if (w) {
                        tma_reduce_add_3d(&tmap_dq, s_base + L::kDqOff + h * kHalf * D * 4, 0, q0 + h * kHalf, bh);
                        bulk_commit_group();
                    }
                    // the reduce issued before this one has read its half: release it
                    bulk_wait_group_read<1>();
                    if (h == 1) mbar_arrive(bar(L::kStEmpty + 0));
                    else if (it > 0) mbar_arrive(bar(L::kStEmpty + 1));
                }
                ok = __all_sync(0xffffffffu, w);
            }
        }
        if (issuer) bulk_wait_group<0>();  // every reduce has landed before the CTA ends
        // dK of this key tile -> bf16
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvDone), 0, ctx));
        if (ok) {
            tc_fence_after_sync();
            const int key = kt * kBc + r;
            const bool key_ok = key < p.N;
            uint4* dst = reinterpret_cast<uint4*>(p.dK + (head + (key_ok ? key : 0)) * D);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_addr + D + c0, v);
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

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Per-row statistics of the backward, on rows padded to whole key tiles
// (Np = ceil(N / 128) * 128 per (batch, head)):
//     D_i = sum_c dO_ic O_ic (fp32), stored as Dvec_i = -scale * D_i, and
//     lse2_i = -LSE_i * log2(e),
// negated so that the gradient kernel adds them inside packed FMAs; padding rows
// get Dvec = 0 and lse2 = -inf (so that exp2(. + lse2) = 0 there).
// Also zeroes the dQ accumulator.  D/8 threads per padded row, 8 elements each.
template <int D>
__global__ void attn_bwd_prep_kernel(const __nv_bfloat16* O, const __nv_bfloat16* dO, const float* LSE,
                                     float* Dvec, float* lse2, float* dQacc, int N, int Np, size_t padded_rows, float scale) {
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
        Dvec[prow] = -scale * acc;
        lse2[prow] = live ? -(LSE[row] * 1.4426950408889634f) : -INFINITY;
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
