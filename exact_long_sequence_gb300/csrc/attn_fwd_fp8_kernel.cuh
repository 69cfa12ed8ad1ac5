// FP8 (E4M3) exact-attention forward for sm_103a with the scores issued ahead
// of the softmax.
//
// Same computation, units, roles and TMEM accumulators as the bf16 forward
// (attn_fwd_kernel.cuh): two query tiles per unit, S_t = Q_t K_j^T and
// O_t += P_t V_j on tcgen05 (kind::f8f6f4, K = 32 per instruction), the online
// softmax in two warpgroups.  What differs is where P lives and therefore the
// order of the MMAs:
//   - P_t (E4M3, 128 bytes per query row) is written to shared memory, into
//     one of two buffers per tile, in the 128-byte swizzled layout of a
//     K-major A operand; O_t += P_t V_j reads it from there (SS form).
//   - S_t's TMEM columns are then read only by the softmax, so S_t(j+1) is
//     issued as soon as the softmax has loaded S_t(j) into registers (barrier
//     SCons), not after O_t += P_t(j) V_j.  The softmax of iteration j+1 finds
//     its scores ready when it finishes iteration j, and the two softmax
//     warpgroups, not the MMA chain, set the pace.
// In the bf16 kernel P (32 KB per tile) stays in TMEM: in shared memory its
// operand reads would make the tensor core shared-memory-bound.
//
// The O rescale of a row whose maximum moved must see O_t with exactly the
// products of the earlier iterations: the softmax waits (barrier ODone) for
// the previous O_t += P V to complete before it rescales, which it does before
// releasing the first half of the current P.
//
// TMEM columns: [0,128) S0 | [128,256) S1 | [256,384) O0 | [384,512) O1.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"
#include "plan.h"
#include "sm103_ptx.cuh"

namespace elsattn {

constexpr int kFp8Stages = 8;  // K/V ring depth (tiles of 16 KB)

// Scores out of every 32 of a row whose exp2 is evaluated on the FMA pipes
// (exp2_poly.h) instead of the special-function unit: 0, 2, 4, ..., 16.
#ifndef ELS_FP8_EXP2_POLY_PER32
#define ELS_FP8_EXP2_POLY_PER32 0
#endif
constexpr int kFp8PolyPer32 = ELS_FP8_EXP2_POLY_PER32;
static_assert(kFp8PolyPer32 >= 0 && kFp8PolyPer32 <= 16 && kFp8PolyPer32 % 2 == 0, "FP8 exp2 offload: even, <= 16");

// P is stored as E4M3, whose largest finite value is 448 (2^8.81).  The
// stale-max rule shared with the bf16 kernel keeps every term of P at most
// 2^kRescaleLog2, so that bound must stay inside E4M3's range.
static_assert(kRescaleLog2 <= 8.8f, "E4M3 P would saturate: the FP8 kernel needs its own threshold");

// A bounded mbarrier wait without a function call, for the one wait that sits
// where a row's 128 scores are live in registers (a call there forces them to
// local memory).  Same semantics as mbar_wait.
__device__ __forceinline__ bool mbar_wait_inline(uint32_t bar, uint32_t parity, const WaitCtx& ctx) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*ctx.abort_flag) return false;
            if (global_timer_ns() - t0 > ctx.timeout_ns) {
                atomicCAS(ctx.error_word, 0u, static_cast<uint32_t>(kDevTimeout));
                *ctx.abort_flag = 1u;
                return false;
            }
        }
    }
}

struct Fp8Layout {
    static constexpr int kTile = 128 * 128;                // [128 rows][128 bytes]
    static constexpr int kQOff = 0;                        // [2] Q tiles
    static constexpr int kRingOff = 2 * kTile;             // [kFp8Stages] K_j or V_j^T tiles
    static constexpr int kPOff = kRingOff + kFp8Stages * kTile;  // [2 tiles][2 buffers] P tiles
    static constexpr int kBarOff = kPOff + 4 * kTile;
    // barriers
    static constexpr int kKvFull = 0;
    static constexpr int kKvEmpty = kKvFull + kFp8Stages;
    static constexpr int kQFull = kKvEmpty + kFp8Stages;   // [2]
    static constexpr int kQEmpty = kQFull + 2;             // [2]
    static constexpr int kSFull = kQEmpty + 2;             // [2] S_t computed
    static constexpr int kSCons = kSFull + 2;              // [2] S_t loaded by the softmax (128)
    // P barriers are per (tile, buffer): with S issued ahead, the softmax can
    // finish P(k+1) before the MMA warp has waited for P(k), and a single
    // barrier would then be two phases ahead of its waiter.  Buffer b's
    // barriers cannot run ahead: P(k+2) needs PFree(b), i.e. the product of P(k).
    static constexpr int kPHalf = kSCons + 2;              // [2 tiles][2 buffers] keys 0-63 stored, O_t rescaled (128)
    static constexpr int kPFull = kPHalf + 4;              // [2 tiles][2 buffers] keys 64-127 stored (128)
    static constexpr int kPFree = kPFull + 4;              // [2 tiles][2 buffers] O_t += P V done reading the buffer
    static constexpr int kODone = kPFree + 4;              // [2] the latest O_t += P V completed
    static constexpr int kOFull = kODone + 2;              // [2]
    static constexpr int kOEmpty = kOFull + 2;             // [2] (128)
    static constexpr int kDrain = kOEmpty + 2;             // [2] one per MMA warp
    static constexpr int kItemFull = kDrain + 2;           // [kItemRing] the slot holds the next item index
    static constexpr int kItemEmpty = kItemFull + kItemRing;  // [kItemRing] both MMA warps + 8 softmax warps read it
    static constexpr int kNumBars = kItemEmpty + kItemRing;
    static constexpr int kFlagsOff = kBarOff + kNumBars * 8;  // tmem base slot, abort flag, item indices
    static constexpr int kItemOff = kFlagsOff + 8;             // [kItemRing] int
    static constexpr int kBytes = kFlagsOff + 16;
    static constexpr int kSmem = kBytes + kSmemAlign;
    static_assert(kSmem <= kSmemLimit, "FP8 forward shared memory");
    static_assert(2 * kSmem > 233472, "one CTA per SM: it allocates all TMEM columns");
};

// Work items as in the bf16 kernel (decode_item): whole units, or K/V segments
// of the units the launch splits, whose partial results the combine kernel
// merges.  DYN: the dynamic item schedule (p.sched_counter is set): each CTA
// starts with item blockIdx.x and then claims the next unclaimed item from the
// counter, the producer passing each claimed item to the MMA and softmax warps
// through a two-slot ring in shared memory (-1 after the last).  Without it,
// the static stride.
// A work item: with SPLIT, decode_item's unit or K/V segment; without it the
// whole unit w (the instantiation that unsplit launches run).
template <bool CAUSAL, bool SPLIT>
__device__ __forceinline__ ItemInfo fp8_item(int w, const FwdParams& p) {
    if constexpr (SPLIT) {
        return decode_item<CAUSAL>(w, p);
    } else {
        ItemInfo it;
        it.ui = decode_unit<CAUSAL>(w, p);
        it.u = w;
        it.seg = 0;
        it.nseg = 1;
        it.jb = 0;
        it.je = it.ui.n[1];
        return it;
    }
}

template <bool CAUSAL, bool DYN = false, bool SPLIT = false>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_vt, const FwdParams p) {
    using L = Fp8Layout;
    constexpr int D = 128;
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

    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        for (int s = 0; s < kFp8Stages; ++s) {
            mbar_init(bar(L::kKvFull + s), 1);
            mbar_init(bar(L::kKvEmpty + s), 2);  // released by both MMA warps
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kQFull + t), 1);
            mbar_init(bar(L::kQEmpty + t), 1);
            mbar_init(bar(L::kSFull + t), 1);
            mbar_init(bar(L::kSCons + t), 128);
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(L::kPHalf + 2 * t + b), 128);
                mbar_init(bar(L::kPFull + 2 * t + b), 128);
            }
            mbar_init(bar(L::kPFree + 2 * t), 1);
            mbar_init(bar(L::kPFree + 2 * t + 1), 1);
            mbar_init(bar(L::kODone + t), 1);
            mbar_init(bar(L::kOFull + t), 1);
            mbar_init(bar(L::kOEmpty + t), 128);
        }
        mbar_init(bar(L::kDrain + 0), 1);
        mbar_init(bar(L::kDrain + 1), 1);
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(bar(L::kItemFull + s), 1);
            mbar_init(bar(L::kItemEmpty + s), 10);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_vt);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // a split launch's combine kernel waits for this whole grid (griddepcontrol.wait)
    if (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kItemOff);
    // Dynamic schedule, reader side (a whole warp calls it): ring entry r is this
    // CTA's item r + 1, or -1 after the last; false if the wait failed.
    auto take_item = [&](uint32_t r, int& w) -> bool {
        const uint32_t s = r % kItemRing;
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar(L::kItemFull + s), (r / kItemRing) & 1u, ctx));
        if (!got) return false;
        w = item_slot[s];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kItemEmpty + s));
        return true;
    };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        // Per item: Q_0, Q_1, then K_jb, V_jb^T, K_jb+1, ... through the ring.
        RingPos pos{0u, 0u};
        uint32_t issued = 0;
        uint32_t ul = 0;
        uint32_t q_issued = 0;  // bit t: a Q_t load of the latest unit was issued ...
        uint32_t q_parity = 0;  // ... and completes this phase parity of QFull[t]
        bool ok = true;
        uint32_t r = 0;  // dynamic schedule: ring entries published
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok; ++ul) {
            const ItemInfo item = fp8_item<CAUSAL, SPLIT>(w, p);
            const UnitInfo& ui = item.ui;
            q_issued = 0;
            q_parity = ul & 1u;
            for (int t = 0; t < 2 && ok; ++t) {
                ok = mbar_wait(bar(L::kQEmpty + t), (ul & 1u) ^ 1u, ctx);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTile);
                tma_load_3d(s_base + L::kQOff + t * L::kTile, &tmap_q, bar(L::kQFull + t), 0, (ui.q0 + t) * kBr, ui.bh);
                q_issued |= 1u << t;
            }
            for (int j = item.jb; j < item.je && ok; ++j) {
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    ok = mbar_wait(bar(L::kKvEmpty + pos.stage), pos.phase ^ 1u, ctx);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(L::kKvFull + pos.stage), L::kTile);
                    const uint32_t dst = s_base + L::kRingOff + pos.stage * L::kTile;
                    if (kv == 0)
                        tma_load_3d(dst, &tmap_k, bar(L::kKvFull + pos.stage), 0, j * kBc, ui.bh);
                    else
                        tma_load_3d(dst, &tmap_vt, bar(L::kKvFull + pos.stage), j * kBc, 0, ui.bh);
                    pos = pos.next(kFp8Stages);
                    ++issued;
                }
            }
            if (!ok) break;
            if constexpr (DYN) {
                // claim this CTA's next item and publish it to the other roles
                // the counter was zeroed by the grid this one depends on: wait for it first
                if (r == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                w = static_cast<int>(gridDim.x) + atomicAdd(p.sched_counter, 1);
                if (w >= p.num_items) w = -1;
                const uint32_t s = r % kItemRing;
                if (r >= kItemRing && !(ok = mbar_wait(bar(L::kItemEmpty + s), ((r / kItemRing) - 1) & 1u, ctx)))
                    break;
                item_slot[s] = w;
                mbar_arrive(bar(L::kItemFull + s));
                ++r;
            } else {
                w += gridDim.x;
            }
        }
        // Every issued copy lands before the CTA's shared memory is released
        // (bounded waits; they return at once after a normal run, whose phases
        // have all completed, and matter after an abort by any role).
        const uint32_t pending = issued < static_cast<uint32_t>(kFp8Stages) ? issued : kFp8Stages;
        RingPos back = pos;
        for (uint32_t i = 0; i < pending; ++i) {
            back = back.stage == 0 ? RingPos{kFp8Stages - 1u, back.phase ^ 1u} : RingPos{back.stage - 1, back.phase};
            mbar_wait_drain(bar(L::kKvFull + back.stage), back.phase, 50000000ull);
        }
        for (int t = 0; t < 2; ++t)
            if (q_issued & (1u << t)) mbar_wait_drain(bar(L::kQFull + t), q_parity, 50000000ull);
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues tile 0's products, warp 2 tile 1's: with P in shared memory
        // the two tiles' chains are independent, and one issuing warp per tile keeps
        // either chain from waiting on the other.  Per work item, over its K/V
        // tiles j = jb .. je: the scores S_t(j) (issued once the softmax has loaded
        // S_t(j-1)), then O_t += P_t(j-1) V_{j-1} (half by half as P_t lands).  Both warps release
        // every K/V stage (kKvEmpty counts 2); for a K/V tile its query tile does not
        // visit (causal), the warp arrives once the stage's fill has landed, so that
        // the arrival counts toward that fill.
        const int t = warp - 1;
        constexpr uint32_t idesc = make_idesc_e4m3_f32(kBr, kBc);  // N = kBc = D = 128
        const uint64_t aq = make_smem_desc_sw128(s_base + L::kQOff + t * L::kTile, 16, 1024);
        const uint64_t dr0 = make_smem_desc_sw128(s_base + L::kRingOff, 16, 1024);
        const uint64_t dp0 = make_smem_desc_sw128(s_base + L::kPOff + 2 * t * L::kTile, 16, 1024);
        const uint32_t t_s = tmem + t * kBc, t_o = tmem + 2 * kBc + t * D;
        uint32_t s_cnt = 0;   // S_t issued so far (all units)
        uint32_t p_cnt = 0;   // O_t += P_t V issued so far (all units)
        RingPos kpos{0u, 0u};  // ring position of the unit's K_0
        uint32_t ul = 0;
        bool ok = true;
        auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
            const bool w = mbar_wait(b, parity, ctx);
            return __all_sync(0xffffffffu, w);
        };
        uint32_t r = 0;
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok; ++ul) {
            const ItemInfo item = fp8_item<CAUSAL, SPLIT>(w, p);
            // the item's K/V tiles are [jb, e1); tile t visits [jb, nt)
            const int jb = item.jb, e1 = item.je, nt = min(item.je, item.ui.n[t]);
            ok = wait_all(bar(L::kQFull + t), ul & 1u);
            RingPos kp = kpos;                    // K_j
            RingPos vp = kpos.next(kFp8Stages);   // V_{j-1}^T
            for (int j = jb; j <= e1 && ok; ++j) {
                if (j < e1) {
                    if (!(ok = wait_all(bar(L::kKvFull + kp.stage), kp.phase))) break;
                    if (j < nt) {
                        if (s_cnt > 0 && !(ok = wait_all(bar(L::kSCons + t), (s_cnt - 1) & 1u))) break;
                        tc_fence_after_sync();
                        if (elect_one()) {
                            const uint64_t b = dr0 + static_cast<uint64_t>((kp.stage * L::kTile) >> 4);
#pragma unroll
                            for (int kk = 0; kk < D / 32; ++kk) {
                                const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                                mma_ss_f8(t_s, aq + off, b + off, idesc, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar(L::kSFull + t));
                            if (j == nt - 1) mma_commit(bar(L::kQEmpty + t));  // Q_t's last reader
                            mma_commit(bar(L::kKvEmpty + kp.stage));
                        }
                        __syncwarp();
                        ++s_cnt;
                    } else {
                        if (lane == 0) mbar_arrive(bar(L::kKvEmpty + kp.stage));
                        __syncwarp();
                    }
                    kp = kp.next(kFp8Stages).next(kFp8Stages);
                }
                if (j == jb) continue;
                const int jj = j - 1;  // O_t += P_t(jj) V_jj
                if (!(ok = wait_all(bar(L::kKvFull + vp.stage), vp.phase))) break;
                if (jj < nt) {
                    const uint32_t pb = p_cnt & 1u;         // P buffer of this product
                    const uint32_t pu = (p_cnt >> 1) & 1u;  // parity of this buffer's use
                    const uint64_t a0 = dp0 + static_cast<uint64_t>((pb * L::kTile) >> 4);
                    const uint64_t b0 = dr0 + static_cast<uint64_t>((vp.stage * L::kTile) >> 4);
                    bool ready = mbar_wait(bar(L::kPHalf + 2 * t + pb), pu, ctx);
                    if (jj == jb) ready = ready && mbar_wait(bar(L::kOEmpty + t), (ul & 1u) ^ 1u, ctx);
                    if (!(ok = __all_sync(0xffffffffu, ready))) break;
                    tc_fence_after_sync();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {  // keys 0-63; the item's first product starts O_t
                            const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                            mma_ss_f8(t_o, a0 + off, b0 + off, idesc, (jj > jb || kk > 0) ? 1u : 0u);
                        }
                    }
                    __syncwarp();
                    if (!(ok = wait_all(bar(L::kPFull + 2 * t + pb), pu))) break;
                    tc_fence_after_sync();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 2; kk < 4; ++kk) {  // keys 64-127
                            const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                            mma_ss_f8(t_o, a0 + off, b0 + off, idesc, 1u);
                        }
                        mma_commit(bar(L::kPFree + 2 * t + pb));
                        mma_commit(bar(L::kODone + t));
                        if (jj == nt - 1) mma_commit(bar(L::kOFull + t));
                        mma_commit(bar(L::kKvEmpty + vp.stage));
                    }
                    __syncwarp();
                    ++p_cnt;
                } else {
                    if (lane == 0) mbar_arrive(bar(L::kKvEmpty + vp.stage));
                    __syncwarp();
                }
                vp = vp.next(kFp8Stages).next(kFp8Stages);
            }
            kpos = kp;
            if constexpr (DYN) {
                if (ok) ok = take_item(r++, w);
            } else {
                w += gridDim.x;
            }
        }
        if (elect_one()) mma_commit(bar(L::kDrain + t));
        __syncwarp();
        mbar_wait_drain(bar(L::kDrain + t), 0, 1000000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int rloc = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_addr + t * kBc;
        const uint32_t t_o = tmem + lane_addr + 2 * kBc + t * D;
        const float sl2 = p.scale_log2;
        uint32_t s_cnt = 0;  // S_t processed (all units)
        uint32_t ul = 0;
        bool ok = true;
        uint32_t r = 0;
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok; ++ul) {
            const ItemInfo item = fp8_item<CAUSAL, SPLIT>(w, p);
            const UnitInfo& ui = item.ui;
            const int qt = ui.q0 + t;
            const int qrow = qt * kBr + rloc;
            const int jb = item.jb, nt = min(item.je, ui.n[t]);  // this tile's K/V tiles are [jb, nt)
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int j = jb; j < nt; ++j, ++s_cnt) {
                // This iteration's P buffer is free once the O_t += P V two iterations
                // back has read it; that also makes the product before the previous
                // one complete, so the rescale's wait on the previous one is exact.
                const uint32_t pb = s_cnt & 1u;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kSFull + t), s_cnt & 1u, ctx) &&
                                                 mbar_wait(bar(L::kPFree + 2 * t + pb), ((s_cnt >> 1) & 1u) ^ 1u, ctx));
                if (!ok) break;
                tc_fence_after_sync();
                // Load S_t (all four loads in flight, one wait) and release its columns.
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(t_s + 0, r0);
                tmem_ld32(t_s + 32, r1);
                tmem_ld32(t_s + 64, r2);
                tmem_ld32(t_s + 96, r3);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
                tmem_wait_ld(r2);
                tmem_wait_ld(r3);
                tc_fence_before_sync();
                mbar_arrive(bar(L::kSCons + t));  // S_t's columns may take the next scores
                float* s0 = reinterpret_cast<float*>(r0);
                float* s1 = reinterpret_cast<float*>(r1);
                float* s2 = reinterpret_cast<float*>(r2);
                float* s3 = reinterpret_cast<float*>(r3);
                const int key0 = j * kBc;
                const bool need_mask = (key0 + kBc > p.N) || (CAUSAL && j >= qt);
                const int lim = CAUSAL ? min(p.N - 1, qrow) : p.N - 1;
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (key0 + c > lim) s0[c] = -INFINITY;
                        if (key0 + 32 + c > lim) s1[c] = -INFINITY;
                    }
                }
                float mx0 = fmax3(s0[0], s0[1], s0[2]), mx1 = fmax3(s1[0], s1[1], s1[2]);
#pragma unroll
                for (int c = 3; c < 31; c += 2) {
                    mx0 = fmax3(mx0, s0[c], s0[c + 1]);
                    mx1 = fmax3(mx1, s1[c], s1[c + 1]);
                }
                mx0 = fmax3(mx0, s0[31], fmaxf(mx1, s1[31]));
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (key0 + 64 + c > lim) s2[c] = -INFINITY;
                        if (key0 + 96 + c > lim) s3[c] = -INFINITY;
                    }
                }
                float mx2 = fmax3(s2[0], s2[1], s2[2]), mx3 = fmax3(s3[0], s3[1], s3[2]);
#pragma unroll
                for (int c = 3; c < 31; c += 2) {
                    mx2 = fmax3(mx2, s2[c], s2[c + 1]);
                    mx3 = fmax3(mx3, s3[c], s3[c + 1]);
                }
                mx0 = fmax3(mx0, fmax3(mx2, s2[31], mx3), s3[31]);
                const float m_tile = mx0 * sl2;
                const bool grow = m_tile > m_ref + kRescaleLog2;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2_approx(m_ref - m_tile);
                    m_ref = m_tile;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                l *= alpha;
                // P = 2^(s*scale*log2e - m) -> E4M3, 32 keys (two 16-byte chunks) at a time,
                // into row rloc of the P buffer (128-byte swizzle: chunk c at c ^ (rloc & 7)).
                uint8_t* prow = smem + L::kPOff + (2 * t + pb) * L::kTile + rloc * 128;
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
                auto exp_chunk = [&](const float* sc, int chunk) {
                    uint32_t pk[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        float x0, x1, x2, x3;  // exponents, two per packed instruction
                        ffma2(x0, x1, sc[2 * c], sc[2 * c + 1], sl2, -m_use);
                        ffma2(x2, x3, sc[2 * c + 2], sc[2 * c + 3], sl2, -m_use);
                        float a0, b0, a1, b1;
                        // the first kFp8PolyPer32 scores of every 32 on the FMA pipes
                        if (2 * c < kFp8PolyPer32) {
                            exp2_poly2(a0, b0, x0, x1);
                        } else {
                            a0 = ex2_approx(x0);
                            b0 = ex2_approx(x1);
                        }
                        if (2 * c + 2 < kFp8PolyPer32) {
                            exp2_poly2(a1, b1, x2, x3);
                        } else {
                            a1 = ex2_approx(x2);
                            b1 = ex2_approx(x3);
                        }
                        fadd2(acc0, acc1, a0, b0);
                        fadd2(acc2, acc3, a1, b1);
                        pk[c / 2] = pack_e4m3x4(a0, b0, a1, b1);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int ch = 2 * chunk + h;
                        *reinterpret_cast<uint4*>(prow + ((ch ^ (rloc & 7)) << 4)) =
                            make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
                    }
                };
                exp_chunk(s0, 0);
                exp_chunk(s1, 1);
                // Rescale the O accumulator when this row's reference maximum moved
                // (after the first half's exponentials, when their scores are dead),
                // before the first half of P_t is released to O_t += P_t V.
                if (__any_sync(0xffffffffu, grow && j > jb)) {
                    // O_t must hold exactly the earlier iterations' products before the rescale
                    ok = __all_sync(0xffffffffu, mbar_wait_inline(bar(L::kODone + t), (s_cnt - 1) & 1u, ctx));
                    if (!ok) break;
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_o + c, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_o + c, o);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();  // P written by threads, read by the tensor core
                tc_fence_before_sync();
                mbar_arrive(bar(L::kPHalf + 2 * t + pb));
                exp_chunk(s2, 2);
                exp_chunk(s3, 3);
                fence_proxy_async_smem();
                l += (acc0 + acc1) + (acc2 + acc3);
                mbar_arrive(bar(L::kPFull + 2 * t + pb));
            }
            if (!ok) break;
            // Epilogue: O = O_acc * v_scale / l -> bf16, LSE = ln 2 * (m + log2 l).
            ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kOFull + t), ul & 1u, ctx));
            if (!ok) break;
            tc_fence_after_sync();
            const float inv_l = p.out_scale / l;
            const bool row_ok = qrow < p.N;
            const size_t grow_idx = static_cast<size_t>(ui.bh) * p.N + (row_ok ? qrow : 0);
            const float lse = ((m_ref == -INFINITY ? 0.f : m_ref) + lg2_approx(l)) * kLn2;
            if (!SPLIT || item.nseg == 1) {
                uint4* orow = reinterpret_cast<uint4*>(p.O + grow_idx * D);
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c, o);
                    tmem_wait_ld(o);
                    uint32_t pw[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pw[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            orow[c / 8 + i] = make_uint4(pw[4 * i], pw[4 * i + 1], pw[4 * i + 2], pw[4 * i + 3]);
                    }
                    __syncwarp();
                }
                if (row_ok) p.LSE[grow_idx] = lse;
            } else {
                // this segment's O v_scale / l (fp32) and LSE, merged by the combine
                // kernel (evict-last in L2: read back right after this grid)
                const size_t pidx = (static_cast<size_t>(item.u - p.split_first) * p.kv_split + item.seg) * (2 * kBr) +
                                    t * kBr + rloc;
                float* orow = p.part_o + pidx * D;
                const uint64_t keep = l2_policy_evict_last();
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c, o);
                    tmem_wait_ld(o);
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            st_global_v4_hint(orow + c + 4 * i, __uint_as_float(o[4 * i]) * inv_l,
                                              __uint_as_float(o[4 * i + 1]) * inv_l, __uint_as_float(o[4 * i + 2]) * inv_l,
                                              __uint_as_float(o[4 * i + 3]) * inv_l, keep);
                    }
                    __syncwarp();
                }
                if (row_ok) st_global_hint(p.part_lse + pidx, lse, keep);
            }
            tc_fence_before_sync();
            mbar_arrive(bar(L::kOEmpty + t));
            if constexpr (DYN) {
                ok = take_item(r++, w);
            } else {
                w += gridDim.x;
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

}  // namespace elsattn
