// Fused exact-attention forward for sm_103a: TMA K/V ring -> tcgen05 S = Q K^T
// into TMEM -> online softmax (exp2) in the softmax warpgroups -> P (bf16)
// back into TMEM -> tcgen05 O += P V -> O / l and LSE to global memory.
//
// The loop structure is the streaming schedule of "From Attention Graph to
// FlashAttention - A Memory-Centric Compilation Approach in AICF", section 5:
// each query tile is loaded once, and for every K/V tile the scores are
// computed, the running softmax is updated and the output accumulated.  Here it
// is mapped onto one GB300 SM:
//
//   warp 0 (one lane)   TMA producer: Q tiles once per unit, then K_j, V_j
//                       into a ring of shared-memory stages.
//   warp 1 (one lane)   tcgen05.mma issuer; warp 1 also owns the TMEM
//                       allocation.
//   warps 4-7, 8-11     softmax warpgroups, one per resident query tile; thread
//                       r owns query row r (TMEM lane r) of its tile.
//
// Two query tiles (Q0, Q1) share every K/V tile.  The MMA warp interleaves
// them so that the tensor core works on one tile while the softmax of the
// other runs (the AttenIO abstract overlaps data movement with computation at
// three levels; here the levels are TMA, the tensor core and the softmax warps):
//     S0_j = Q0 K_j^T ; O1 += P1_{j-1} V_{j-1} ; S1_j = Q1 K_j^T ; O0 += P0_j V_j
//
// Work: a unit is a pair of query tiles of one (batch, head) against all the
// K/V tiles they see.  A work item is a unit, or one segment of a unit's K/V
// range when the launch is split (FwdParams::kv_split; a second kernel merges
// the segments).  Persistent CTAs take items by a fixed stride, or claim them
// from a counter when the kernel is instantiated with DYN (launches whose
// items differ in length), the producer passing each claimed item to the
// other roles through a two-slot shared-memory ring.
//
// TMEM columns: [0,128) S0 | [128,256) S1 | [256,256+d) O0 | [256+d,256+2d) O1.
// P_t (bf16, two per column) is written over the first 64 columns of S_t once
// the softmax has read S_t into registers.  The next S_t = Q_t K^T is issued
// after O_t += P_t V has been issued; tcgen05.mma operations of one thread run
// in issue order on the SM's tensor core.
//
// Online softmax (the streaming reformulation of the IO-Aware Algorithms
// page): per row, a reference maximum m (log2 units, scale folded in) and a
// running sum l.  A tile whose row maximum exceeds m by more than
// kRescaleLog2Bf16 moves m up and rescales l and the O accumulator by
// 2^(m_old - m_new); smaller increases keep the stale m (the terms stay below
// 2^kRescaleLog2Bf16 and the final O / l and LSE are unchanged by the choice
// of m).  On N(0, 1) inputs no row moves m after its first tile; on inputs
// with rare large entries (1 % of Q and K entries times 10) a warp rescales on
// about 40 % of its tiles at a threshold of 8 and about 12 % at 32.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "exp2_poly.h"
#include "plan.h"
#include "sm103_ptx.cuh"

// Scores out of every 32 of a row whose exp2 is evaluated on the FMA pipes
// (exp2_poly.h) instead of the special-function unit: 0, 2, 4, 6 or 8.
#ifndef ELS_EXP2_POLY_PER32
#define ELS_EXP2_POLY_PER32 0
#endif
// Stale-maximum threshold of this kernel, log2 units (see kRescaleLog2Bf16).
#ifndef ELS_RESCALE_LOG2_BF16
#define ELS_RESCALE_LOG2_BF16 32
#endif

namespace elsattn {

// Threshold of the FP8 kernel, whose P is E4M3 (at most 448): terms must stay
// at most 2^8.
constexpr float kRescaleLog2 = 8.0f;
// Threshold of the bf16 kernel: terms stay at most 2^T, so l <= N 2^T and
// |O_acc| <= N 2^T max|V| in fp32, which at T = 32 leaves room for
// max|V| < 2^96 / N (2^65 at N = 2^31).  A larger T moves the reference
// maximum, and rescales O, less often on rows whose large scores arrive late
// (about 3 % faster than T = 8 on the stress recipe, measured).
constexpr float kRescaleLog2Bf16 = ELS_RESCALE_LOG2_BF16;
static_assert(kRescaleLog2Bf16 >= 1.0f && kRescaleLog2Bf16 <= 64.0f, "stale-maximum threshold out of range");
constexpr int kPolyPer32 = ELS_EXP2_POLY_PER32;
static_assert(kPolyPer32 >= 0 && kPolyPer32 <= 8 && kPolyPer32 % 2 == 0, "exp2 offload: 0, 2, 4, 6 or 8 per 32");
constexpr float kLn2 = 0.693147180559945309f;

struct FwdParams {
    __nv_bfloat16* O;      // [BH, N, d]
    float* LSE;            // [BH, N]
    uint32_t* error_word;  // device error word (first error wins)
    uint64_t timeout_ns;   // limit for any single wait
    int N;
    int BH;
    int num_q_tiles;       // ceil(N / kBr)
    int num_kv_tiles;      // ceil(N / kBc)
    int num_pairs;         // ceil(num_q_tiles / 2): units per (batch, head)
    int num_units;         // BH * num_pairs
    int heads_per_group;   // causal schedule only
    float scale_log2;      // scale * log2(e) (times the Q and K scales for the FP8 kernel)
    float out_scale;       // FP8 kernel: the V scale, applied with 1 / l; unused here
    // K/V split (this kernel only; the FP8 kernel runs whole units): the units
    // [split_first, split_first + split_units) in schedule order are cut into
    // kv_split segments of consecutive K/V tiles, one work item each; the other
    // units are one item each, and the items follow unit order.  A split item
    // writes O / l and its LSE to part_o / part_lse at its unit's ordinal among
    // the split units, and attn_fwd_combine_kernel merges the segments.
    int kv_split;          // segments per split unit (1: no split)
    int split_first;       // first split unit
    int split_units;       // units that are split (0: none)
    int num_items;         // num_units + split_units * (kv_split - 1)
    float* part_o;         // [split_units, kv_split, 2 * kBr rows of the pair, d] fp32
    float* part_lse;       // [split_units, kv_split, 2 * kBr] fp32 (natural log)
    // Dynamic work-item schedule (kernel instantiated with DYN): each CTA starts
    // with item blockIdx.x and then claims the next unclaimed item from this
    // counter (zero at launch), so items go out in schedule order to whichever
    // CTA is free first.  Static schedule (nullptr): CTA b takes items b,
    // b + grid, b + 2 grid, ...
    int* sched_counter;
    // Nonzero: S = Q (-K)^T (the instruction descriptor's negate-B bit).  A
    // negative scale is run as |scale| on the negated scores, so the kernel's
    // running maximum always tracks the largest scaled score.  (bf16 kernel only.)
    uint32_t negate_scores = 0;
    // Factor of a tile's raw score maximum in the running maximum: scale_log2,
    // except 0 for a zero scale, whose scale_log2 is the smallest normal float
    // (every term is then exactly 1 and the running maximum stays exactly 0,
    // so LSE = ln(#visible keys) exactly).  (bf16 kernel only.)
    float max_scale_log2 = 0.f;
    // Test hook: nonzero makes CTA 0 arm the barrier of its first Q_0 load
    // without issuing the copy, so that a wait on it runs out of time and the
    // kernel takes its abort path.  Zero in every normal launch.
    uint32_t withhold_first_q = 0;
};

struct UnitInfo {
    int bh;
    int q0;      // first query tile of the pair (second is q0 + 1)
    int n[2];    // K/V tiles each query tile visits
};

// Unit order.  Non-causal: head-major, so the CTAs running at the same time
// read the K/V of few heads and share them in L2.  Causal: heads are taken in
// groups; inside a group the heaviest query tiles (most visible keys) go first
// and the heads of the group interleave, which keeps the L2 working set to a
// group's K/V while starting long units early.
template <bool CAUSAL>
__device__ __forceinline__ UnitInfo decode_unit(int u, const FwdParams& p) {
    UnitInfo ui;
    int pair;
    if (!CAUSAL) {
        ui.bh = u / p.num_pairs;
        pair = u - ui.bh * p.num_pairs;
    } else {
        const int G = p.heads_per_group;
        const int g = u / (G * p.num_pairs);
        const int r = u - g * G * p.num_pairs;
        const int heads_here = min(G, p.BH - g * G);
        const int rank = r / heads_here;
        pair = p.num_pairs - 1 - rank;
        ui.bh = g * G + (r - rank * heads_here);
    }
    ui.q0 = 2 * pair;
    for (int t = 0; t < 2; ++t) {
        const int qt = ui.q0 + t;
        ui.n[t] = CAUSAL ? min(qt + 1, p.num_kv_tiles) : p.num_kv_tiles;
    }
    return ui;
}


// Work item w: segment `seg` of `nseg` of a unit, covering the pair's K/V tiles
// [jb, je); tile t visits [jb, min(je, n[t])).  The host splits a unit into s
// segments only when s (s - 1) < n[0]; with n[1] equal to n[0] or n[0] + 1 each
// segment then holds at least one K/V tile of tile 0, so every row sees at
// least one key in every segment.
struct ItemInfo {
    UnitInfo ui;
    int u;       // unit index
    int seg;
    int nseg;
    int jb, je;
};

template <bool CAUSAL>
__device__ __forceinline__ ItemInfo decode_item(int w, const FwdParams& p) {
    ItemInfo it;
    const int split_items = p.split_units * p.kv_split;
    int u;
    if (w < p.split_first) {  // whole units before the split range
        u = w;
        it.seg = 0;
        it.nseg = 1;
    } else if (w < p.split_first + split_items) {
        const int r = w - p.split_first;
        const int ord = r / p.kv_split;
        u = p.split_first + ord;
        it.seg = r - ord * p.kv_split;
        it.nseg = p.kv_split;
    } else {  // whole units after it
        u = w - split_items + p.split_units;
        it.seg = 0;
        it.nseg = 1;
    }
    it.u = u;
    it.ui = decode_unit<CAUSAL>(u, p);
    const int n1 = it.ui.n[1];
    const int c = (n1 + it.nseg - 1) / it.nseg;
    it.jb = it.seg * c;
    it.je = min(n1, it.jb + c);
    return it;
}

// The producer hands each CTA's work items to the other roles through a ring of
// this many shared-memory slots (an item index, -1 at the end).
constexpr int kItemRing = 2;

// Position in the shared-memory K/V ring: stage index and the parity of the
// stage's current fill.
struct RingPos {
    uint32_t stage;
    uint32_t phase;
    __device__ __forceinline__ RingPos next(uint32_t stages) const {
        return stage + 1 == stages ? RingPos{0u, phase ^ 1u} : RingPos{stage + 1, phase};
    }
};

template <int D>
struct SmemLayout {
    static constexpr int kTile = tile_bytes(D);
    static constexpr int kStages = kv_stages_for(D);
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQTiles * kTile;
    static constexpr int kBarOff = kRingOff + kStages * kTile;
    // barrier indices
    static constexpr int kKvFull = 0;
    static constexpr int kKvEmpty = kKvFull + kStages;
    static constexpr int kQFull = kKvEmpty + kStages;   // [2]
    static constexpr int kQEmpty = kQFull + 2;          // [2]
    static constexpr int kSFull = kQEmpty + 2;          // [2]
    static constexpr int kPHalf = kSFull + 2;           // [2] first half of P_t (keys 0-63) stored, O_t rescaled
    static constexpr int kPFull = kPHalf + 2;           // [2] second half of P_t stored
    static constexpr int kOFull = kPFull + 2;           // [2]
    static constexpr int kOEmpty = kOFull + 2;          // [2]
    static constexpr int kDrain = kOEmpty + 2;
    static constexpr int kItemFull = kDrain + 1;        // [kItemRing] the slot holds the next item index
    static constexpr int kItemEmpty = kItemFull + kItemRing;  // [kItemRing] MMA warp + 8 softmax warps read it
    static constexpr int kNumBars = kItemEmpty + kItemRing;
    static constexpr int kFlagsOff = kBarOff + kNumBars * 8;  // tmem base slot, abort flag, item indices
    static constexpr int kItemOff = kFlagsOff + 8;             // [kItemRing] int
    static constexpr int kBytes = kFlagsOff + 16;
    static_assert(kNumBars == 2 * kStages + kFixedBarriers, "barrier count differs from the plan");
    static_assert(kBytes + kSmemAlign <= smem_bytes_for(D), "shared memory layout exceeds the plan");
};

// DYN: the dynamic work-item schedule (p.sched_counter is set); without it the
// static schedule is compiled with no trace of the item ring.
template <int D, bool CAUSAL, bool DYN = false>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
    using L = SmemLayout<D>;
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
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar(L::kKvFull + s), 1);
            mbar_init(bar(L::kKvEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kQFull + t), 1);
            mbar_init(bar(L::kQEmpty + t), 1);
            mbar_init(bar(L::kSFull + t), 1);
            mbar_init(bar(L::kPHalf + t), 128);
            mbar_init(bar(L::kPFull + t), 128);
            mbar_init(bar(L::kOFull + t), 1);
            mbar_init(bar(L::kOEmpty + t), 128);
        }
        mbar_init(bar(L::kDrain), 1);
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(bar(L::kItemFull + s), 1);
            mbar_init(bar(L::kItemEmpty + s), 9);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // A split launch's combine kernel may be scheduled onto SMs as this grid's
    // CTAs retire; it waits for this whole grid (griddepcontrol.wait) before it
    // reads the partial results.
    if (p.kv_split > 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kItemOff);
    // Every role starts with item blockIdx.x (the grid never exceeds the item
    // count).  The static schedule then advances by gridDim.x; the dynamic one
    // takes the next items from the producer's ring: ring entry r is this CTA's
    // item r + 1, or -1 after the last.  Consumer side (a whole warp calls it):
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
        RingPos pos{0u, 0u};      // next ring position to fill
        uint32_t issued = 0;      // ring fills issued so far
        uint32_t ul = 0;
        uint32_t q_issued = 0;    // bit t: a Q_t load of the latest item was issued ...
        uint32_t q_parity = 0;    // ... and completes this phase parity of QFull[t]
        bool ok = true;
        uint32_t r = 0;  // dynamic schedule: ring entries published
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok;) {
            q_issued = 0;
            q_parity = ul & 1u;
            const ItemInfo item = decode_item<CAUSAL>(w, p);
            const UnitInfo& ui = item.ui;
            for (int t = 0; t < 2 && ok; ++t) {
                ok = mbar_wait(bar(L::kQEmpty + t), (ul & 1u) ^ 1u, ctx);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTile);
                const uint32_t dst = s_base + L::kQOff + t * L::kTile;
                if (!(p.withhold_first_q && blockIdx.x == 0 && ul == 0 && t == 0)) {
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(dst + b * (kBr * 128), &tmap_q, bar(L::kQFull + t), b * 64, (ui.q0 + t) * kBr, ui.bh);
                }
                q_issued |= 1u << t;
            }
            for (int j = item.jb; j < item.je && ok; ++j) {
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    ok = mbar_wait(bar(L::kKvEmpty + pos.stage), pos.phase ^ 1u, ctx);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(L::kKvFull + pos.stage), L::kTile);
                    const uint32_t dst = s_base + L::kRingOff + pos.stage * L::kTile;
                    const CUtensorMap* tm = kv == 0 ? &tmap_k : &tmap_v;
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(dst + b * (kBc * 128), tm, bar(L::kKvFull + pos.stage), b * 64, j * kBc, ui.bh);
                    pos = pos.next(L::kStages);
                    ++issued;
                }
            }
            if (!ok) break;
            ++ul;
            if constexpr (DYN) {
                // claim this CTA's next item and publish it to the other roles
                // the counter was zeroed by the grid this one depends on (see
                // zero_sched_counter_kernel): wait for it before the first claim
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
        // (bounded waits).  Only the last min(issued, stages) fills and the
        // latest item's Q loads can still be pending: after a normal run their
        // phases have completed and these waits return at once; after an abort
        // (this role's wait or another role's gave up) they may not have.
        const uint32_t pending = issued < static_cast<uint32_t>(L::kStages) ? issued : L::kStages;
        RingPos back = pos;
        for (uint32_t i = 0; i < pending; ++i) {
            back = back.stage == 0 ? RingPos{L::kStages - 1u, back.phase ^ 1u} : RingPos{back.stage - 1, back.phase};
            mbar_wait_drain(bar(L::kKvFull + back.stage), back.phase, 50000000ull);
        }
        for (int t = 0; t < 2; ++t)
            if (q_issued & (1u << t)) mbar_wait_drain(bar(L::kQFull + t), q_parity, 50000000ull);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop and waits; one elected lane issues the
        // MMAs and commits (a converged warp issues tcgen05.mma faster than a
        // lone divergent lane).
        const uint32_t idesc_s = make_idesc_bf16_f32(kBr, kBc, false, false) | (p.negate_scores ? kIdescNegateB : 0u);
        constexpr uint32_t idesc_o = make_idesc_bf16_f32(kBr, D, false, true);
        // The descriptor's start-address field holds (address >> 4), so a move
        // inside shared memory is an add on the descriptor.
        const uint64_t dq0 = make_smem_desc_sw128(s_base + L::kQOff, 16, 1024);
        const uint64_t dk0 = make_smem_desc_sw128(s_base + L::kRingOff, 16, 1024);
        const uint64_t dv0 = make_smem_desc_sw128(s_base + L::kRingOff, kBc * 128, 1024);
        RingPos kpos{0u, 0u};  // ring position of the next unit's K_0
        uint32_t ul = 0;
        uint32_t p_phase[2] = {0u, 0u};
        bool ok = true;
        // S_t = Q_t K^T with K in ring stage `slot`.
        auto gemm_s = [&](int t, uint32_t slot) {
            const uint64_t a = dq0 + static_cast<uint64_t>((t * L::kTile) >> 4);
            const uint64_t b = dk0 + static_cast<uint64_t>((slot * L::kTile) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * (kBr * 128) + (kk & 3) * 32) >> 4);
                mma_ss(tmem + t * kBc, a + off, b + off, idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        // O_t (+)= P_t V over keys [64 half, 64 half + 64) with V in ring stage
        // `slot`; P_t is read from TMEM.
        auto gemm_o = [&](int t, uint32_t slot, int half, bool accumulate) {
            const uint64_t b = dv0 + static_cast<uint64_t>((slot * L::kTile) >> 4);
#pragma unroll
            for (int kk = half * 4; kk < half * 4 + 4; ++kk)
                mma_ts(tmem + 2 * kBc + t * D, tmem + t * kBc + kk * 8,
                       b + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_o, (accumulate || kk > 0) ? 1u : 0u);
        };
        uint32_t r = 0;
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok;) {
            const ItemInfo item = decode_item<CAUSAL>(w, p);
            // K/V tiles [jb, e1) of the pair; tile 0 stops at e0 (causal: one earlier)
            const int jb = item.jb, e1 = item.je, e0 = min(item.je, item.ui.n[0]);
            ok = mbar_wait(bar(L::kQFull + 0), ul & 1u, ctx) && mbar_wait(bar(L::kQFull + 1), ul & 1u, ctx);
            ok = __all_sync(0xffffffffu, ok);
            // O_t += P_t V_j with V_j at ring position `vp`, with the waits it needs.
            auto pv = [&](int t, int j, RingPos vp) -> bool {
                bool w = true;
                if (t == 0 || j >= e0)  // first use of V_j
                    w = mbar_wait(bar(L::kKvFull + vp.stage), vp.phase, ctx);
                // The softmax releases P_t in two halves, so the tensor core
                // starts on keys 0-63 while the exponentials of 64-127 run.
                w = w && mbar_wait(bar(L::kPHalf + t), p_phase[t], ctx);
                if (j == jb) w = w && mbar_wait(bar(L::kOEmpty + t), (ul & 1u) ^ 1u, ctx);
                if (!__all_sync(0xffffffffu, w)) return false;
                tc_fence_after_sync();  // P_t and the O_t rescale came from other threads' tcgen05.st
                if (elect_one()) gemm_o(t, vp.stage, 0, j > jb);
                __syncwarp();
                w = mbar_wait(bar(L::kPFull + t), p_phase[t], ctx);
                p_phase[t] ^= 1u;
                if (!__all_sync(0xffffffffu, w)) return false;
                tc_fence_after_sync();
                if (elect_one()) {
                    gemm_o(t, vp.stage, 1, true);
                    if (t == 1) mma_commit(bar(L::kKvEmpty + vp.stage));  // V_j's last reader
                    if (j == (t == 0 ? e0 : e1) - 1) mma_commit(bar(L::kOFull + t));
                }
                __syncwarp();
                return true;
            };
            RingPos vpos = kpos.next(L::kStages);  // V_j
            RingPos vprev = vpos;                  // V_{j-1}
            for (int j = jb; j < e1 && ok; ++j) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvFull + kpos.stage), kpos.phase, ctx));
                if (!ok) break;
                if (j < e0) {
                    if (elect_one()) {
                        gemm_s(0, kpos.stage);
                        mma_commit(bar(L::kSFull + 0));
                        if (j == e0 - 1) mma_commit(bar(L::kQEmpty + 0));
                    }
                    __syncwarp();
                }
                if (j > jb && !(ok = pv(1, j - 1, vprev))) break;
                if (elect_one()) {
                    gemm_s(1, kpos.stage);
                    mma_commit(bar(L::kSFull + 1));
                    mma_commit(bar(L::kKvEmpty + kpos.stage));  // K_j's last reader
                    if (j == e1 - 1) mma_commit(bar(L::kQEmpty + 1));
                }
                __syncwarp();
                if (j < e0 && !(ok = pv(0, j, vpos))) break;
                vprev = vpos;
                kpos = kpos.next(L::kStages).next(L::kStages);
                vpos = vpos.next(L::kStages).next(L::kStages);
            }
            if (ok) ok = pv(1, e1 - 1, vprev);
            ++ul;
            if constexpr (DYN) {
                if (ok) ok = take_item(r++, w);
            } else {
                w += gridDim.x;
            }
        }
        // Make sure no MMA is still writing TMEM when it is released.
        if (elect_one()) mma_commit(bar(L::kDrain));
        __syncwarp();
        mbar_wait_drain(bar(L::kDrain), 0, 1000000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 4) >> 2;          // query tile of this warpgroup
        const int quad = warp & 3;              // TMEM lane quadrant this warp may access
        const int rloc = quad * 32 + lane;      // row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_addr + t * kBc;
        const uint32_t t_o = tmem + lane_addr + 2 * kBc + t * D;
        const float sl2 = p.scale_log2;
        uint32_t s_cnt = 0;
        uint32_t ul = 0;
        bool ok = true;
        uint32_t r = 0;
        for (int w = blockIdx.x; (DYN ? w >= 0 : w < p.num_items) && ok;) {
            const ItemInfo item = decode_item<CAUSAL>(w, p);
            const UnitInfo& ui = item.ui;
            const int qt = ui.q0 + t;
            const int qrow = qt * kBr + rloc;
            const int jb = item.jb;
            const int et = min(item.je, t == 0 ? ui.n[0] : ui.n[1]);  // this tile's K/V tiles are [jb, et)
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int j = jb; j < et; ++j) {
                ok = mbar_wait(bar(L::kSFull + t), s_cnt & 1u, ctx);
                ++s_cnt;
                __syncwarp();
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after_sync();
                // Load S_t in two halves: the second load is in flight while the
                // first half is masked and reduced.
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(t_s + 0, r0);
                tmem_ld32(t_s + 32, r1);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
                tmem_ld32(t_s + 64, r2);
                tmem_ld32(t_s + 96, r3);
                float* s0 = reinterpret_cast<float*>(r0);
                float* s1 = reinterpret_cast<float*>(r1);
                float* s2 = reinterpret_cast<float*>(r2);
                float* s3 = reinterpret_cast<float*>(r3);
                const int key0 = j * kBc;
                const bool need_mask = (key0 + kBc > p.N) || (CAUSAL && j >= qt);
                const int lim = CAUSAL ? min(p.N - 1, qrow) : p.N - 1;  // last visible key
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (key0 + c > lim) s0[c] = -INFINITY;
                        if (key0 + 32 + c > lim) s1[c] = -INFINITY;
                    }
                }
                // row max: 3-input max, two independent chains per half
                float mx0 = fmax3(s0[0], s0[1], s0[2]), mx1 = fmax3(s1[0], s1[1], s1[2]);
#pragma unroll
                for (int c = 3; c < 31; c += 2) {
                    mx0 = fmax3(mx0, s0[c], s0[c + 1]);
                    mx1 = fmax3(mx1, s1[c], s1[c + 1]);
                }
                mx0 = fmax3(mx0, s0[31], fmaxf(mx1, s1[31]));
                tmem_wait_ld(r2);
                tmem_wait_ld(r3);
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
                const float m_tile = mx0 * p.max_scale_log2;
                const bool grow = m_tile > m_ref + kRescaleLog2Bf16;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2_approx(m_ref - m_tile);  // 0 on the first tile
                    m_ref = m_tile;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                l *= alpha;
                // P = 2^(s*scale*log2e - m), packed as bf16 pairs over the first
                // 64 columns of S_t, stored 16 columns (32 scores) at a time.
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
                auto exp_chunk = [&](const float* sc, uint32_t col) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        float x0, x1, x2, x3;  // exponents, two per packed instruction
                        ffma2(x0, x1, sc[2 * c], sc[2 * c + 1], sl2, -m_use);
                        ffma2(x2, x3, sc[2 * c + 2], sc[2 * c + 3], sl2, -m_use);
                        float a0, b0, a1, b1;
                        // the first kPolyPer32 scores of every 32 on the FMA pipes
                        if (2 * c < kPolyPer32) {
                            exp2_poly2(a0, b0, x0, x1);
                        } else {
                            a0 = ex2_approx(x0);
                            b0 = ex2_approx(x1);
                        }
                        if (2 * c + 2 < kPolyPer32) {
                            exp2_poly2(a1, b1, x2, x3);
                        } else {
                            a1 = ex2_approx(x2);
                            b1 = ex2_approx(x3);
                        }
                        fadd2(acc0, acc1, a0, b0);
                        fadd2(acc2, acc3, a1, b1);
                        pk[c] = pack_bf16x2(a0, b0);
                        pk[c + 1] = pack_bf16x2(a1, b1);
                    }
                    tmem_st16(t_s + col, pk);
                };
                exp_chunk(s0, 0);
                exp_chunk(s1, 16);
                // Rescale the O accumulator when this row's reference max moved,
                // before the first half of P_t is released to O_t += P_t V.
                // O_t's previous P V has completed: it was issued before this
                // S_t, whose completion was just observed.
                if (__any_sync(0xffffffffu, grow && j > jb)) {
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_o + c, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_o + c, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(bar(L::kPHalf + t));
                exp_chunk(s2, 32);
                exp_chunk(s3, 48);
                l += (acc0 + acc1) + (acc2 + acc3);
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(bar(L::kPFull + t));
            }
            if (!ok) break;
            // Epilogue: O = O_acc / l -> bf16, LSE = ln 2 * (m + log2 l).
            ok = mbar_wait(bar(L::kOFull + t), ul & 1u, ctx);
            __syncwarp();
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after_sync();
            const float inv_l = 1.f / l;
            const bool row_ok = qrow < p.N;
            const size_t grow_idx = static_cast<size_t>(ui.bh) * p.N + (row_ok ? qrow : 0);
            const float lse = ((m_ref == -INFINITY ? 0.f : m_ref) + lg2_approx(l)) * kLn2;
            if (item.nseg == 1) {
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
                }
                if (row_ok) p.LSE[grow_idx] = lse;
            } else {
                // This segment's O / l (fp32) and LSE, merged by the combine
                // kernel.  Stored with an evict-last L2 policy: they are read
                // back right after this grid, and the combine kernel drops them
                // from L2 after reading, so they need not reach device memory.
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
                }
                if (row_ok) st_global_hint(p.part_lse + pidx, lse, keep);
            }
            tc_fence_before_sync();
            mbar_arrive(bar(L::kOEmpty + t));
            ++ul;
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

// Zeroes the dynamic schedule's claim counter ahead of an attention launch that
// depends on it programmatically: that launch's CTAs start at once (each first
// runs item blockIdx.x) and its producer waits for this grid only before its
// first claim, so the zeroing overlaps the attention kernel's start.
static __global__ void zero_sched_counter_kernel(int* counter) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    *counter = 0;
}

// Merge the segments of the split units: per row, with the segments' partial
// results (O_s = softmax over the segment's keys times V, LSE_s),
//     LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s,
// the same online-softmax combination as inside the kernel, across segments,
// in the fixed segment order.  SEG is the launch's segment count, so that a
// thread holds only the partials that exist (its registers set how many CTAs
// an SM holds at once).  One warp per row of the split units (2 kBr rows
// each); lane l holds columns [kPer l, kPer l + kPer) of the row, one vector
// load per segment, so every partial row is one coalesced read.  The rows of
// the other units were written by the attention kernel itself.  After the
// merged row is written, its partial O lines are discarded from L2: nothing
// reads them again, so they are not written back to device memory.
constexpr int kCombineRowsPerCta = 8;  // 256 threads, one warp per row

template <int D>
struct CombineVec;  // one lane's kPer = D / 32 fp32 columns of a partial row
template <>
struct CombineVec<64> {
    __device__ static void load(const float* src, float (&x)[2]) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
        x[0] = v.x, x[1] = v.y;
    }
};
template <>
struct CombineVec<128> {
    __device__ static void load(const float* src, float (&x)[4]) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
        x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
    }
};

template <int D, bool CAUSAL, int SEG>
__global__ void __launch_bounds__(256) attn_fwd_combine_kernel(const FwdParams p) {
    static_assert(SEG >= 2 && SEG <= kMaxKvSplit, "segments");
    constexpr int kPer = D / 32;                 // columns per lane
    constexpr int kLinesPerRow = D * 4 / 128;   // 128-byte lines of one partial row
    // launched as a programmatic dependent of the attention kernel: wait until
    // that grid has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int prow = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);  // over split_units * 2 kBr
    const int lane = threadIdx.x & 31;
    if (prow >= p.split_units * 2 * kBr) return;
    const int ord = prow / (2 * kBr);
    const int rr = prow - ord * 2 * kBr;  // row within the pair: tile rr / kBr, row rr % kBr
    const UnitInfo ui = decode_unit<CAUSAL>(p.split_first + ord, p);
    const int qrow = ui.q0 * kBr + rr;
    if (qrow >= p.N) return;
    const size_t row = static_cast<size_t>(ui.bh) * p.N + qrow;
    const size_t base = static_cast<size_t>(ord) * SEG * (2 * kBr) + rr;  // segment s at base + s * 2 kBr
    float w[SEG];
    float x[SEG][kPer];
#pragma unroll
    for (int s = 0; s < SEG; ++s) {
        w[s] = __ldcg(p.part_lse + base + s * (2 * kBr));
        CombineVec<D>::load(p.part_o + (base + s * (2 * kBr)) * D + lane * kPer, x[s]);
    }
    float mx = w[0];
#pragma unroll
    for (int s = 1; s < SEG; ++s) mx = fmaxf(mx, w[s]);
    float wsum = 0.f;
#pragma unroll
    for (int s = 0; s < SEG; ++s) {
        w[s] = expf(w[s] - mx);  // now the segment weights
        wsum += w[s];
    }
    const float inv = 1.f / wsum;
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
#pragma unroll
    for (int s = 0; s < SEG; ++s) {
        const float ws = w[s] * inv;
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] = fmaf(ws, x[s][c], acc[c]);
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.O + row * D + lane * kPer);
#pragma unroll
    for (int c = 0; c < kPer; c += 2) dst[c / 2] = pack_bf16x2(acc[c], acc[c + 1]);
    if (lane == 0) p.LSE[row] = mx + logf(wsum);
    // every value read above has been consumed by the stores: drop the lines
    if (lane < SEG * kLinesPerRow) {
        const int s = lane / kLinesPerRow, part = lane - s * kLinesPerRow;
        l2_discard_line(reinterpret_cast<const char*>(p.part_o + (base + s * (2 * kBr)) * D) + part * 128);
    }
}

}  // namespace elsattn
