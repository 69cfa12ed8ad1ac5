// Tile planner: an I/O count of the two tall-and-skinny products of
// attention against the on-chip capacity of one sm_103 SM.
//
// The AttenIO abstract ("I/O Analysis is All You Need: An I/O Analysis for
// Long-Sequence Attention", ASPLOS 2026) derives its tiling from an I/O
// analysis of tall-and-skinny matrix multiplication; the IO-Aware Algorithms
// page gives the tiling rule behind it (staging a tile on chip and reusing it
// S times divides the GEMM traffic 2MNK by S).  For one (batch, head), with
// q query tiles of Br rows resident per CTA and K/V streamed in tiles of Bc
// keys:
//     Q is read once                     N d
//     K and V are streamed once per CTA  2 N d * ceil(N / (q Br))
//     O is written once                  N d
// so the streamed K/V term shrinks with the resident query rows q Br, and the
// best tiling is the largest q Br the SM can run.  Br = 128 (one TMEM lane per
// query row, tcgen05 M = 128).  The constraints:
//     shared memory  q Br d 2B + stages Bc d 2B   <= 227 KB   (stages >= 3)
//     tensor memory  q (Bc + d) fp32 columns       <= 512     (S and O per tile)
//     registers      128 (q + 1) threads x (Bc + 40) <= 65536 (a softmax thread
//                    holds its row's Bc scores plus about 40 of state; one
//                    warpgroup besides the q softmax warpgroups loads and issues)
//     tensor rate    S = Q K^T reads both operands from shared memory: per
//                    16-deep step, 2 * 128 * Bc * 16 FLOP take Bc / 2 cycles at
//                    8192 FLOP per cycle, and (128 + Bc) * 16 * 2 bytes take
//                    (128 + Bc) / 4 cycles at 128 B per cycle; the product runs
//                    at the full rate only for Bc >= 128 (O += P V reads P from
//                    tensor memory and only V from shared memory: always full)
// The planner searches every (q, Bc) and keeps the least I/O among the tilings
// that meet all four (on a tie, the more resident rows, then the larger Bc).  That optimum is q = 2, Bc = 128
// for both head dimensions, the tiling the kernel is compiled for.  Without the
// tensor-rate constraint the count alone would favour Bc = 64 with three
// resident tiles at d = 64, whose S products would run at two thirds of the
// rate to save L2 -> shared-memory traffic that is nowhere near its bound.
//
// Device-memory traffic: each (batch, head)'s K and V come from HBM once when
// the K/V of the heads streamed at the same time fit in the L2 budget (the
// head-major order keeps the CTAs in flight on few heads; the causal order
// runs heads in groups sized to that budget); beyond it, every wave of a
// head's units after the first re-reads the share that L2 no longer holds.
// Against ncu DRAM counts on a GB300 the estimate is within about 30 %: the
// headline workload 270 MB (measured 276), B1 H8 N65536 causal 539 MB (reads
// 589), one causal head of 262144 keys 460 MB (reads 547).
#include <cmath>

#include "../../include/exact_attn.h"
#include "plan.h"

namespace elsattn {

constexpr int kRegsPerSm = 65536;
constexpr int kSoftmaxStateRegs = 40;  // registers of a softmax thread besides its row of scores
constexpr double kL2KvBudget = 96.0 * 1024 * 1024;  // of the 126 MB L2, for K/V of the heads in flight

struct Candidate {
    int q, Bc, stages;
    double l2_bytes;
    bool fits;       // shared memory, tensor memory, registers
    bool full_rate;  // S = Q K^T at the tensor core's full rate
};

// K/V bytes the CTAs stream from L2 for one (batch, head), plus Q read and O written.
static double l2_traffic_per_head(int N, int d, int q, int causal) {
    const double nd = static_cast<double>(N) * d;
    const double units = std::ceil(static_cast<double>(N) / (q * kBr));
    // causal: a unit streams only the keys up to its last query row; on average half.
    const double kv_passes = causal ? 0.5 * (units + 1) : units;
    return 2.0 * (nd + 2.0 * nd * kv_passes + nd);
}

static Candidate evaluate(int N, int d, int causal, int q, int Bc) {
    Candidate c{q, Bc, 0, 0.0, false, false};
    const int q_bytes = q * kBr * d * 2;
    const int stage_bytes = Bc * d * 2;
    const int tmem = q * (Bc + d);
    const int threads = 128 * (q + 1);
    const int regs = Bc + kSoftmaxStateRegs;
    c.stages = (kSmemLimit - overhead_bytes(0) - q_bytes) / (stage_bytes + 16);
    c.fits = tmem <= 512 && c.stages >= 3 && regs <= 255 && threads * regs <= kRegsPerSm;
    // per 16-deep step of S: Bc / 2 cycles of arithmetic against (128 + Bc) / 4 of operand reads
    c.full_rate = 2 * Bc >= kBr + Bc;
    c.l2_bytes = l2_traffic_per_head(N, d, q, causal);
    return c;
}

}  // namespace elsattn

using namespace elsattn;

extern "C" int attn_plan_impl(int B, int H, int N, int d, int causal, int num_sms, attn_plan_t* out) {
    if (!out || B < 1 || H < 1 || N < 1 || num_sms < 1) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * N >= (1LL << 31)) return ATTN_ERR_INVALID_ARG;

    // The least-traffic tiling among those the SM runs at the full tensor rate.
    Candidate best{0, 0, 0, 0.0, false, false};
    const int qs[] = {1, 2, 3, 4};
    const int bcs[] = {64, 128, 256};
    for (int q : qs)
        for (int bc : bcs) {
            const Candidate c = evaluate(N, d, causal, q, bc);
            if (!c.fits || !c.full_rate) continue;
            // less traffic first; on a tie (short sequences, where every tiling
            // streams K/V once) more resident query rows, then the larger K/V
            // tile (fewer pipeline steps)
            const bool tie = std::fabs(c.l2_bytes - best.l2_bytes) <= best.l2_bytes * 1e-12;
            if (!best.fits || (!tie && c.l2_bytes < best.l2_bytes) ||
                (tie && (c.q > best.q || (c.q == best.q && c.Bc > best.Bc))))
                best = c;
        }
    // The kernel is compiled for one tiling; the planner must arrive at it.
    if (!best.fits || best.q != kQTiles || best.Bc != kBc) return ATTN_ERR_UNSUPPORTED;
    out->io_opt_q_tiles = best.q;
    out->io_opt_Bc = best.Bc;
    out->io_opt_l2_bytes = static_cast<double>(B) * H * best.l2_bytes + static_cast<double>(B) * H * 4.0 * N;

    const long long BH = static_cast<long long>(B) * H;
    const int q_tiles = (N + kBr - 1) / kBr;
    const int pairs = (q_tiles + kQTiles - 1) / kQTiles;
    const long long units = BH * pairs;

    out->Br = kBr;
    out->Bc = kBc;
    out->q_tiles = kQTiles;
    out->kv_stages = kv_stages_for(d);
    out->tmem_cols = kTmemCols;
    out->smem_bytes = smem_bytes_for(d);
    out->threads = kThreads;
    out->num_units = static_cast<int>(units);
    out->grid = static_cast<int>(units < num_sms ? units : num_sms);

    // Causal scheduling groups: as many heads as keep their K and V within
    // about half of the 126 MB L2.
    const double kv_head_bytes = 2.0 * N * d * 2.0;
    long long g = static_cast<long long>(64.0 * 1024 * 1024 / kv_head_bytes);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    out->heads_per_group = static_cast<int>(g);

    const double nd = static_cast<double>(N) * d;
    out->flops = 4.0 * BH * static_cast<double>(N) * N * d * (causal ? 0.5 : 1.0);
    out->io_bytes = BH * (2.0 * 4.0 * nd + 4.0 * N);
    out->l2_bytes = BH * l2_traffic_per_head(N, d, kQTiles, causal) + BH * 4.0 * N;

    // Heads whose K/V are streamed at the same time.  Non-causal, head-major:
    // the grid's CTAs cover `grid` consecutive units, which span at most
    // ceil(grid / pairs) + 1 heads.  Causal: one group of heads, and the first
    // head of the next group, whose heaviest units start while the current
    // group's lightest ones end.
    long long heads_in_flight = causal ? g + 1 : (out->grid + pairs - 1) / pairs + 1;
    if (heads_in_flight > BH) heads_in_flight = BH;
    out->kv_in_flight_bytes = static_cast<double>(heads_in_flight) * kv_head_bytes;
    out->l2_fit = out->kv_in_flight_bytes <= kL2KvBudget ? 1.0 : kL2KvBudget / out->kv_in_flight_bytes;
    // HBM: K/V once per head.  A head's units run in waves of grid /
    // heads_in_flight CTAs; the first wave streams the head's K/V in near
    // lockstep, and each later wave re-reads the share of it that L2 no longer
    // holds.
    const double per_head_ctas = static_cast<double>(out->grid) / heads_in_flight;
    const double waves = per_head_ctas > 0 ? static_cast<double>(pairs) / per_head_ctas : 1.0;
    const double rereads = waves > 1.0 ? (waves - 1.0) * (1.0 - out->l2_fit) : 0.0;
    out->hbm_bytes = out->io_bytes + BH * kv_head_bytes * rereads;
    return ATTN_OK;
}
