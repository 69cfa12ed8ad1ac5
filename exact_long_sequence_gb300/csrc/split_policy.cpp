// Work schedule of a forward launch (host only): the K/V split of the units and
// the dynamic schedule.  See split_policy.h.
#include "split_policy.h"

#include <algorithm>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "plan.h"

namespace elsattn {

// Units the split policy considers (a launch with more units than SMs is not split).
static constexpr int kMaxUnitsForSplit = 1024;

// Per-item cost besides its K/V steps (Q load, pipeline fill, epilogue), in K/V
// steps of a query-tile pair (one step measured at about 1.2 us).
constexpr int kItemSteps = 2;
// Cost of the combine kernel (measured: about 4 us).
constexpr int kCombineSteps = 4;
// Whether causal launches with fewer units than SMs may split under the
// dynamic schedule (compile-time switch for measurements).
#ifndef ELS_SPLIT_DYNAMIC
#define ELS_SPLIT_DYNAMIC 1
#endif
// The estimate overstates what dynamic claiming gains (measured on a GB300:
// predicted -28 % / -18 % / -7 % against the best static choice, measured
// -7 % / -8 % / +9 % on causal B1 H8 N4096 d64 / B3 H1 N7000 d64 /
// B1 H4 N6000 d128), so a dynamic split is taken only when its estimate is at
// most this fraction of the best static one.
constexpr double kDynamicMargin = 0.85;

// Greedy list scheduling of work items of the given costs (in order) on `grid`
// CTAs: CTA i starts with item i, then every further item goes to the CTA that
// becomes free first, as the dynamic schedule's counter hands them out.
// Returns the time the last CTA finishes.
static int greedy_makespan(const int* cost, int items, int grid) {
    std::priority_queue<int, std::vector<int>, std::greater<int>> free_at;
    int i = 0;
    for (; i < items && i < grid; ++i) free_at.push(cost[i]);
    int end = 0;
    for (; i < items; ++i) {
        const int t = free_at.top();
        free_at.pop();
        free_at.push(t + cost[i]);
    }
    while (!free_at.empty()) {
        end = free_at.top() > end ? free_at.top() : end;
        free_at.pop();
    }
    return end;
}

// The work schedule of attn_fwd_split for a launch on num_sms SMs; one K/V
// step is one K/V tile for a query-tile pair.
//   - More causal units than SMs: the dynamic schedule, no split.
//   - More non-causal (equal) units than SMs: the units of the last, partial
//     wave are split so that their segments spread over all SMs.
//   - Fewer units than SMs: the heaviest units (a prefix in the kernel's
//     schedule order, decode_unit) are cut into s segments.  Either the split
//     stays one wave on the SMs the units leave idle (static), or, for causal
//     launches, any number of units are split and the CTAs claim the items
//     dynamically, heaviest first (greedy_makespan estimates it).
// A unit takes s segments only when s (s - 1) < n0 (see decode_item).  The
// estimate with the least time wins; no split when none beats the unsplit one.
static KvSplit choose_kv_split_uncached(const attn_plan_t& plan, int num_sms, int BH, int N, int causal) {
    KvSplit best{1, 0, 0, false};
    const int units = plan.num_units;
    if (units < 1) return best;
    if (units >= num_sms) {
        if (causal) return KvSplit{1, 0, 0, units > num_sms};
        // The static stride gives every CTA q = units / num_sms units and R =
        // units % num_sms CTAs one more, a last wave that leaves the other SMs
        // idle.  Splitting those R units into s segments spreads the last wave
        // over all SMs: the first units - R items are whole (q per CTA), then
        // come R * s segments in turn.
        const int L = (N + kBc - 1) / kBc;  // K/V steps of every unit
        const int q = units / num_sms, R = units % num_sms;
        if (R == 0) return best;
        int best_cost = (q + 1) * (L + kItemSteps);
        for (int s = 2; s <= kMaxKvSplit; ++s) {
            if (s * (s - 1) >= L) break;
            const int pieces_per_sm = (R * s + num_sms - 1) / num_sms;
            const int cost = q * (L + kItemSteps) + pieces_per_sm * ((L + s - 1) / s + kItemSteps) + kCombineSteps;
            if (cost < best_cost) {
                best_cost = cost;
                best = KvSplit{s, R, units - R, false};
            }
        }
        return best;
    }
    if (units > kMaxUnitsForSplit) return best;
    const int nq = (N + kBr - 1) / kBr, nkv = (N + kBc - 1) / kBc, pairs = (nq + 1) / 2;
    const int G = plan.heads_per_group > 0 ? plan.heads_per_group : 1;
    std::vector<int> n0(units), n1(units);
    int longest = 0;
    for (int u = 0; u < units; ++u) {
        int pair;
        if (!causal) {
            pair = u % pairs;
        } else {
            const int g = u / (G * pairs), r = u - g * G * pairs;
            const int heads_here = (BH - g * G) < G ? (BH - g * G) : G;
            pair = pairs - 1 - r / heads_here;
        }
        const int q0 = 2 * pair;
        n0[u] = causal ? (q0 + 1 < nkv ? q0 + 1 : nkv) : nkv;
        n1[u] = causal ? (q0 + 2 < nkv ? q0 + 2 : nkv) : nkv;
        if (n1[u] > longest) longest = n1[u];
    }
    int best_cost = longest + kItemSteps;
    // the static candidates first (one wave on the idle SMs), then the dynamic
    // ones, which must beat the best static estimate by the margin
    for (int s = 2; s <= kMaxKvSplit; ++s) {
        int Umax = 0;  // the longest prefix of units that can take s segments
        while (Umax < units && s * (s - 1) < n0[Umax]) ++Umax;
        const int U1 = std::min(Umax, (num_sms - units) / (s - 1));
        if (U1 <= 0) continue;
        int c = 0;
        for (int u = 0; u < units; ++u) {
            const int steps = u < U1 ? (n1[u] + s - 1) / s : n1[u];
            c = std::max(c, steps + kItemSteps);
        }
        c += kCombineSteps;
        if (c < best_cost) {
            best_cost = c;
            best = KvSplit{s, U1, 0, false};
        }
    }
    if (!causal || !ELS_SPLIT_DYNAMIC) return best;
    const int static_cost = best_cost;
    std::vector<int> cost(units * kMaxKvSplit);
    for (int s = 2; s <= kMaxKvSplit; ++s) {
        int Umax = 0;
        while (Umax < units && s * (s - 1) < n0[Umax]) ++Umax;
        // dynamic: every prefix length at which the split units' length changes
        for (int U = 1; U <= Umax; ++U) {
            if (U < Umax && n1[U] == n1[U - 1]) continue;
            int items = 0;
            for (int u = 0; u < units; ++u) {
                if (u < U) {
                    const int c = (n1[u] + s - 1) / s;
                    for (int seg = 0; seg < s; ++seg) {
                        const int jb = seg * c, je = std::min(n1[u], jb + c);
                        cost[items++] = (je - jb) + kItemSteps;
                    }
                } else {
                    cost[items++] = n1[u] + kItemSteps;
                }
            }
            const int c = greedy_makespan(cost.data(), items, std::min(items, num_sms)) + kCombineSteps;
            if (c < best_cost && c <= kDynamicMargin * static_cost) {
                best_cost = c;
                best = KvSplit{s, U, 0, true};
            }
        }
    }
    return best;
}

// The choice for a shape is computed once and kept (the dynamic candidates
// take a few hundred simulations of the item schedule).
KvSplit choose_kv_split(const attn_plan_t& plan, int num_sms, int BH, int N, int causal) {
    static std::mutex m;
    static std::map<std::tuple<int, int, int, int, int, int>, KvSplit> cache;
    const auto key = std::make_tuple(BH, N, plan.heads_per_group, plan.num_units, causal, num_sms);
    {
        std::lock_guard<std::mutex> lock(m);
        const auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const KvSplit s = choose_kv_split_uncached(plan, num_sms, BH, N, causal);
    std::lock_guard<std::mutex> lock(m);
    if (cache.size() >= 4096) cache.clear();
    cache.emplace(key, s);
    return s;
}

size_t split_part_o_bytes(const KvSplit& s, int d) {
    if (s.segs <= 1) return 0;
    return align256(static_cast<size_t>(s.units) * s.segs * (2 * kBr) * d * 4);
}

size_t split_part_lse_bytes(const KvSplit& s) {
    return s.segs > 1 ? align256(static_cast<size_t>(s.units) * s.segs * (2 * kBr) * 4) : 0;
}

}  // namespace elsattn
