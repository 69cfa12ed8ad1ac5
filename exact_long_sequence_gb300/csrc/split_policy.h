// Work schedule of a forward launch: which units are cut into K/V segments,
// and whether the persistent CTAs claim their work items dynamically.  Shared
// by the bf16 forward (attn_fwd_split) and the FP8 forward (attn_fwd_fp8).
#pragma once

#include <cstddef>

#include "../../include/exact_attn.h"

namespace elsattn {

struct KvSplit {
    int segs;      // segments per split unit (1: no split)
    int units;     // how many units are split ...
    int first;     // ... starting at this unit in schedule order
    bool dynamic;  // CTAs claim work items from a counter instead of a fixed stride
};

// The schedule for a launch of `plan` on num_sms SMs (host only; cached per shape).
KvSplit choose_kv_split(const attn_plan_t& plan, int num_sms, int BH, int N, int causal);

// The workspace a split launch needs beyond its schedule counter: [partial O]
// [partial LSE], each 256-byte aligned; 0 for no split.
size_t split_part_o_bytes(const KvSplit& s, int d);
size_t split_part_lse_bytes(const KvSplit& s);

// The 256-byte block of the schedule counter.
constexpr size_t kCounterBlock = 256;

inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace elsattn
