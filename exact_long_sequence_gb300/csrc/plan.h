// Tile geometry shared by the planner (host) and the kernel (device).
//
// The kernel keeps kQTiles query tiles of kBr rows resident per CTA and
// streams K/V tiles of kBc keys through a shared-memory ring.  These numbers
// are what the planner's I/O count selects for an sm_103 SM at both head
// dimensions (plan.cpp, which checks that it does); they are compile-time
// constants here because the kernel is specialised on them.
#pragma once

#include <cstdint>

namespace elsattn {

constexpr int kBr = 128;          // query rows per tile: the tcgen05 M = 128, one TMEM lane per row
constexpr int kBc = 128;          // keys per K/V tile: N of S = Q K^T, K of O += P V
constexpr int kQTiles = 2;        // query tiles per CTA, processed in ping-pong
constexpr int kThreads = 384;     // warp 0 TMA, warp 1 MMA, warps 4-7 / 8-11 softmax of tile 0 / 1
constexpr int kTmemCols = 512;    // S0 | S1 | O0 | O1 (P aliases the first half of S)
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per CTA on sm_100-family SMs
constexpr int kSmemAlign = 1024;    // slack to align the tiles to the 1024-byte swizzle atom
constexpr int kFixedBarriers = 19;  // mbarriers besides the two per K/V stage
constexpr int kFlagBytes = 16;      // TMEM base address slot, abort flag, two work-item slots
constexpr int kMaxKvSplit = 4;      // most K/V segments a unit is cut into

// Bytes of one [128 x d] tile of `esize`-byte elements (Q, K and V tiles all
// have this size since kBr == kBc): bf16 (esize 2) by default, E4M3 (esize 1)
// for the FP8 forward.
constexpr int tile_bytes(int d, int esize = 2) { return kBr * d * esize; }

// Bytes besides the tiles: alignment slack, mbarriers, flags.
constexpr int overhead_bytes(int stages) { return kSmemAlign + (2 * stages + kFixedBarriers) * 8 + kFlagBytes; }

// Deepest K/V ring that fits next to the resident query tiles, capped at 8.
constexpr int kv_stages_for(int d, int esize = 2) {
    return ((kSmemLimit - overhead_bytes(0) - kQTiles * tile_bytes(d, esize)) / (tile_bytes(d, esize) + 16)) > 8
               ? 8
               : ((kSmemLimit - overhead_bytes(0) - kQTiles * tile_bytes(d, esize)) / (tile_bytes(d, esize) + 16));
}

constexpr int smem_bytes_for(int d, int esize = 2) {
    return overhead_bytes(kv_stages_for(d, esize)) + kQTiles * tile_bytes(d, esize) +
           kv_stages_for(d, esize) * tile_bytes(d, esize);
}

static_assert(kv_stages_for(128) >= 3, "d=128 ring too shallow");
static_assert(smem_bytes_for(128) <= kSmemLimit && smem_bytes_for(64) <= kSmemLimit, "smem");
// Two CTAs must never share an SM (each allocates all 512 TMEM columns).
static_assert(2 * smem_bytes_for(64) > 233472 && 2 * smem_bytes_for(128) > 233472, "1 CTA/SM");
static_assert(2 * smem_bytes_for(128, 1) > 233472, "1 CTA/SM (E4M3)");

}  // namespace elsattn
