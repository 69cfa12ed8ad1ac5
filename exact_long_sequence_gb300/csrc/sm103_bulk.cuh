// Bulk-copy building blocks used by the backward, beside the tile loads of
// sm103_ptx.cuh: a plain (untiled) bulk load into shared memory, and the
// tiled bulk reduce-add from shared memory into global memory with its
// completion groups.  Written from the public PTX ISA.
#pragma once

#include <cstdint>

namespace elsattn {

// `bytes` (a multiple of 16) from global `src` to shared `dst` (both 16-byte
// aligned); completion counted in bytes on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Element-wise fp32 add of a shared-memory box into the global tensor of
// `tmap` at coordinates {c0, c1, c2}; parts of the box outside the tensor are
// dropped.  Tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace elsattn
