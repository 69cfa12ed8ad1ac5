// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tile loads, and the tcgen05 family (TMEM allocation, MMA into TMEM, TMEM
// loads/stores, commit-to-mbarrier).  Written from the public PTX ISA; every
// wait here has a time limit so that a broken pipeline reports an error
// instead of hanging the GPU.
#pragma once

#include <cstdint>

namespace elsattn {

// ---------------------------------------------------------------------------
// Error reporting shared by every role of a CTA.
// ---------------------------------------------------------------------------
enum DeviceError : uint32_t {
    kDevOk = 0,
    kDevTimeout = 1,  // an mbarrier wait ran out of time
};

struct WaitCtx {
    volatile uint32_t* abort_flag;  // in shared memory: set once any role gives up
    uint32_t* error_word;           // in global memory: first error code wins
    uint64_t timeout_ns;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// CTA was aborted by another role or if the time limit ran out (in which case
// this call records the timeout and aborts the CTA).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& ctx) {
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

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& ctx) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, ctx);
}

// Bounded wait that ignores the abort flag (used while draining in-flight
// copies on the abort path).  Returns false if the limit ran out.
static __device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA: 3-D tiled load global -> shared, completion counted in bytes on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns (power of two, 32..512); the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05.mma descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor for a tile stored in the 128-byte swizzled
// layout that TMA writes with SWIZZLE_128B (rows of 128 bytes, 8-row swizzle
// atoms of 1024 bytes, atom base 1024-byte aligned).
//   lbo: byte distance between 64-element column blocks (MN-major operands)
//   sbo: byte distance between consecutive 8-row groups
__device__ __forceinline__ uint64_t make_smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t desc = 0;
    desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    desc |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    desc |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    desc |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    desc |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return desc;
}

// Instruction descriptor, kind::f16 with bf16 A and B and an fp32 accumulator.
//   a_mn / b_mn: operand stored MN-major (transposed) instead of K-major.
__host__ __device__ constexpr uint32_t make_idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction-descriptor bit that negates the B operand (bit 14; bit 13 negates A).
constexpr uint32_t kIdescNegateB = 1u << 14;

// Instruction descriptor, kind::f8f6f4 with E4M3 A and B (type code 0) and an
// fp32 accumulator; both operands K-major.
__host__ __device__ constexpr uint32_t make_idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                    // A, B format: E4M3
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 8-bit operands (kind::f8f6f4): K = 32 elements per instruction.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05.ld / tcgen05.st, shape 32x32b: thread i of the warp owns TMEM lane
// (quadrant base + i); consecutive registers are consecutive 32-bit columns.
// ---------------------------------------------------------------------------
#define ELS_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define ELS_U8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                  "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define ELS_I8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                  "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// Issue a 32-column load; the registers are valid only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : ELS_R8(0), ELS_R8(8), ELS_R8(16), ELS_R8(24)
        : "r"(taddr));
}

// Wait for every outstanding tcgen05.ld of this thread.  The registers of the
// loads are passed through so that no use of them can be scheduled earlier.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : ELS_U8(0), ELS_U8(8), ELS_U8(16), ELS_U8(24)
                 :
                 : "memory");
}

// 16-column variants.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : ELS_R8(0), ELS_R8(8)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : ELS_U8(0), ELS_U8(8) : : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        ELS_I8(0), ELS_I8(8), ELS_I8(16), ELS_I8(24)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        ELS_I8(0), ELS_I8(8)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef ELS_R8
#undef ELS_U8
#undef ELS_I8

// An L2 cache policy that keeps the lines it is attached to over others
// (evict last), for data that is read back soon.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global stores carrying an L2 cache policy.
__device__ __forceinline__ void st_global_v4_hint(float* p, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_global_hint(float* p, float a, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(a), "l"(pol) : "memory");
}

// Invalidate one 128-byte line of global memory in L2 without writing it back
// (its contents become undefined): for scratch data that nothing reads again.
__device__ __forceinline__ void l2_discard_line(const void* line128) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(line128) : "memory");
}

// ---------------------------------------------------------------------------
// Scalar helpers
// ---------------------------------------------------------------------------
// One lane of a converged warp (the same lane every time) returns true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Pack two floats as bf16 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic):
//   (x0, x1) = (a0 * b + c, a1 * b + c),  each correctly rounded like fmaf;
//   (s0, s1) += (a0, a1),                  each correctly rounded like a float add.
__device__ __forceinline__ void ffma2(float& x0, float& x1, float a0, float a1, float b, float c) {
    uint64_t r;
    asm("{\n\t.reg .b64 pa, pb, pc;\n\tmov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %3};\n\t"
        "mov.b64 pc, {%4, %4};\n\tfma.rn.f32x2 %0, pa, pb, pc;\n\t}"
        : "=l"(r)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(r));
}
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
    uint64_t r;
    asm("{\n\t.reg .b64 pa, pb;\n\tmov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %4};\n\tadd.rn.f32x2 %0, pa, pb;\n\t}"
        : "=l"(r)
        : "f"(s0), "f"(s1), "f"(a0), "f"(a1));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(r));
}

// Four floats -> four E4M3 bytes (round to nearest, saturating), x0 in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

}  // namespace elsattn
