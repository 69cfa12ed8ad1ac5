/*
 * exact_attn.h - C ABI of the GB300 (sm_103a) exact self-attention forward.
 *
 * The operation is the attention graph of "From Attention Graph to
 * FlashAttention - A Memory-Centric Compilation Approach in AICF", section 1
 * (Introduction): the query-key products, masked, normalised row by row with
 * a softmax and applied to the values,
 *     O = softmax(mask(scale * Q K^T)) V,
 * plus the per-row log-sum-exp
 *     LSE_i = ln sum_j exp(scale * q_i . k_j)   (over the keys the mask keeps).
 * It is computed as the streaming pass of section 3 of that page: a query
 * tile stays on chip while the K/V tiles stream past it, each contributing its
 * scores to a running softmax and to the output, so the N x N score and
 * probability matrices never reach device memory.  The library is the
 * `flash_attention(Q, K, V)` call of section 4 of the same page, with the
 * optional mask of section 5 as a flag.
 *
 * Conventions for every entry point:
 *   - Q, K, V, O are bf16 tensors laid out [B, H, N, d], contiguous, d fastest;
 *     LSE is fp32 [B, H, N].  All five live in device memory, are owned by the
 *     caller and must not overlap (not checked).
 *   - causal != 0 keeps key j for query i iff j <= i; masked scores are
 *     -infinity, i.e. they drop out of the softmax.
 *   - Calls are asynchronous on `stream` and never synchronise it.
 *   - Errors are returned as attn_status codes; nothing aborts or throws
 *     across this boundary.
 */
#ifndef EXACT_ATTN_H
#define EXACT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, or a scale out of range (see each call) */
    ATTN_ERR_UNSUPPORTED = 2,  /* head dim other than 64/128, or a device other than sm_103 */
    ATTN_ERR_MISALIGNED = 3,   /* a tensor base address is not 16-byte aligned */
    ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed: see attn_last_cuda_error() */
    ATTN_ERR_TIMEOUT = 5,      /* a kernel-side wait ran out of time (reported by attn_last_device_error) */
    ATTN_ERR_NO_DEVICE = 6     /* no CUDA device is visible */
} attn_status;

/*
 * Tile plan chosen by the I/O-count planner (see attn_plan).  Sizes are in
 * elements unless named *_bytes.
 */
typedef struct {
    int Br;               /* query rows per tile (the tcgen05 M dimension) */
    int Bc;               /* keys per streamed K/V tile */
    int q_tiles;          /* query tiles resident per CTA (they share every K/V tile) */
    int kv_stages;        /* depth of the shared-memory K/V ring (one tile per stage) */
    int tmem_cols;        /* tensor-memory columns allocated per CTA */
    int smem_bytes;       /* dynamic shared memory per CTA */
    int threads;          /* threads per CTA */
    int num_units;        /* work units: (batch*head, group of q_tiles query tiles) */
    int grid;             /* persistent CTAs launched (<= SM count) */
    int heads_per_group;  /* causal schedule: heads interleaved per scheduling group */
    double flops;         /* 4*B*H*N^2*d, halved when causal */
    double io_bytes;      /* Theta(N*d) bound: bf16 Q,K,V read + bf16 O, fp32 LSE written once */
    double l2_bytes;      /* modelled L2->SMEM traffic of the chosen tiling */
    double hbm_bytes;     /* modelled HBM traffic: io_bytes, plus the K/V re-reads that miss L2 when
                             the K/V of the heads in flight exceed the L2 budget */
    int io_opt_q_tiles;   /* the tiling with least L2->SMEM traffic among those the SM runs at the   */
    int io_opt_Bc;        /* full tensor rate within its shared memory, tensor memory and registers */
    double io_opt_l2_bytes; /* its modelled L2->SMEM traffic (the kernel runs this tiling) */
    double kv_in_flight_bytes; /* K/V bytes of the heads the schedule streams at the same time */
    double l2_fit;        /* fraction of those that fit the L2 budget (1: every head's K/V read once) */
} attn_plan_t;

/*
 * attn_fwd - O = softmax(scale * Q K^T + mask) V and LSE, for B*H independent
 * (batch, head) problems.
 *   Q, K, V : const bf16 [B,H,N,d] device pointers, 16-byte aligned
 *   O       : bf16 [B,H,N,d] device pointer, 16-byte aligned (written)
 *   LSE     : fp32 [B,H,N] device pointer, 4-byte aligned (written; natural log)
 *   B, H, N : >= 1 with B*H*N < 2^31;  d : 64 or 128
 *   causal  : 0 = no mask, nonzero = causal mask (key j visible to query i iff j <= i)
 *   scale   : any finite value (typically 1/sqrt(d)).  A negative scale is run
 *             as |scale| on the negated scores (the tensor core's negate bit), so
 *             the running maximum tracks the largest scaled score; zero gives
 *             the plain average of the visible values (LSE = ln #visible).
 *   stream  : CUDA stream on the current device (0 = legacy default stream)
 * Returns ATTN_OK when the launch was queued.  Kernel-side timeouts are
 * reported later by attn_last_device_error().
 */
int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
             int causal, float scale, cudaStream_t stream);

/*
 * attn_fwd_host - the same operation on HOST buffers: copies Q, K, V to the
 * device, runs attn_fwd and copies O and LSE back.  The work is split into up
 * to 8 chunks of (batch, head) pairs whose copies in, kernels and copies out
 * run on the library's own per-device streams, so transfers overlap compute:
 * each chunk's kernel starts once its inputs are in, and the copies out start
 * once every copy in has landed (the two directions share the host link).
 * It is ordered after the work already queued on `stream`, and `stream` waits
 * for the last copy out.  Pinned host memory makes the copies asynchronous.
 * The caller synchronises `stream` before reading O / LSE.  Calls from several
 * host threads are serialised while they queue their work.
 *   Qh, Kh, Vh, Oh, LSEh : host pointers with the layouts of attn_fwd
 *   workspace            : device buffer of at least attn_fwd_host_workspace_bytes()
 *                          bytes, 16-byte aligned, owned by the caller
 */
int attn_fwd_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh, int B, int H, int N,
                  int d, int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Device bytes attn_fwd_host needs for its staging copies of Q, K, V, O, LSE. */
size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_fwd_split - attn_fwd with a work schedule chosen for the launch's shape.
 * A work unit is a pair of 128-row query tiles of one (batch, head) against
 * every key they see.
 *   - Fewer units than SMs (few heads, or a causal mask whose longest query
 *     tiles dominate): the K/V range of the heaviest units is cut into
 *     segments, either run on the SMs the units leave idle (one wave), or,
 *     for a causal mask, claimed dynamically with the other units (below),
 *     whichever the host's schedule estimate finds shorter.
 *   - More equal units than SMs (no mask): the units of the last, partial wave
 *     are cut into segments that spread over all SMs.
 *   - More causal units than SMs (units of unequal length): no segments; the
 *     persistent CTAs claim units dynamically, heaviest first, from a counter
 *     in `workspace`.  Every unit is computed exactly as by attn_fwd, so the
 *     outputs are bit-identical to it.
 * A segment is a work item of its own: it writes its partial result (O over
 * the segment's keys, normalised, fp32, and that segment's LSE) to `workspace`
 * (with an L2 evict-last policy), and a second kernel on `stream` merges the
 * segments of each row by
 *     LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s,
 * the combination step of the online softmax (the streaming reformulation of
 * the IO-Aware Algorithms page) applied across segments, then drops the
 * partial rows from L2 without writing them back.  The result is the same
 * operation as attn_fwd, up to floating-point rounding.  Launches on `stream`:
 * a one-thread kernel that zeroes the schedule counter (dynamic schedule only;
 * the attention kernel is its programmatic dependent and waits for it only
 * before its first claim), the attention kernel, and the combine kernel (split
 * launches only).
 *   arguments as attn_fwd, plus
 *   workspace       : device buffer of at least attn_fwd_split_workspace_bytes()
 *                     bytes, 16-byte aligned, owned by the caller, not used by
 *                     other work while this call runs; may be NULL when that
 *                     size is 0 (this call then runs exactly attn_fwd)
 *   workspace_bytes : its size
 * Returns ATTN_ERR_INVALID_ARG when a workspace is needed and it is missing,
 * misaligned or too small; otherwise as attn_fwd.
 */
int attn_fwd_split(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                   int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_fwd_split needs on the current device; 0 when it needs
 * none (or the shape is invalid). */
size_t attn_fwd_split_workspace_bytes(int B, int H, int N, int d, int causal);

/* K/V segments per split unit that attn_fwd_split chooses on the current
 * device: 1 when it does not split, 0 for an invalid shape or no device. */
int attn_fwd_split_segments(int B, int H, int N, int d, int causal);

/*
 * attn_fwd_split_choice - host only: the work split attn_fwd_split would use on
 * a device with num_sms SMs.  Writes the segments per split unit (1: no split),
 * the first split unit and the number of split units (in the kernel's unit
 * order), and whether the dynamic schedule is used (0 or 1).  Returns
 * ATTN_ERR_INVALID_ARG for a null pointer, num_sms < 1 or a shape out of range,
 * ATTN_ERR_UNSUPPORTED for d other than 64 or 128.
 */
int attn_fwd_split_choice(int B, int H, int N, int d, int causal, int num_sms, int* segs, int* first, int* units,
                          int* dynamic);

/*
 * attn_bwd - gradients of attn_fwd for an upstream gradient dO of O:
 *     dV = P^T dO,  dS = P * (dO V^T - D) with D_i = sum_c dO_ic O_ic,
 *     dQ = scale * dS K,  dK = scale * dS^T Q,
 * where P = softmax(scale * Q K^T + mask) is recomputed from Q, K and the
 * forward's LSE instead of being stored (FlashAttention's recomputation in the
 * backward pass, "IO-Aware Algorithms").  No gradient flows into LSE.
 *   Q, K, V, O, dO : const bf16 [B,H,N,d] device pointers (O and LSE as written
 *                    by attn_fwd for the same Q, K, V, causal, scale)
 *   LSE            : const fp32 [B,H,N]
 *   dQ, dK, dV     : bf16 [B,H,N,d] device pointers (written)
 *   workspace      : device buffer of at least attn_bwd_workspace_bytes() bytes,
 *                    16-byte aligned, owned by the caller: the fp32 dQ accumulator
 *                    [B,H,N,d], then the row statistics -scale * D and
 *                    -LSE * log2(e) (negated for the kernel's packed FMAs) on rows
 *                    padded to a multiple of 128 per (batch, head)
 * Same size, alignment, scale and error rules as attn_fwd; asynchronous on `stream`.
 */
int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO, void* dQ,
             void* dK, void* dV, int B, int H, int N, int d, int causal, float scale, void* workspace,
             size_t workspace_bytes, cudaStream_t stream);

/* Device bytes attn_bwd needs as workspace:
 * align256(4*B*H*N*d) + 2 * align256(4*B*H*ceil(N/128)*128); 0 for a
 * non-positive size. */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_plan - host only, launches nothing.  Fills *out with the tiling the
 * planner derives from an I/O count of the two tall-and-skinny products
 * (S = Q K^T and O = P V): the least-traffic tiling among those an sm_103 SM
 * holds (shared memory, tensor memory, registers) and runs at the full tensor
 * rate (the I/O-optimal tiling of the AttenIO abstract, "I/O Analysis is All
 * You Need", ASPLOS 2026).  That is the tiling the kernel is compiled for;
 * ATTN_ERR_UNSUPPORTED if it ever were not.  num_sms <= 0 queries the current
 * device.
 */
int attn_plan(int B, int H, int N, int d, int causal, int num_sms, attn_plan_t* out);

/*
 * attn_last_device_error - synchronises `stream`, then reads and clears the
 * current device's kernel error word.  Returns ATTN_OK or ATTN_ERR_TIMEOUT.
 */
int attn_last_device_error(cudaStream_t stream);

/* The cudaError_t of the most recent ATTN_ERR_CUDA on this thread (0 if none). */
int attn_last_cuda_error(void);

/* A static, human-readable description of a status code. */
const char* attn_strerror(int status);

/*
 * attn_debug_wait_timeout - test hook for the bounded-wait machinery: launches
 * one CTA that waits on an mbarrier nobody arrives on, with the given limit in
 * nanoseconds (<= 10 s).  The kernel gives up, records ATTN_ERR_TIMEOUT in the
 * device error word and exits normally, so the context stays usable; read the
 * result with attn_last_device_error().
 */
int attn_debug_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

/*
 * attn_debug_arm_timeout - test hook for the forward kernel's own abort path
 * (every wait is bounded: a role whose wait runs out records ATTN_ERR_TIMEOUT,
 * the other roles leave their loops, in-flight copies and MMAs are drained
 * and tensor memory is freed before the kernel returns).  Arms a one-shot:
 * the next forward launch of this process (attn_fwd, attn_fwd_split,
 * attn_fwd_noalloc; the first chunk of attn_fwd_host) runs with a wait limit
 * of timeout_ns (1 us .. 1 s) instead of 4 s, and its CTA 0 arms the barrier
 * of its first query-tile copy without issuing the copy, so the wait on it
 * runs out.  That launch's outputs are left partly unwritten; the status is
 * read with attn_last_device_error() (attn_noalloc_last_device_error() after
 * attn_fwd_noalloc).  Launches after it are normal.  ATTN_ERR_INVALID_ARG for
 * a limit out of range.  Not for production use.
 */
int attn_debug_arm_timeout(uint64_t timeout_ns);

/*
 * attn_fwd_noalloc - attn_fwd for callers that must not let the library
 * allocate device memory: applications that reserve all of device memory for
 * their own pool up front (such as a server handing the rest of HBM to its
 * cache), or that cannot afford the implicit device synchronisation of
 * cudaMalloc on their path.  The paper has no counterpart; it is an interface
 * variant of attn_fwd with the same arguments, layouts and results.
 *
 * The kernel's only scratch memory is its 4-byte error word.  attn_fwd keeps
 * it in a block the library allocates on first use; this entry point keeps it
 * instead in a fixed 256-byte array compiled into the library (a static
 * __device__ array), which every device that loads the library holds until
 * exit.  The scratch a call needs does not grow with B, H, N or d; a
 * requirement above 256 bytes would be rejected with ATTN_ERR_INVALID_ARG.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device also does that device's one-time set-up
 *     (it looks up the array's device address and sets the kernel's
 *     shared-memory limit); make that first call before any stream capture.
 *   - Every call shares the one array and clears its error word before the
 *     launch.  Calls that overlap on the GPU (other streams, other threads)
 *     race on that word; serialise them.
 *   - A kernel-side timeout is recorded in the array: read it with
 *     attn_noalloc_last_device_error() before the next call clears it.
 * Returns the same status codes as attn_fwd.
 */
int attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                     int causal, float scale, cudaStream_t stream);

/*
 * attn_noalloc_last_device_error - the error word of attn_fwd_noalloc: waits
 * for `stream`, then reads the word in the fixed array and clears it (an
 * asynchronous copy and memset on `stream`, each waited for); allocates
 * nothing.  Returns ATTN_OK or ATTN_ERR_TIMEOUT for the most recent
 * attn_fwd_noalloc on the current device, or a set-up error (as attn_fwd_noalloc).
 */
int attn_noalloc_last_device_error(cudaStream_t stream);

/*
 * attn_fwd_fp8 - the same forward on 8-bit inputs (the FP8 variant that the
 * quantisation effects of the Neural Circuit Graph (NCG) abstract's
 * performance modelling motivate: halved I/O and twice the tensor-core rate).  Q, K and V are given as
 * E4M3 codes (OCP 8-bit floating point, E4M3: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits) with one fp32 scale per tensor; the real inputs are
 * q_scale * e4m3(Q8) and likewise K, V.  Computes
 *     O = softmax(scale * Q K^T + mask) V   (bf16 [B,H,N,d]),  LSE (fp32 [B,H,N])
 * with S accumulated in fp32 from the exact code products, P rounded to E4M3
 * and staged in shared memory for the second product, and O / l in fp32.
 * Causal launches with more work units than SMs run a dynamic schedule: CTAs
 * claim units, heaviest first, from a counter in `workspace` that this call
 * zeroes on `stream`; each unit is computed as under the static schedule.
 *   Q8, K8, V8 : const uint8 [B,H,N,d] E4M3 codes, device, 16-byte aligned
 *   O, LSE     : as attn_fwd
 *   scale, q_scale, k_scale, v_scale : finite and > 0
 *   workspace  : device buffer of at least attn_fwd_fp8_workspace_bytes(), 16-byte
 *                aligned, owned by the caller, not used by other work while this
 *                call runs: V transposed to [B,H,d,N] (rows padded to 16 bytes),
 *                then the schedule counter, written by this call
 * d must be 128 (ATTN_ERR_UNSUPPORTED otherwise).  Launches on `stream`: the
 * transpose of V, then the attention kernel; under the dynamic schedule a
 * one-thread kernel zeroing the schedule counter comes between them, and a
 * split launch ends with the combine kernel.  The same argument, size and error
 * rules as attn_fwd otherwise.
 */
int attn_fwd_fp8(const void* Q8, const void* K8, const void* V8, void* O, float* LSE, int B, int H, int N, int d,
                 int causal, float scale, float q_scale, float k_scale, float v_scale, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* Device bytes attn_fwd_fp8 needs as workspace: B*H*d*ceil16(N) rounded up to 256,
 * plus 256 for the schedule counter; 0 for a non-positive size. */
size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_softmax_rows - standalone streaming row softmax ("Softmax streaming",
 * section 8 of "From Attention Graph to FlashAttention - A Memory-Centric
 * Compilation Approach in AICF"):
 *     Y[r, i] = exp(X[r, i] - max_j X[r, j]) / sum_j exp(X[r, j] - max_j X[r, j])
 * with the row statistics gathered in one pass by the online-softmax
 * recurrence and fp32 arithmetic.
 *   X, Y      : bf16 [R, N] row-major device arrays, 16-byte aligned (may alias: in place is allowed)
 *   R, N      : 1 <= R < 2^31; N >= 1 and a multiple of 8 (ATTN_ERR_UNSUPPORTED otherwise)
 *   workspace : needed when N > 65536: attn_softmax_rows_workspace_bytes() bytes,
 *               8-byte aligned, owned by the caller; may be NULL otherwise
 * Rows of N <= 65536 are held by one CTA; rows of up to 4 * 65536 by a
 * thread-block cluster of ceil(N / 65536) CTAs that exchange their partial
 * statistics through distributed shared memory: both read X once and write Y
 * once.  Longer rows (or a device that cannot hold the cluster) are handled in
 * segments of 16384 with a second read of X, using the workspace for the
 * per-segment statistics.  Asynchronous on `stream`.
 */
int attn_softmax_rows(const void* X, void* Y, int64_t R, int N, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* Device bytes attn_softmax_rows needs as workspace (0 when N <= 65536). */
size_t attn_softmax_rows_workspace_bytes(int64_t R, int N);

/*
 * attn_layernorm_rows - standalone streaming layer normalisation ("LayerNorm
 * streaming", same section): per row,
 *     mean = sum_j x_j / N,  var = sum_j (x_j - mean)^2 / N,
 *     Y[r, i] = (X[r, i] - mean) / sqrt(var + eps) * gamma[i] + beta[i],
 * the statistics gathered in one pass (running mean and sum of squared
 * deviations, merged pairwise) in fp32.
 *   X, Y        : bf16 [R, N] row-major device arrays, 16-byte aligned (in place is allowed)
 *   gamma, beta : bf16 [N] device arrays, 16-byte aligned
 *   R, N        : 1 <= R < 2^31; N a multiple of 8, at most 65536 (ATTN_ERR_UNSUPPORTED otherwise)
 *   eps         : finite, >= 0
 * Each row is read once and written once.  Asynchronous on `stream`.
 */
int attn_layernorm_rows(const void* X, const void* gamma, const void* beta, void* Y, int64_t R, int N, float eps,
                        cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTN_H */
