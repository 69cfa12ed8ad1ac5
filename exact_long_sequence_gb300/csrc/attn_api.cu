// C ABI of the exact-attention forward: argument checks, tile plan, TMA
// descriptors, the kernel launch, and the device error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "../../include/exact_attn.h"
#include "api_common.h"
#include "attn_fwd_kernel.cuh"
#include "plan.h"
#include "split_policy.h"

extern "C" int attn_plan_impl(int B, int H, int N, int d, int causal, int num_sms, attn_plan_t* out);

namespace elsattn {
namespace {

// The scale's sign and size as the kernel takes them.  The kernel keeps a
// running maximum of scale * s, so a negative scale runs as |scale| on the
// negated scores (S = Q (-K)^T on the tensor core).  A zero scale (uniform
// weights over the visible keys) runs with the smallest normal fp32 factor in
// the exponents and 0 in the running maximum: every |factor * s| is then far
// below 2^-24, so every exp2 term is exactly 1 in fp32, as it is for a zero
// scale, masked scores still give 0, and LSE = ln(#visible) exactly.
void set_scale(FwdParams& p, float scale) {
    p.negate_scores = scale < 0.f ? 1u : 0u;
    p.scale_log2 = scale == 0.f ? FLT_MIN : std::fabs(scale) * 1.4426950408889634f;
    p.max_scale_log2 = scale == 0.f ? 0.f : p.scale_log2;
}

// Test hook (attn_debug_arm_timeout): a one-shot time limit for the next
// forward launch, which also withholds CTA 0's first Q_0 copy; 0 = not armed.
std::atomic<uint64_t> g_armed_timeout_ns{0};

// Applies and disarms the hook, if armed.
void take_armed_hook(FwdParams& p) {
    const uint64_t t = g_armed_timeout_ns.exchange(0);
    if (t != 0) {
        p.timeout_ns = t;
        p.withhold_first_q = 1u;
    }
}

template <int D, bool CAUSAL, bool DYN = false>
int launch(DeviceState& dev, const attn_plan_t& plan, const CUtensorMap& tq, const CUtensorMap& tk,
           const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream) {
    if constexpr (CAUSAL && !DYN) {
        // causal launches with a schedule counter take the dynamic instantiation
        if (p.sched_counter != nullptr) return launch<D, CAUSAL, true>(dev, plan, tq, tk, tv, p, stream);
    }
    auto kernel = attn_fwd_kernel<D, CAUSAL, DYN>;
    bool& configured = dev.smem_configured[D == 128][CAUSAL][DYN];
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e);
        configured = true;
    }
    // every CTA starts with item blockIdx.x: the grid never exceeds the items
    const int grid = p.num_items < dev.num_sms ? p.num_items : dev.num_sms;
    cudaError_t e;
    if constexpr (DYN) {
        // a programmatic dependent of the counter's zeroing kernel (see there)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(static_cast<unsigned>(plan.threads));
        cfg.dynamicSmemBytes = static_cast<size_t>(plan.smem_bytes);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p)) != cudaSuccess) return cuda_fail(e);
    } else {
        kernel<<<grid, plan.threads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    }
    if (p.kv_split > 1) {
        // programmatic dependent launch: the combine kernel's CTAs may start as the
        // attention kernel's retire, and wait in-kernel for its completion
        const int rows = p.split_units * 2 * kBr;  // the rows of the split units
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((rows + kCombineRowsPerCta - 1) / kCombineRowsPerCta));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        auto combine = p.kv_split == 2 ? attn_fwd_combine_kernel<D, CAUSAL, 2>
                       : p.kv_split == 3 ? attn_fwd_combine_kernel<D, CAUSAL, 3> : attn_fwd_combine_kernel<D, CAUSAL, 4>;
        if ((e = cudaLaunchKernelEx(&cfg, combine, p)) != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
}


// Workspace of attn_fwd_split: [256 B: the schedule counter][O partials][LSE
// partials], each part 256-aligned.
size_t split_workspace_bytes(const KvSplit& s, int d) {
    if (s.segs <= 1 && !s.dynamic) return 0;
    return kCounterBlock + split_part_o_bytes(s, d) + split_part_lse_bytes(s);
}

int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d, int causal,
             float scale, bool allow_split, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
    if (st != ATTN_OK) return st;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    attn_plan_t plan;
    if ((st = attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan)) != ATTN_OK) return st;

    const int BH = B * H;
    const KvSplit split = allow_split ? choose_kv_split(plan, dev->num_sms, BH, N, causal) : KvSplit{1, 0, 0, false};
    const int kv_split = split.segs;
    const bool dynamic = split.dynamic;
    const size_t need = split_workspace_bytes(split, d);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need))
        return ATTN_ERR_INVALID_ARG;
    CUtensorMap tq, tk, tv;
    if ((st = encode_rows_map(&tq, Q, BH, N, d, kBr)) != ATTN_OK || (st = encode_rows_map(&tk, K, BH, N, d, kBc)) != ATTN_OK ||
        (st = encode_rows_map(&tv, V, BH, N, d, kBc)) != ATTN_OK)
        return st;

    FwdParams p;
    p.O = static_cast<__nv_bfloat16*>(O);
    p.LSE = LSE;
    p.error_word = dev->error_word;
    p.timeout_ns = kDefaultTimeoutNs;
    p.N = N;
    p.BH = BH;
    p.num_q_tiles = (N + kBr - 1) / kBr;
    p.num_kv_tiles = (N + kBc - 1) / kBc;
    p.num_pairs = (p.num_q_tiles + 1) / 2;
    p.num_units = plan.num_units;
    p.heads_per_group = plan.heads_per_group;
    set_scale(p, scale);
    p.kv_split = kv_split;
    p.split_first = split.first;
    p.split_units = split.units;
    p.num_items = plan.num_units + split.units * (kv_split - 1);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part_o = kv_split > 1 ? reinterpret_cast<float*>(ws + kCounterBlock) : nullptr;
    p.part_lse = kv_split > 1 ? reinterpret_cast<float*>(ws + kCounterBlock + split_part_o_bytes(split, d)) : nullptr;
    p.sched_counter = dynamic ? reinterpret_cast<int*>(ws) : nullptr;
    if (dynamic) {
        zero_sched_counter_kernel<<<1, 1, 0, stream>>>(reinterpret_cast<int*>(ws));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    take_armed_hook(p);

    if (d == 64)
        return causal ? launch<64, true>(*dev, plan, tq, tk, tv, p, stream)
                      : launch<64, false>(*dev, plan, tq, tk, tv, p, stream);
    return causal ? launch<128, true>(*dev, plan, tq, tk, tv, p, stream)
                  : launch<128, false>(*dev, plan, tq, tk, tv, p, stream);
}

}  // namespace
}  // namespace elsattn

using namespace elsattn;

extern "C" int attn_plan(int B, int H, int N, int d, int causal, int num_sms, attn_plan_t* out) {
    if (!out) return ATTN_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        DeviceState* dev = nullptr;
        int st = device_state(&dev);
        if (st != ATTN_OK) return st;
        num_sms = dev->num_sms;
    }
    return attn_plan_impl(B, H, N, d, causal, num_sms, out);
}

extern "C" int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                        int d, int causal, float scale, cudaStream_t stream) {
    return fwd_impl(Q, K, V, O, LSE, B, H, N, d, causal, scale, false, nullptr, 0, stream);
}

extern "C" size_t attn_fwd_split_workspace_bytes(int B, int H, int N, int d, int causal) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    if (static_cast<long long>(B) * H * N >= (1ll << 31)) return 0;
    DeviceState* dev = nullptr;
    if (device_state(&dev) != ATTN_OK) return 0;
    attn_plan_t plan;
    if (attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan) != ATTN_OK) return 0;
    return split_workspace_bytes(choose_kv_split(plan, dev->num_sms, B * H, N, causal), d);
}

extern "C" int attn_fwd_split_choice(int B, int H, int N, int d, int causal, int num_sms, int* segs,
                                     int* first, int* units, int* dynamic) {
    if (!segs || !first || !units || !dynamic || num_sms < 1) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || static_cast<long long>(B) * H * N >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    attn_plan_t plan;
    const int st = attn_plan_impl(B, H, N, d, causal, num_sms, &plan);
    if (st != ATTN_OK) return st;
    const KvSplit s = choose_kv_split(plan, num_sms, B * H, N, causal);
    *segs = s.segs;
    *first = s.first;
    *units = s.units;
    *dynamic = s.dynamic ? 1 : 0;
    return ATTN_OK;
}

extern "C" int attn_fwd_split_segments(int B, int H, int N, int d, int causal) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    if (static_cast<long long>(B) * H * N >= (1ll << 31)) return 0;
    DeviceState* dev = nullptr;
    if (device_state(&dev) != ATTN_OK) return 0;
    attn_plan_t plan;
    if (attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan) != ATTN_OK) return 0;
    return choose_kv_split(plan, dev->num_sms, B * H, N, causal).segs;
}

extern "C" int attn_fwd_split(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                              int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    return fwd_impl(Q, K, V, O, LSE, B, H, N, d, causal, scale, true, workspace, workspace_bytes, stream);
}

extern "C" size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    const size_t elems = static_cast<size_t>(B) * H * N * d;
    const size_t t = (elems * 2 + 255) & ~static_cast<size_t>(255);
    return 4 * t + static_cast<size_t>(B) * H * N * 4;
}

namespace elsattn {
namespace {

// Streams and events of the host-buffer entry point, one set per device,
// created on first use.  Copies in, kernels and copies out of consecutive
// chunks of (batch, head) pairs run on separate streams so that the transfers
// overlap the computation; rotating compute streams let one chunk's kernel
// start on the SMs the previous chunk's kernel has finished with.
constexpr int kMaxChunks = 8;
constexpr int kCompStreams = 3;
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, comp[kCompStreams] = {};
    cudaEvent_t start = nullptr, done = nullptr, in[kMaxChunks] = {}, out[kMaxChunks] = {};
};
std::mutex g_pipe_mutex;
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        const unsigned f = cudaStreamNonBlocking;
        for (int c = 0; c < kCompStreams; ++c)
            if ((e = cudaStreamCreateWithFlags(&hp.comp[c], f)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamCreateWithFlags(&hp.h2d, f)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.d2h, f)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e);
        for (int c = 0; c < kMaxChunks; ++c)
            if ((e = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
        hp.ready = true;
    }
    *out = &hp;
    return ATTN_OK;
}

}  // namespace
}  // namespace elsattn

extern "C" int attn_fwd_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh, int B, int H,
                             int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    int st = check_args(Qh, Kh, Vh, Oh, LSEh, B, H, N, d, scale);
    if (st != ATTN_OK && st != ATTN_ERR_MISALIGNED) return st;
    if (!workspace || !aligned16(workspace)) return workspace ? ATTN_ERR_MISALIGNED : ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < attn_fwd_host_workspace_bytes(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t t = (bytes + 255) & ~static_cast<size_t>(255);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    uint8_t *q = w, *k = w + t, *v = w + 2 * t, *o = w + 3 * t;
    float* lse = reinterpret_cast<float*>(w + 4 * t);
    const uint8_t *qh = static_cast<const uint8_t*>(Qh), *kh = static_cast<const uint8_t*>(Kh),
                  *vh = static_cast<const uint8_t*>(Vh);
    uint8_t* oh = static_cast<uint8_t*>(Oh);

    // Chunks of (batch, head) pairs: up to kMaxChunks of equal size.
    const int BH = B * H;
    const int chunks = BH < kMaxChunks ? BH : kMaxChunks;
    const int per = (BH + chunks - 1) / chunks;
    const size_t head_bytes = static_cast<size_t>(N) * d * 2;
    const size_t head_lse = static_cast<size_t>(N);

    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* hp = nullptr;
    if ((st = host_pipe(&hp)) != ATTN_OK) return st;
    cudaError_t e;
    // Everything queued here runs after the work already on `stream`, and
    // `stream` continues only after the last copy out.
    if ((e = cudaEventRecord(hp->start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->h2d, hp->start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->d2h, hp->start, 0)) != cudaSuccess)
        return cuda_fail(e);
    // 1. every chunk's copies in, back to back: the two directions share the
    //    host link, and interleaved with the copies out each ran at about two
    //    thirds of its rate alone
    int c = 0;
    for (int h0 = 0; h0 < BH; h0 += per, ++c) {
        const int hn = (BH - h0) < per ? (BH - h0) : per;
        const size_t off = static_cast<size_t>(h0) * head_bytes, len = static_cast<size_t>(hn) * head_bytes;
        if ((e = cudaMemcpyAsync(q + off, qh + off, len, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaMemcpyAsync(k + off, kh + off, len, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaMemcpyAsync(v + off, vh + off, len, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaEventRecord(hp->in[c], hp->h2d)) != cudaSuccess)
            return cuda_fail(e);
    }
    // 2. each chunk's kernel once its inputs are in, on rotating compute streams
    //    so that a chunk's kernel can take the SMs the previous one leaves idle
    c = 0;
    for (int h0 = 0; h0 < BH; h0 += per, ++c) {
        const int hn = (BH - h0) < per ? (BH - h0) : per;
        const size_t off = static_cast<size_t>(h0) * head_bytes;
        const size_t loff = static_cast<size_t>(h0) * head_lse;
        cudaStream_t comp = hp->comp[c % kCompStreams];
        if ((e = cudaStreamWaitEvent(comp, hp->in[c], 0)) != cudaSuccess) return cuda_fail(e);
        if ((st = attn_fwd(q + off, k + off, v + off, o + off, lse + loff, 1, hn, N, d, causal, scale, comp)) !=
            ATTN_OK)
            return st;
        if ((e = cudaEventRecord(hp->out[c], comp)) != cudaSuccess) return cuda_fail(e);
    }
    // 3. the copies out, once every copy in has landed, each after its chunk's kernel
    if ((e = cudaStreamWaitEvent(hp->d2h, hp->in[c - 1], 0)) != cudaSuccess) return cuda_fail(e);
    c = 0;
    for (int h0 = 0; h0 < BH; h0 += per, ++c) {
        const int hn = (BH - h0) < per ? (BH - h0) : per;
        const size_t off = static_cast<size_t>(h0) * head_bytes, len = static_cast<size_t>(hn) * head_bytes;
        const size_t loff = static_cast<size_t>(h0) * head_lse;
        if ((e = cudaStreamWaitEvent(hp->d2h, hp->out[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(oh + off, o + off, len, cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess ||
            (e = cudaMemcpyAsync(LSEh + loff, lse + loff, static_cast<size_t>(hn) * head_lse * 4,
                                 cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess)
            return cuda_fail(e);
    }
    if ((e = cudaEventRecord(hp->done, hp->d2h)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, hp->done, 0)) != cudaSuccess)
        return cuda_fail(e);
    return ATTN_OK;
}

extern "C" int attn_last_device_error(cudaStream_t stream) {
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t word = 0;
    if ((e = cudaMemcpy(&word, dev->error_word, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    if (word != 0 && (e = cudaMemset(dev->error_word, 0, sizeof word)) != cudaSuccess) return cuda_fail(e);
    return word == kDevTimeout ? ATTN_ERR_TIMEOUT : (word == 0 ? ATTN_OK : ATTN_ERR_CUDA);
}

extern "C" int attn_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* attn_strerror(int status) {
    switch (status) {
        case ATTN_OK: return "success";
        case ATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, size out of range, or a scale out of range)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported (head dim must be 64 or 128; device must be sm_103)";
        case ATTN_ERR_MISALIGNED: return "misaligned pointer (tensors need 16-byte alignment, LSE 4-byte)";
        case ATTN_ERR_CUDA: return "CUDA call failed (see attn_last_cuda_error)";
        case ATTN_ERR_TIMEOUT: return "a kernel-side wait ran out of time";
        case ATTN_ERR_NO_DEVICE: return "no CUDA device";
        default: return "unknown status";
    }
}

// ----------------------------------------------------------------- test hook
namespace elsattn {
__global__ void wait_timeout_kernel(uint32_t* error_word, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx ctx{&abort_flag, error_word, timeout_ns};
        mbar_wait(smem_u32(&bar), 0, ctx);  // nobody arrives: gives up after timeout_ns
    }
    __syncthreads();
}
}  // namespace elsattn

extern "C" int attn_debug_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int st = device_state(&dev);
    if (st != ATTN_OK) return st;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(dev->error_word, timeout_ns);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

extern "C" int attn_debug_arm_timeout(uint64_t timeout_ns) {
    if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return ATTN_ERR_INVALID_ARG;
    g_armed_timeout_ns.store(timeout_ns);
    return ATTN_OK;
}

// ----------------------------------------------------- allocation-free entry point
// attn_fwd_noalloc runs the same kernel as attn_fwd for callers that must not
// let the library allocate device memory: an application that reserves all of
// device memory for its own pool up front (a server that hands the rest of HBM
// to its cache), or one on a latency-critical path that cannot afford
// cudaMalloc's implicit device synchronisation.  attn_fwd allocates one small
// block per device on first use for the kernel's error word; here that word
// lives in the fixed array below, compiled into the library, so the call never
// allocates.  Every device that loads the library holds the array until exit.
namespace elsattn {
namespace {
constexpr size_t kNoAllocScratchBytes = 256;           // the array's size: the most any call may use
constexpr size_t kFwdScratchBytes = sizeof(uint32_t);  // what one forward launch uses: its error word
}  // namespace
}  // namespace elsattn

static __device__ __align__(256) uint32_t els_noalloc_scratch[elsattn::kNoAllocScratchBytes / sizeof(uint32_t)];

namespace elsattn {
namespace {

struct NoAllocDevice {
    bool ready = false;
    int num_sms = 0;
    uint32_t* scratch = nullptr;  // device address of els_noalloc_scratch on this device
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Once per device, with that device current: look up the device address of the
// static array (its name in host code is only a stand-in, not an address the
// kernel may use), and set the kernels' shared-memory limit.
int noalloc_device(NoAllocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return ATTN_ERR_NO_DEVICE;
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& s = g_noalloc_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
        const int st = resolve_tensor_map_encoder();
        if (st != ATTN_OK) return st;
        void* ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, els_noalloc_scratch)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaFuncSetAttribute(attn_fwd_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem_bytes_for(64))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn_fwd_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem_bytes_for(64))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn_fwd_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem_bytes_for(128))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(attn_fwd_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem_bytes_for(128))) != cudaSuccess)
            return cuda_fail(e);
        s.scratch = static_cast<uint32_t*>(ptr);
        s.ready = true;
    }
    *out = &s;
    return ATTN_OK;
}

}  // namespace
}  // namespace elsattn

extern "C" int attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                int N, int d, int causal, float scale, cudaStream_t stream) {
    int st = check_args(Q, K, V, O, LSE, B, H, N, d, scale);
    if (st != ATTN_OK) return st;
    // The scratch a launch needs does not grow with B, H, N or d; it must fit the array.
    if (kFwdScratchBytes > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;
    NoAllocDevice* dev = nullptr;
    if ((st = noalloc_device(&dev)) != ATTN_OK) return st;
    attn_plan_t plan;
    if ((st = attn_plan_impl(B, H, N, d, causal, dev->num_sms, &plan)) != ATTN_OK) return st;

    const int BH = B * H;
    CUtensorMap tq, tk, tv;
    if ((st = encode_rows_map(&tq, Q, BH, N, d, kBr)) != ATTN_OK || (st = encode_rows_map(&tk, K, BH, N, d, kBc)) != ATTN_OK ||
        (st = encode_rows_map(&tv, V, BH, N, d, kBc)) != ATTN_OK)
        return st;

    // The array keeps the previous call's contents: the error word must start at zero.
    cudaError_t e = cudaMemsetAsync(dev->scratch, 0, kFwdScratchBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e);

    FwdParams p;
    p.O = static_cast<__nv_bfloat16*>(O);
    p.LSE = LSE;
    p.error_word = dev->scratch;
    p.timeout_ns = kDefaultTimeoutNs;
    p.N = N;
    p.BH = BH;
    p.num_q_tiles = (N + kBr - 1) / kBr;
    p.num_kv_tiles = (N + kBc - 1) / kBc;
    p.num_pairs = (p.num_q_tiles + 1) / 2;
    p.num_units = plan.num_units;
    p.heads_per_group = plan.heads_per_group;
    set_scale(p, scale);
    p.kv_split = 1;
    p.split_first = 0;
    p.split_units = 0;
    p.num_items = plan.num_units;
    p.part_o = nullptr;
    p.part_lse = nullptr;
    p.sched_counter = nullptr;
    take_armed_hook(p);

    if (d == 64) {
        if (causal)
            attn_fwd_kernel<64, true><<<plan.grid, plan.threads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
        else
            attn_fwd_kernel<64, false><<<plan.grid, plan.threads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
    } else {
        if (causal)
            attn_fwd_kernel<128, true><<<plan.grid, plan.threads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
        else
            attn_fwd_kernel<128, false><<<plan.grid, plan.threads, plan.smem_bytes, stream>>>(tq, tk, tv, p);
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

extern "C" int attn_noalloc_last_device_error(cudaStream_t stream) {
    NoAllocDevice* dev = nullptr;
    int st = noalloc_device(&dev);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t word = 0;
    if ((e = cudaMemcpyAsync(&word, dev->scratch, sizeof word, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e);
    if (word != 0 && ((e = cudaMemsetAsync(dev->scratch, 0, sizeof word, stream)) != cudaSuccess ||
                      (e = cudaStreamSynchronize(stream)) != cudaSuccess))
        return cuda_fail(e);
    return word == kDevTimeout ? ATTN_ERR_TIMEOUT : (word == 0 ? ATTN_OK : ATTN_ERR_CUDA);
}
