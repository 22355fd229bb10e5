// C ABI of the ragged log-probability library (declared in include/lp_ragged.h).
//
// Host side: argument checks, launch-shape choice (persistent grid = SMs x
// resident CTAs), and the workspace layout. Every step of the path runs in the
// kernels of lp_kernels.cuh.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "lp_kernels.cuh"
#include "lp_ragged.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr uint32_t kMaxCtasPerSm = 4;           // launch cap; sizes the workspace
constexpr uint32_t kMinPieceVec = 1024;         // 16 KB of logits per warp at least
constexpr uint32_t kMinSplitVec = 2688;         // 42 KB of logits per row-queue piece at least
constexpr uint32_t kSplitRowVec = 12288;        // rows shorter than 192 KB are not split
constexpr uint32_t kMaxSplit = 64;              // pieces per row in the row-queue kernel
constexpr uint32_t kStageOffsetsMax = 2048;     // stage off/out_off in smem when B+1 <= this
constexpr uint32_t kUnroll = LP_UNROLL;
constexpr uint32_t kStages = LP_STAGES;
constexpr size_t kRingBytes = lpk::ring_bytes<kUnroll, kStages>();
// Largest dynamic shared memory a launch asks for: the rings + staged offsets (input
// positions, output rows, logits rows when they differ) and echo flags.
constexpr size_t kMaxDynSmem = kRingBytes + 3 * kStageOffsetsMax * 4 + kStageOffsetsMax;
constexpr int kQW = lpk::kQueueWarps;  // warps per CTA of the row-queue kernel
constexpr int kQS = lpk::kQueueStages;
constexpr int kQU = lpk::kQueueUnroll;
constexpr size_t kQueueRingBytes = (size_t)kQW * kQS * kQU * 512;
constexpr size_t kMaxDynSmemQueue = kQueueRingBytes + 3 * kStageOffsetsMax * 4 + kStageOffsetsMax;
// Dynamic shared memory the row-queue kernel may ask for next to its ~17 KB of static
// shared memory (227 KB per CTA in all).
constexpr size_t kQueueDynSmemBudget = 208 * 1024;
#ifndef LP_PDL
#define LP_PDL 1  // launch the row kernel as a programmatic dependent of the plan
#endif
// (levels 0 | 1..5 | 6) x (warp ranges | row queue | row queue in a one-call step)
// x (plain | extended inputs). The step's row-queue instantiation holds the code that
// streams before the plan has finished; the others compile without it.
constexpr int kKinds = 3;
constexpr int kVariants = 3 * kKinds * 2;
enum Kind { kWarpRanges = 0, kRowQueue = 1, kRowQueueStep = 2 };

struct DeviceInfo {
    bool ready = false;
    bool smem_attr[kVariants] = {};
    int sms = 0;
    int occ[kVariants] = {};
    size_t occ_smem[kVariants] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using RowsKernel = void (*)(lpk::RowsParams);

template <bool EXT>
RowsKernel variant_kernel(int v) {
    switch (v) {
        case 0: return &lpk::k_rows<1, false, kUnroll, kStages, EXT>;
        case 1: return &lpk::k_rows<1, true, kUnroll, kStages, EXT>;
        case 2: return &lpk::k_rows<2, true, kUnroll, kStages, EXT>;
        case 3: return &lpk::k_rows_cta<1, false, kQU, kQS, kQW, EXT, false>;
        case 4: return &lpk::k_rows_cta<1, true, kQU, kQS, kQW, EXT, false>;
        case 5: return &lpk::k_rows_cta<2, true, kQU, kQS, kQW, EXT, false>;
        case 6: return &lpk::k_rows_cta<1, false, kQU, kQS, kQW, EXT, true>;
        case 7: return &lpk::k_rows_cta<1, true, kQU, kQS, kQW, EXT, true>;
        default: return &lpk::k_rows_cta<2, true, kQU, kQS, kQW, EXT, true>;
    }
}

// Variant v = levels class + 3 * kind + 9 * extended.
constexpr int kPerExt = 3 * kKinds;
RowsKernel variant_kernel(int v) {
    return v >= kPerExt ? variant_kernel<true>(v - kPerExt) : variant_kernel<false>(v);
}
Kind kind_of(int v) { return (Kind)((v % kPerExt) / 3); }
bool is_queue(int v) { return kind_of(v) != kWarpRanges; }
int block_threads(int v) { return is_queue(v) ? kQW * 32 : lpk::kThreads; }
const void* variant_fn(int v) { return reinterpret_cast<const void*>(variant_kernel(v)); }

int variant_of(uint32_t levels) { return levels == 0 ? 0 : (levels < 6 ? 1 : 2); }

// The row kernel for at most r_max scored rows of V logits (R <= min(T, T_logits) is all
// the host knows before the plan has run). The row queue pays a fixed cost per task (its
// ring restarts, the CTA's merges), the warp ranges stream on across rows but bound the
// top-k by one warp's values only; measured on next-token shapes and the workloads:
// - up to three rows per SM: the row queue (every row starts at once);
// - rows of 60 KB or more, up to seven per SM: the row queue (128 KB rows: 6.5 per SM
//   33.1 against 34.8 us, 8 per SM 38.3 against 33.8 us);
// - rows of 384 KB or more with K <= 31, any count: the row queue (500 KB rows at 50 per
//   SM 541 against 569 us; the mixed workload's 594 KB rows 476 against 506 us; but
//   250 KB rows at 16 per SM 104 against 98 us, and top-63 over 1 MB rows 3.60 against
//   3.23 ms);
// - otherwise warp ranges. LP_RAGGED_KERNEL=warp|queue forces one (a test hook).
bool use_row_queue(uint32_t r_max, uint32_t V, uint32_t levels, int sms) {
    const char* force = std::getenv("LP_RAGGED_KERNEL");
    if (force && std::strcmp(force, "warp") == 0) return false;
    if (force && std::strcmp(force, "queue") == 0) return true;
    const uint64_t row_bytes = (uint64_t)V * 4u, per_sm = (uint64_t)sms;
    if (r_max <= 3u * per_sm) return true;
    if (row_bytes >= 60u * 1024u && r_max <= 7u * per_sm) return true;
    return levels >= 1 && levels <= 5 && row_bytes >= 384u * 1024u;
}

bool device_info(int* dev_out, DeviceInfo** info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return false;
        d.sms = sms;
        d.ready = true;
    }
    *dev_out = dev;
    *info = &d;
    return true;
}

// Allow the variant's largest dynamic shared memory (once per device); false on failure.
bool set_smem_attr(DeviceInfo* d, int v) {
    if (d->smem_attr[v]) return true;
    const size_t dyn = is_queue(v) ? kMaxDynSmemQueue : kMaxDynSmem;
    if (cudaFuncSetAttribute(variant_fn(v), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    d->smem_attr[v] = true;
    return true;
}

int occupancy(DeviceInfo* d, int v, size_t smem) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!set_smem_attr(d, v)) return 0;
    if (d->occ[v] == 0 || d->occ_smem[v] != smem) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, variant_fn(v), block_threads(v), smem) != cudaSuccess)
            n = 1;
        if (n < 1) n = 1;
        if (n > (int)kMaxCtasPerSm) n = kMaxCtasPerSm;
        d->occ[v] = n;
        d->occ_smem[v] = smem;
    }
    return d->occ[v];
}

// Arrival counters: one u32 word per warp, padded to 256 B.
size_t counters_bytes(uint32_t g_max) { return ((size_t)g_max * 4 + 255) & ~(size_t)255; }

// Largest number of warps a launch can have on a device with `sms` SMs.
uint32_t max_warps(int sms) { return (uint32_t)sms * kMaxCtasPerSm * lpk::kWarps; }

size_t workspace_bytes_for(int sms, uint32_t levels) {
    const uint32_t K = (1u << levels) - 1u;
    const uint32_t nw = max_warps(sms);
    return sizeof(lpk::WsHeader) + counters_bytes(nw) + (size_t)2 * nw * lpk::partial_stride_bytes(K);
}

}  // namespace

extern "C" {

size_t lp_ragged_workspace_size(uint32_t B, uint32_t T, uint32_t V, uint32_t levels) {
    (void)B; (void)T; (void)V;
    if (levels > LP_MAX_LEVELS) return 0;
    int dev;
    DeviceInfo* d;
    if (!device_info(&dev, &d)) return 0;
    return workspace_bytes_for(d->sms, levels);
}

}  // extern "C"

// The plan kernel's launch (lp_ragged_plan without the host copy). With
// validate_only the kernel writes no output offsets (output_row_offsets may be NULL):
// it checks the offsets, counts the rows and clears the status word and counters.
static lp_status plan_launch(const uint32_t* logit_row_offsets, const uint8_t* echo, uint32_t B, uint32_t T,
                             uint32_t* output_row_offsets, void* workspace, size_t workspace_bytes,
                             cudaStream_t s, bool validate_only = false, bool programmatic = false) {
    if (!logit_row_offsets || !echo || (!output_row_offsets && !validate_only)) return LP_ERR_NULL;
    if (!workspace) return LP_ERR_WORKSPACE;
    if (B == 0 || T == 0) return LP_ERR_SHAPE;
    if (((uintptr_t)workspace & 255u) != 0) return LP_ERR_WORKSPACE;
    int dev;
    DeviceInfo* d;
    if (!device_info(&dev, &d)) return LP_ERR_CUDA;
    const uint32_t g_max = max_warps(d->sms);
    if (workspace_bytes < sizeof(lpk::WsHeader) + counters_bytes(g_max)) return LP_ERR_WORKSPACE;
    auto* hdr = static_cast<lpk::WsHeader*>(workspace);
    auto* counters = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + sizeof(lpk::WsHeader));
    uint32_t* oo = validate_only ? nullptr : output_row_offsets;
    if (!programmatic) {
        lpk::k_plan<<<1, lpk::kPlanThreads, 0, s>>>(logit_row_offsets, echo, B, T, oo, hdr, counters, g_max);
    } else {
        // a programmatic dependent of the previous kernel: k_plan waits for it on the device
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(lpk::kPlanThreads);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, lpk::k_plan, logit_row_offsets, echo, B, T, oo, hdr, counters, g_max) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return LP_ERR_CUDA;
        }
    }
    if (cudaPeekAtLastError() != cudaSuccess) { (void)cudaGetLastError(); return LP_ERR_CUDA; }
    return LP_OK;
}

// Header words {status, rows} -> host {rows, status}.
static lp_status copy_rows_and_status(uint32_t* host_rows_and_status, void* workspace, cudaStream_t s) {
    auto* hdr = static_cast<lpk::WsHeader*>(workspace);
    if (cudaMemcpyAsync(host_rows_and_status, &hdr->rows, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(host_rows_and_status + 1, &hdr->status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return LP_ERR_CUDA;
    return LP_OK;
}

extern "C" {

lp_status lp_ragged_plan(const uint32_t* logit_row_offsets, const uint8_t* echo, uint32_t B, uint32_t T,
                         uint32_t* output_row_offsets, uint32_t* host_rows_and_status, void* workspace,
                         size_t workspace_bytes, lp_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const lp_status st = plan_launch(logit_row_offsets, echo, B, T, output_row_offsets, workspace, workspace_bytes, s);
    if (st != LP_OK || !host_rows_and_status) return st;
    return copy_rows_and_status(host_rows_and_status, workspace, s);
}

// The row kernels' launch: writes rows (tuples == nullptr) or, for a vocab shard,
// one row tuple per output row with ids offset by vocab_base.
// The row kernels' host checks (every one that can fail before a launch).
static lp_status compute_checks(const float* logits, uint32_t T_logits, uint32_t V, const uint32_t* logit_row_offsets,
                                const uint32_t* input_row_offsets, uint32_t T, uint32_t B, const uint32_t* tokens,
                                const uint32_t* sampled_tokens, const uint32_t* output_row_offsets,
                                const uint8_t* echo, uint32_t levels, const float* out_logprobs,
                                const uint32_t* out_tokens, const void* tuples, const void* workspace,
                                size_t workspace_bytes, DeviceInfo** dev_info) {
    if (!logits || !logit_row_offsets || !tokens || !sampled_tokens || !output_row_offsets || !echo ||
        (!tuples && (!out_logprobs || !out_tokens)))
        return LP_ERR_NULL;
    if (!workspace) return LP_ERR_WORKSPACE;
    if (levels > LP_MAX_LEVELS) return LP_ERR_LEVELS;
    if (!input_row_offsets && T != T_logits) return LP_ERR_SHAPE;
    if (B == 0 || T == 0 || T_logits == 0 || V == 0 || V >= 0x7FFFFFFFu) return LP_ERR_SHAPE;
    if (((uintptr_t)logits & 3u) != 0) return LP_ERR_SHAPE;
    if (((uintptr_t)workspace & 255u) != 0) return LP_ERR_WORKSPACE;
    int dev;
    if (!device_info(&dev, dev_info)) return LP_ERR_CUDA;
    if (workspace_bytes < workspace_bytes_for((*dev_info)->sms, levels)) return LP_ERR_WORKSPACE;
    return LP_OK;
}

static lp_status compute_impl(const float* logits, uint32_t T_logits, uint32_t V, const uint32_t* logit_row_offsets,
                              const uint32_t* input_row_offsets, uint32_t T, uint32_t B, const uint32_t* tokens,
                              const uint32_t* sampled_tokens, const uint32_t* output_row_offsets, const uint8_t* echo,
                              const float* temperatures, uint32_t levels, float* out_logprobs, uint32_t* out_tokens,
                              void* tuples, uint32_t vocab_base, uint32_t tuple_rows, uint32_t out_rows, bool early,
                              void* workspace, size_t workspace_bytes, lp_stream_t stream) {
    DeviceInfo* d;
    const lp_status chk = compute_checks(logits, T_logits, V, logit_row_offsets, input_row_offsets, T, B, tokens,
                                         sampled_tokens, output_row_offsets, echo, levels, out_logprobs, out_tokens,
                                         tuples, workspace, workspace_bytes, &d);
    if (chk != LP_OK) return chk;

    const uint32_t K = (1u << levels) - 1u;
    const uint32_t W = levels ? (1u << levels) : 1u;
    const uint32_t g_max = max_warps(d->sms);
    unsigned char* ws = static_cast<unsigned char*>(workspace);

    lpk::RowsParams p;
    p.logits = logits;
    p.off = input_row_offsets ? input_row_offsets : logit_row_offsets;
    p.loff = logit_row_offsets;
    p.tau = temperatures;
    p.tuple_out = static_cast<unsigned char*>(tuples);
    p.vocab_base = vocab_base;
    p.tuple_rows = tuple_rows;
    p.tokens = tokens;
    p.sampled = sampled_tokens;
    p.out_off = output_row_offsets;
    p.echo = echo;
    p.out_lp = out_logprobs;
    p.out_tok = out_tokens;
    p.status = &reinterpret_cast<lpk::WsHeader*>(ws)->status;
    p.plan_status = &reinterpret_cast<lpk::WsHeader*>(ws)->plan_status;
    p.counters = reinterpret_cast<uint32_t*>(ws + sizeof(lpk::WsHeader));
    p.partials = ws + sizeof(lpk::WsHeader) + counters_bytes(g_max);
    p.T = T;
    p.T_logits = T_logits;
    p.V = V;
    p.B = B;
    p.K = K;
    p.W = W;
    const bool aligned = (((uintptr_t)logits & 15u) == 0) && (V % 4u == 0);
    p.nq = aligned ? V / 4u : (V + 6u) / 4u;
    p.stride = lpk::partial_stride_bytes(K);
    p.min_piece = kMinPieceVec;
    p.stage_offsets = (B + 1u <= kStageOffsetsMax) ? 1u : 0u;
    p.num_sms = (uint32_t)d->sms;
    p.split = 1;
    p.split_rows = 0;
    p.early = early ? 1u : 0u;
    p.out_rows = out_rows;
    // next-token logits: one logits row per batch and per position
    p.next_token = (T == B && T_logits == B && input_row_offsets == nullptr) ? 1u : 0u;
    p.spread_first = 0;

    const uint32_t staged_arrays = (p.loff != p.off) ? 3u : 2u;
    const size_t smem =
        kRingBytes + (p.stage_offsets ? (size_t)staged_arrays * (B + 1u) * sizeof(uint32_t) + ((B + 3u) & ~3u) : 0);

    // The row kernel by the bound R <= min(T, T_logits) and the row size (use_row_queue;
    // the two kernels give the same result). Plain instantiation unless an extended input
    // is given (it compiles without them).
    const bool ext = input_row_offsets != nullptr || temperatures != nullptr || tuples != nullptr;
    int v = variant_of(levels) + (ext ? kPerExt : 0);
    int occ = occupancy(d, v, smem);
    if (occ == 0) return LP_ERR_CUDA;
    uint32_t grid = (uint32_t)d->sms * (uint32_t)occ;  // occ <= kMaxCtasPerSm
    const uint32_t r_max = T < T_logits ? T : T_logits;
    const bool queue = use_row_queue(r_max, V, levels, d->sms);
    size_t launch_smem = smem;
    unsigned block = lpk::kThreads;
    if (queue) {
        v += 3 * (early ? kRowQueueStep : kRowQueue);
        block = kQW * 32;
        launch_smem = smem - kRingBytes + kQueueRingBytes;
        if (launch_smem > kQueueDynSmemBudget) {  // very many batches: read offsets from global memory
            p.stage_offsets = 0;
            launch_smem = kQueueRingBytes;
        }
        occ = occupancy(d, v, launch_smem);
        if (occ == 0) return LP_ERR_CUDA;
        grid = (uint32_t)d->sms * (uint32_t)occ;
        // split-vocab for small batches: pieces per row so that the tasks number about two per
        // SM, of at least 42 KB each, and only for rows of 192 KB or more (a piece costs a
        // publish, a ticket and a merge, ~5 us, which pays only where one CTA would otherwise
        // stream a long row)
        uint32_t S = (2u * (uint32_t)d->sms) / (r_max ? r_max : 1u);
        const uint32_t by_len = p.nq >= kSplitRowVec ? p.nq / kMinSplitVec : 1u;
        if (S > by_len) S = by_len;
        if (S > kMaxSplit) S = kMaxSplit;
        const char* fs = std::getenv("LP_RAGGED_SPLIT");  // test hook: pieces per row
        if (fs) S = (uint32_t)std::strtoul(fs, nullptr, 10);
        if (S < 1) S = 1;
        if (S > kMaxSplit) S = kMaxSplit;
        p.split = S;
        // a step on next-token logits whose tasks fit the CTAs: no CTA waits for the plan
        p.spread_first = (early && p.next_token && (uint64_t)B * S <= grid) ? 1u : 0u;
        // rows the workspace holds a ticket (after the 2 queue words) and S piece slots for
        const uint32_t by_words = g_max - 2u;
        const uint32_t by_slots = 2u * g_max / S;
        p.split_rows = by_words < by_slots ? by_words : by_slots;
    }
    // Launched as a programmatic dependent of the previous kernel on the stream (normally
    // lp_ragged_plan): its CTAs become resident while the plan runs and wait on device.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = launch_smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = LP_PDL ? 1 : 0;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, variant_kernel(v), p);
    if (err != cudaSuccess) { (void)cudaGetLastError(); return LP_ERR_CUDA; }
    if (cudaPeekAtLastError() != cudaSuccess) { (void)cudaGetLastError(); return LP_ERR_CUDA; }
    return LP_OK;
}

lp_status lp_ragged_compute_ex(const float* logits, uint32_t T_logits, uint32_t V,
                               const uint32_t* logit_row_offsets, const uint32_t* input_row_offsets, uint32_t T,
                               uint32_t B, const uint32_t* tokens, const uint32_t* sampled_tokens,
                               const uint32_t* output_row_offsets, const uint8_t* echo, const float* temperatures,
                               uint32_t levels, float* out_logprobs, uint32_t* out_tokens, void* workspace,
                               size_t workspace_bytes, lp_stream_t stream) {
    return compute_impl(logits, T_logits, V, logit_row_offsets, input_row_offsets, T, B, tokens, sampled_tokens,
                        output_row_offsets, echo, temperatures, levels, out_logprobs, out_tokens, nullptr, 0u, 0u, 0u,
                        false, workspace, workspace_bytes, stream);
}

lp_status lp_ragged_compute(const float* logits, uint32_t T, uint32_t V, const uint32_t* logit_row_offsets,
                            uint32_t B, const uint32_t* tokens, const uint32_t* sampled_tokens,
                            const uint32_t* output_row_offsets, const uint8_t* echo, uint32_t levels,
                            float* out_logprobs, uint32_t* out_tokens, void* workspace, size_t workspace_bytes,
                            lp_stream_t stream) {
    return compute_impl(logits, T, V, logit_row_offsets, nullptr, T, B, tokens, sampled_tokens, output_row_offsets,
                        echo, nullptr, levels, out_logprobs, out_tokens, nullptr, 0u, 0u, 0u, false, workspace,
                        workspace_bytes, stream);
}

lp_status lp_ragged_step(const float* logits, uint32_t T_logits, uint32_t V, const uint32_t* logit_row_offsets,
                         const uint32_t* input_row_offsets, uint32_t T, uint32_t B, const uint32_t* tokens,
                         const uint32_t* sampled_tokens, const uint8_t* echo, const float* temperatures,
                         uint32_t levels, uint32_t* output_row_offsets, uint32_t* host_rows_and_status,
                         float* out_logprobs, uint32_t* out_tokens, uint32_t out_rows, void* workspace,
                         size_t workspace_bytes, lp_stream_t stream) {
    // every check of both launches first, so that an error leaves nothing enqueued
    if (out_rows == 0) return LP_ERR_SHAPE;
    DeviceInfo* d;
    const lp_status chk = compute_checks(logits, T_logits, V, logit_row_offsets, input_row_offsets, T, B, tokens,
                                         sampled_tokens, output_row_offsets, echo, levels, out_logprobs, out_tokens,
                                         nullptr, workspace, workspace_bytes, &d);
    if (chk != LP_OK) return chk;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The reduction directly follows the plan and reads its inputs before the plan has
    // finished: the plan lets it launch only once everything earlier on the stream is done.
    // On next-token logits (one logits row per batch and per position) the plan is itself a
    // programmatic dependent of the previous kernel (it waits for it on the device, so no
    // launch gap) and the reduction streams without reading the offsets first; otherwise
    // the plan is an ordinary launch.
    const bool next_token = T == B && T_logits == B && input_row_offsets == nullptr;
    lp_status st = plan_launch(input_row_offsets ? input_row_offsets : logit_row_offsets, echo, B, T,
                               output_row_offsets, workspace, workspace_bytes, s, false, next_token);
    if (st != LP_OK) return st;
    st = compute_impl(logits, T_logits, V, logit_row_offsets, input_row_offsets, T, B, tokens, sampled_tokens,
                      output_row_offsets, echo, temperatures, levels, out_logprobs, out_tokens, nullptr, 0u, 0u,
                      out_rows, true, workspace, workspace_bytes, stream);
    if (st != LP_OK || !host_rows_and_status) return st;
    return copy_rows_and_status(host_rows_and_status, workspace, s);  // rows, and the step's status
}

uint32_t lp_ragged_tuple_bytes(uint32_t levels) {
    return levels > LP_MAX_LEVELS ? 0u : lpk::partial_stride_bytes((1u << levels) - 1u);
}

lp_status lp_ragged_shard_partials(const float* logits, uint32_t T_logits, uint32_t V_shard, uint32_t vocab_base,
                                   const uint32_t* logit_row_offsets, const uint32_t* input_row_offsets, uint32_t T,
                                   uint32_t B, const uint32_t* tokens, const uint32_t* sampled_tokens,
                                   const uint32_t* output_row_offsets, const uint8_t* echo,
                                   const float* temperatures, uint32_t levels, void* tuples,
                                   uint32_t rows_capacity, void* workspace, size_t workspace_bytes,
                                   lp_stream_t stream) {
    if (!tuples) return LP_ERR_NULL;
    if (rows_capacity == 0) return LP_ERR_SHAPE;
    if (((uintptr_t)tuples & 15u) != 0) return LP_ERR_SHAPE;
    if ((uint64_t)vocab_base + V_shard >= 0x7FFFFFFFull) return LP_ERR_SHAPE;
    return compute_impl(logits, T_logits, V_shard, logit_row_offsets, input_row_offsets, T, B, tokens,
                        sampled_tokens, output_row_offsets, echo, temperatures, levels, nullptr, nullptr, tuples,
                        vocab_base, rows_capacity, 0u, false, workspace, workspace_bytes, stream);
}

lp_status lp_ragged_shard_merge(const void* tuples, uint32_t P, uint32_t rows_capacity, uint32_t V,
                                const uint32_t* output_row_offsets, uint32_t B, const float* temperatures,
                                uint32_t levels, float* out_logprobs, uint32_t* out_tokens, void* workspace,
                                size_t workspace_bytes, lp_stream_t stream) {
    if (!tuples || !output_row_offsets || !out_logprobs || !out_tokens) return LP_ERR_NULL;
    if (!workspace || workspace_bytes < sizeof(lpk::WsHeader)) return LP_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return LP_ERR_WORKSPACE;
    if (levels > LP_MAX_LEVELS) return LP_ERR_LEVELS;
    if (P == 0 || B == 0 || V == 0 || V >= 0x7FFFFFFFu || rows_capacity == 0) return LP_ERR_SHAPE;
    if (((uintptr_t)tuples & 15u) != 0) return LP_ERR_SHAPE;
    int dev;
    DeviceInfo* d;
    if (!device_info(&dev, &d)) return LP_ERR_CUDA;
    lpk::RowsParams p = {};
    p.out_off = output_row_offsets;
    p.tau = temperatures;
    p.out_lp = out_logprobs;
    p.out_tok = out_tokens;
    p.status = &static_cast<lpk::WsHeader*>(workspace)->status;
    p.B = B;
    p.V = V;
    p.K = (1u << levels) - 1u;
    p.W = levels ? (1u << levels) : 1u;
    p.stride = lpk::partial_stride_bytes(p.K);
    const uint32_t per_cta = lpk::kMergeWarps;
    uint32_t grid = (rows_capacity + per_cta - 1) / per_cta;
    const uint32_t cap = (uint32_t)d->sms * 4u;
    if (grid > cap) grid = cap;
    const auto* tp = static_cast<const unsigned char*>(tuples);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (levels == 0)
        lpk::k_shard_merge<1, false><<<grid, per_cta * 32, 0, s>>>(p, tp, P, rows_capacity);
    else if (levels < 6)
        lpk::k_shard_merge<1, true><<<grid, per_cta * 32, 0, s>>>(p, tp, P, rows_capacity);
    else
        lpk::k_shard_merge<2, true><<<grid, per_cta * 32, 0, s>>>(p, tp, P, rows_capacity);
    if (cudaPeekAtLastError() != cudaSuccess) { (void)cudaGetLastError(); return LP_ERR_CUDA; }
    return LP_OK;
}

lp_status lp_ragged_read_status(const void* workspace, uint32_t* host_status, lp_stream_t stream) {
    if (!workspace || !host_status) return LP_ERR_NULL;
    const auto* hdr = static_cast<const lpk::WsHeader*>(workspace);
    if (cudaMemcpyAsync(host_status, &hdr->status, 4, cudaMemcpyDeviceToHost,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LP_ERR_CUDA;
    return LP_OK;
}

extern "C" lp_status lp_ragged_row_kernel(uint32_t T_logits, uint32_t T, uint32_t V, uint32_t levels,
                                          int* kind) {
    if (!kind) return LP_ERR_NULL;
    if (levels > LP_MAX_LEVELS) return LP_ERR_LEVELS;
    int dev;
    DeviceInfo* d;
    if (!device_info(&dev, &d)) return LP_ERR_CUDA;
    *kind = use_row_queue(T < T_logits ? T : T_logits, V, levels, d->sms) ? 1 : 0;
    return LP_OK;
}

const char* lp_ragged_strerror(lp_status status) {
    switch (status) {
        case LP_OK: return "ok";
        case LP_ERR_NULL: return "a required pointer is NULL";
        case LP_ERR_LEVELS: return "levels exceeds 6 (top-k capacity 63)";
        case LP_ERR_SHAPE: return "B, T or V is zero or too large, or logits are not 4-byte aligned";
        case LP_ERR_OFFSETS:
            return "row offsets invalid: empty/decreasing batch, range past T, echo mismatch, or fewer logits "
                   "rows than scored positions";
        case LP_ERR_TOKEN_RANGE: return "an actual or sampled token id is >= V";
        case LP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case LP_ERR_CUDA: return "CUDA launch or copy failed";
        case LP_ERR_TEMPERATURE: return "a temperature is not a positive finite number";
        default: return "unknown lp_status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Allocation-free variant of lp_ragged_compute.
//
// Its scratch (status word, arrival counters, split-row partial tuples) lives in one
// file-scope device array instead of a caller-provided workspace. Every GPU that loads
// this library holds the array until the process exits; all calls on a device share
// it, so calls that overlap on the GPU (two streams, two threads) race and corrupt each
// other's results.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LP_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device. Host code cannot use
// the symbol itself (on the host it names a stand-in object, not device memory).
// Resolved once per device, on the first call made with that device current.
bool noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return false;
        }
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return true;
}

}  // namespace

extern "C" lp_status lp_ragged_compute_noalloc(const float* logits, uint32_t T, uint32_t V,
                                               const uint32_t* logit_row_offsets, uint32_t B,
                                               const uint32_t* tokens, const uint32_t* sampled_tokens,
                                               const uint32_t* output_row_offsets, const uint8_t* echo,
                                               uint32_t levels, float* out_logprobs, uint32_t* out_tokens,
                                               uint32_t* host_status, lp_stream_t stream) {
    if (!logits || !logit_row_offsets || !tokens || !sampled_tokens || !output_row_offsets || !echo ||
        !out_logprobs || !out_tokens)
        return LP_ERR_NULL;
    if (levels > LP_MAX_LEVELS) return LP_ERR_LEVELS;
    int dev;
    DeviceInfo* d;
    if (!device_info(&dev, &d)) return LP_ERR_CUDA;
    const size_t need = workspace_bytes_for(d->sms, levels);
    if (need > (size_t)LP_NOALLOC_SCRATCH_BYTES) return LP_ERR_WORKSPACE;  // GPU has too many SMs for it
    void* scratch = nullptr;
    if (!noalloc_scratch(dev, &scratch)) return LP_ERR_CUDA;
    // Every host check before anything is enqueued: a call that fails one leaves the
    // shared array untouched (another call may still be using it).
    const lp_status chk = compute_checks(logits, T, V, logit_row_offsets, nullptr, T, B, tokens, sampled_tokens,
                                         output_row_offsets, echo, levels, out_logprobs, out_tokens, nullptr,
                                         scratch, LP_NOALLOC_SCRATCH_BYTES, &d);
    if (chk != LP_OK) return chk;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents. The plan kernel, run here to validate
    // only (it writes no output offsets), clears the status word and the arrival counters
    // and sets the offsets bit for a layout lp_ragged_plan rejects, in which case the
    // reduction writes no row, as lp_ragged_compute does after lp_ragged_plan. (The
    // partial tuples are always written before they are read.)
    lp_status st = plan_launch(logit_row_offsets, echo, B, T, nullptr, scratch, LP_NOALLOC_SCRATCH_BYTES, s, true);
    if (st != LP_OK) return st;
    st = lp_ragged_compute(logits, T, V, logit_row_offsets, B, tokens, sampled_tokens, output_row_offsets, echo,
                           levels, out_logprobs, out_tokens, scratch, LP_NOALLOC_SCRATCH_BYTES, stream);
    if (st != LP_OK) return st;
    if (host_status) {
        if (cudaMemcpyAsync(host_status, &static_cast<lpk::WsHeader*>(scratch)->status, 4, cudaMemcpyDeviceToHost,
                            s) != cudaSuccess)
            return LP_ERR_CUDA;
    }
    return LP_OK;
}
