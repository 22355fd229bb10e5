// Kernels of the ragged log-probability path.
//
//  k_plan   one CTA: output_row_offsets = [0, cumsum(echo ? len : 1)], validation,
//           clears the workspace status word and arrival counters.
//  k_rows   persistent, warp-granular stream-K reduction over all scored logits rows.
//
// The operation follows "MAX Python SDK 中 log_probabilities 模块解析" (sections
// "ragged 数据编排：从输入缓冲到 kernel 调用" and "top-k 语义：堆式 kernel 与「采样
// token 兜底」") and the logprob definition of "logprob、finish reason 与 output
// processing" (section "logprob 的数值形态").
//
// Work split. The scored rows form a vector space of R * nq 16-byte vectors (row o,
// vector q). Warp g of the grid owns the contiguous range [start(g), start(g+1)) of
// that space. A row that falls inside one warp's range is finished by that warp
// alone; a row cut by range boundaries is processed as pieces by consecutive warps,
// each of which stores a partial tuple (reference, sum, top-k, target logit) and
// takes a ticket; the warp that takes the last ticket merges the pieces and writes
// the row. Nothing waits on another warp, so there is no inter-warp spin.
//
// Sum-exp in the log2 domain. A lane keeps m (largest logit seen), c = m*k rounded to
// fp32 with k = log2(e)/tau (tau = 1 unless a temperature is given), and
// s = sum 2^(x*k - c): one FFMA, one EX2 and one FADD per logit. A logprob is then
// x/tau - c/(k*tau) - ln(s), formed in fp64: c/k is the reference on the logit scale
// taken with the same fp32 k the sum used, so s = sum exp((x_i - c/k)(1 + d)/tau) with
// |d| <= 2^-24 the rounding of k. That rounding only reweights the terms: ln(s) moves
// by about d times the softmax-weighted mean of (x_i - c/k)/tau (a few units at most),
// far below the fp32 sum's own rounding, and no error grows with |logprob|.
#pragma once

#include <cstdint>

#include "lp_device.cuh"

namespace lpk {

// Tuning knobs (compile-time): 16-byte vectors per lane per block, and the minimum
// resident CTAs per SM the register budget is cut for.
#ifndef LP_UNROLL
#define LP_UNROLL 4
#endif
#ifndef LP_MIN_BLOCKS
#define LP_MIN_BLOCKS 2
#endif
#ifndef LP_STAGES
#define LP_STAGES 5  // blocks per warp in the shared-memory ring
#endif
#ifndef LP_QUEUE_WARPS
#define LP_QUEUE_WARPS 12  // warps per CTA of the row-queue kernel
#endif
#ifndef LP_QUEUE_STAGES
#define LP_QUEUE_STAGES 3  // ring depth of the row-queue kernel
#endif
#ifndef LP_QUEUE_UNROLL
#define LP_QUEUE_UNROLL 4  // vectors per lane per block in the row-queue kernel
#endif
#ifndef LP_NEXT_TOKEN_FAST
#define LP_NEXT_TOKEN_FAST 1  // row queue: next-token compute launches stream before reading offsets
#endif
#ifndef LP_PREFETCH_BEFORE_WAIT
#define LP_PREFETCH_BEFORE_WAIT 1  // row queue, next-token compute launches: L2 prefetch before the wait
#endif
#ifndef LP_EARLY_TRIGGER
#define LP_EARLY_TRIGGER 1  // row kernels let their programmatic dependents launch at once
#endif

// A row kernel lets the next kernel on the stream, when that one is launched as a
// programmatic dependent, become resident on SMs this launch no longer uses (its tail);
// such a dependent waits in griddepcontrol.wait for this launch to finish and flush
// before it reads anything, so this only hides its launch.
__device__ __forceinline__ void trigger_dependents() {
    if (LP_EARLY_TRIGGER) pdl_launch_dependents();
}


constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
#ifndef LP_THR_EVERY
#define LP_THR_EVERY 8
#endif
constexpr uint32_t kThrEvery = LP_THR_EVERY;  // blocks between lane-maximum threshold refreshes (power of 2)
constexpr int kPlanThreads = 1024;
constexpr uint32_t kStatusOffsets = 1u << 4;     // bit of LP_ERR_OFFSETS
constexpr uint32_t kStatusTokenRange = 1u << 5;  // bit of LP_ERR_TOKEN_RANGE
constexpr uint32_t kStatusTemperature = 1u << 8; // bit of LP_ERR_TEMPERATURE

// Workspace: [header 256 B][arrival counters u32 x max warps, zeroed by plan, padded
// to 256 B][partial slots].
struct WsHeader {
    uint32_t status;       // status bits of the plan and of every launch after it
    uint32_t rows;
    uint32_t plan_status;  // the plan's own bits: no row kernel writes it, so every CTA of a
                           // launch reads the same value whatever the others have flagged
    uint32_t reserved[61];
};

// Partial tuple of one piece of a split row (u32 words):
//   [0] reference c  [1] sum s  [2] target logit  [3] 1 if [2] is valid
//   [4, 4+K) top-k logits (sorted)   [4+K, 4+2K) their ids
__host__ __device__ inline uint32_t partial_stride_bytes(uint32_t K) {
    return ((4u + 2u * K) * 4u + 15u) & ~15u;
}

struct RowsParams {
    const float* logits;
    const uint32_t* off;     // input positions (and tokens) per batch
    const uint32_t* tokens;
    const uint32_t* sampled;
    const uint32_t* out_off;
    const uint8_t* echo;
    float* out_lp;
    uint32_t* out_tok;
    uint32_t* status;
    const uint32_t* plan_status;  // the plan's bits alone (WsHeader::plan_status)
    uint32_t* counters;      // per split row (indexed by its first warp): pieces arrived
    unsigned char* partials;
    uint32_t T, V, B, K, W;
    uint32_t nq;             // 16-byte vectors per row in the stream-K space
    uint32_t stride;         // partial slot bytes
    uint32_t min_piece;      // minimum vectors per warp
    uint32_t stage_offsets;  // 1: copy off / out_off / echo to shared memory
    uint32_t num_sms;        // SMs of the device (row-queue kernel: tasks started without a queue)
    // Extended inputs (read only by the EXT instantiations; kept last so the fields above
    // keep their parameter offsets):
    uint32_t T_logits;       // rows of logits
    const uint32_t* loff;    // logits rows per batch: the batch's last positions (== off
                             // when every position has a logits row)
    const float* tau;        // per-batch temperature, or nullptr for raw logits
    unsigned char* tuple_out;  // vocab shard mode: one row tuple per output row instead of
                               // logprobs (nullptr: write rows)
    uint32_t vocab_base;     // vocab shard mode: global id of the shard's column 0
    uint32_t tuple_rows;     // vocab shard mode: rows the tuple buffer holds
    uint32_t split;          // row-queue kernel: pieces per row (1: whole rows)
    uint32_t split_rows;     // row-queue kernel: rows the workspace holds tickets and pieces for
    // Launched by lp_ragged_step directly after its lp_ragged_plan (which ran after all
    // earlier work): with staged offsets the row kernel derives the output rows itself and
    // streams before the plan has finished, waiting for it only before it touches the
    // counters or the status word.
    uint32_t early;
    uint32_t out_rows;       // rows out_lp / out_tok hold (0: not checked)
    // Row-queue kernel, compute launch on next-token logits (T == T_logits == B, every
    // position its own logits row): valid offsets are then 0..B, so output row o is batch
    // o and reads logits row o, and a CTA streams its first task before any offset is read.
    uint32_t next_token;
    // Row-queue kernel, a step on next-token logits with more tasks than SMs but no more
    // than CTAs: every task has a CTA from the start (see k_rows_cta), so no CTA waits for
    // the plan (which clears the queue) before its first task.
    uint32_t spread_first;
};

// Row tuple of one vocab shard (lp_ragged_shard_partials), u32 words:
//   [0] reference c (NaN: the row is invalid)  [1] sum s  [2] target logit
//   [3] target id (bits 0-30; ids >= 2^31 are stored as 2^31-1) | bit 31: this shard
//       holds the target
//   [4, 4+K) top-k logits (sorted)  [4+K, 4+2K) their global ids
// Same stride as a split-row partial slot.
constexpr uint32_t kTupleHolds = 0x80000000u;

// ---------------------------------------------------------------------------------
// Plan: one CTA, chunked block-wide exclusive scan. With out_off == nullptr it only
// validates the offsets, counts the rows and clears the status word and counters.
__global__ void __launch_bounds__(kPlanThreads) k_plan(const uint32_t* __restrict__ off,
                                                       const uint8_t* __restrict__ echo, uint32_t B,
                                                       uint32_t T, uint32_t* __restrict__ out_off,
                                                       WsHeader* hdr, uint32_t* counters,
                                                       uint32_t n_counters) {
    __shared__ uint32_t s_warp[kPlanThreads / 32];
    __shared__ uint32_t s_carry;
    __shared__ uint32_t s_bad;
    // Launched as a programmatic dependent (a next-token step): everything earlier on the
    // stream has finished, the previous row kernel's use of the counters included, before
    // the inputs are read or anything is written (a no-op for an ordinary launch). Only then
    // may the row kernel launch: it reads the logits before it waits for this plan.
    pdl_wait();
    pdl_launch_dependents();  // the row kernel may launch now; it waits for our writes
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) { s_carry = 0; s_bad = 0; }
    for (uint32_t i = tid; i < n_counters; i += kPlanThreads) counters[i] = 0;
    __syncthreads();
    for (uint32_t base = 0; base < B; base += kPlanThreads) {
        const uint32_t i = base + tid;
        uint32_t cnt = 0;
        bool bad = false;
        if (i < B) {
            uint32_t s = off[i], e = off[i + 1];
            if (e <= s || e > T) bad = true;
            else cnt = echo[i] ? (e - s) : 1u;
        }
        uint32_t x = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) s_warp[w] = x;
        if (bad) atomicOr(&s_bad, 1u);
        __syncthreads();
        if (w == 0) {
            uint32_t v = s_warp[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                uint32_t y = __shfl_up_sync(kFull, v, d);
                if (lane >= d) v += y;
            }
            s_warp[lane] = v;  // inclusive over warps
        }
        __syncthreads();
        const uint32_t incl = x + (w ? s_warp[w - 1] : 0u);
        if (i < B && out_off != nullptr) out_off[i] = s_carry + incl - cnt;
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry += incl;
        __syncthreads();
    }
    if (tid == 0) {
        if (out_off != nullptr) out_off[B] = s_carry;
        hdr->rows = s_carry;
        hdr->status = s_bad ? kStatusOffsets : 0u;
        hdr->plan_status = s_bad ? kStatusOffsets : 0u;
    }
}

// ---------------------------------------------------------------------------------
// Stream-K schedule over the vector space [0, Q): warp g owns [start(g), start(g+1)).
__device__ __forceinline__ uint64_t sk_start(uint64_t g, uint64_t Q, uint64_t G) { return g * Q / G; }
// Warp that owns global vector v.
__device__ __forceinline__ uint64_t sk_owner(uint64_t v, uint64_t Q, uint64_t G) {
    return ((v + 1) * G - 1) / Q;
}

// Per-lane running sum in the log2 domain: s = sum of 2^(x*k - c) over the logits seen,
// with a reference c that moves lazily. It is set by the first finite block and moved
// up only when a block's maximum exceeds it by more than kHeadroom (so every term stays
// below 2^kHeadroom: a lane's sum of even 2^60 terms stays below the fp32 range); any
// reference gives the same logsumexp, c + log2(s), with the same relative rounding. m,
// the lane's true running maximum, feeds the top-k bound. A move costs a rescale and the
// block's terms again; with 32 doublings of headroom it is rare even at small
// temperatures (k = log2(e)/tau large).
constexpr float kHeadroom = 32.f;
constexpr float kNoRef = 3.402823466e38f;  // nc before the first finite logit
struct LaneSum {
    float m;   // largest logit seen (-inf: none)
    float nc;  // minus the reference c (kNoRef while m is -inf)
    float2 s;  // sum of 2^(x * k - c), in two halves (packed adds)
    float k;   // log2(e) / temperature
    __device__ __forceinline__ void init(float scale) {
        m = neg_inf();
        nc = kNoRef;
        s = make_float2(0.f, 0.f);
        k = scale;
    }
    __device__ __forceinline__ float ref() const { return -nc; }
    __device__ __forceinline__ float sum() const { return s.x + s.y; }
    // Account for a block whose largest logit is bm, before its terms are added.
    // Without a reference, bm*k + kNoRef is above the headroom for every finite bm
    // (and -inf for an all -inf block, whose terms are then 2^-inf = 0).
    __device__ __forceinline__ void note(float bm) {
        m = fmaxf(m, bm);
        if (fmaf(bm, k, nc) > kHeadroom) rebase(bm);
    }
    __device__ __forceinline__ void rebase(float nm) {
        const float c_new = nm * k;
        if (s.x != 0.f || s.y != 0.f) {
            const float f = ex2(-nc - c_new);
            s = ffma2(s, make_float2(f, f), make_float2(0.f, 0.f));
        }
        nc = -c_new;
    }
    // The terms of one ring block under the current reference, summed in pairs (packed).
    template <int U>
    __device__ __forceinline__ float2 block_terms(const float4 (&v)[U]) const {
        const float2 l2e = make_float2(k, k), mc = make_float2(nc, nc);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float2 y0 = ffma2(make_float2(v[u].x, v[u].y), l2e, mc);
            const float2 y1 = ffma2(make_float2(v[u].z, v[u].w), l2e, mc);
            acc = fadd2(acc, fadd2(make_float2(ex2(y0.x), ex2(y0.y)), make_float2(ex2(y1.x), ex2(y1.y))));
        }
        return acc;
    }
    // Account for a block whose largest logit is bm and add its terms. They are computed
    // under the current reference without waiting for bm, and only in the rare case that
    // the reference moves up (the first finite block, or a maximum beyond the headroom)
    // computed again after the rebase.
    template <int U>
    __device__ __forceinline__ void add_block(const float4 (&v)[U], float bm) {
        m = fmaxf(m, bm);
        float2 acc = block_terms<U>(v);
        if (fmaf(bm, k, nc) > kHeadroom) {
            rebase(bm);
            acc = block_terms<U>(v);
        }
        s = fadd2(s, acc);
    }
    // Add the terms of four logits: two packed FMAs, four EX2, two packed adds.
    __device__ __forceinline__ void add4(const float4& v) {
        const float2 l2e = make_float2(k, k), mc = make_float2(nc, nc);
        const float2 y0 = ffma2(make_float2(v.x, v.y), l2e, mc);
        const float2 y1 = ffma2(make_float2(v.z, v.w), l2e, mc);
        s = fadd2(s, fadd2(make_float2(ex2(y0.x), ex2(y0.y)), make_float2(ex2(y1.x), ex2(y1.y))));
    }
};

template <int SLOTS>
struct WarpList {
    float x[SLOTS];
    uint32_t id[SLOTS];
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) { x[k] = neg_inf(); id[k] = kPadId; }
    }
    // Value of entry K-1, broadcast to the warp.
    __device__ __forceinline__ float kth(uint32_t K) const {
        const uint32_t s = K - 1;
        float v = x[0];
        if constexpr (SLOTS == 2) v = (s >> 5) ? x[1] : x[0];
        return __shfl_sync(kFull, v, s & 31);
    }
    // Merge one candidate per lane (32 in all, any order) into the list.
    __device__ __forceinline__ void insert32(float cx, uint32_t ci, int lane) {
        bitonic_sort32(cx, ci, lane);
        float bx[SLOTS];
        uint32_t bi[SLOTS];
        bx[0] = cx;
        bi[0] = ci;
        if constexpr (SLOTS == 2) { bx[1] = neg_inf(); bi[1] = kPadId; }
        merge_lists<SLOTS>(x, id, bx, bi, lane);
    }
};

// Top-k selection state of one warp: sorted list in registers, a 64-entry candidate
// buffer in shared memory, and the filter threshold thr = the list's K-th value. An
// element below thr cannot enter the top-k (K better elements are already known), so
// only elements >= thr are buffered; a full buffer is sorted into the list.
template <int SLOTS>
struct Selector {
    WarpList<SLOTS> L;
    float* cx;
    uint32_t* ci;
    float thr;
    int cnt;
    uint32_t K;

    __device__ __forceinline__ void init(float* bx, uint32_t* bi, uint32_t k) {
        L.reset();
        cx = bx;
        ci = bi;
        thr = neg_inf();
        cnt = 0;
        K = k;
    }
    __device__ __forceinline__ void flush(int lane) {
        __syncwarp();
        const float x = lane < cnt ? cx[lane] : neg_inf();
        const uint32_t id = lane < cnt ? ci[lane] : kPadId;
        const bool more = lane + 32 < cnt;
        float mx = 0.f;
        uint32_t mi = 0;
        if (more) { mx = cx[lane + 32]; mi = ci[lane + 32]; }
        __syncwarp();
        if (more) { cx[lane] = mx; ci[lane] = mi; }
        __syncwarp();
        L.insert32(x, id, lane);
        cnt = cnt > 32 ? cnt - 32 : 0;
        thr = fmaxf(thr, L.kth(K));
    }
    // The last flush of a piece when at most 8 candidates wait and K <= 8, for callers
    // that read only the list's first 8 entries afterwards: the candidates sorted
    // ascending in lanes 0..7 (a bitonic sort of 8), which pairs them reversed with the
    // list's first 8 for the merge. Entries 8..31 are left unordered. The threshold is
    // not updated.
    __device__ __forceinline__ void flush_top8(int lane) {
        __syncwarp();
        float x = lane < cnt ? cx[lane] : neg_inf();
        uint32_t id = lane < cnt ? ci[lane] : kPadId;
#pragma unroll
        for (int k = 2; k <= 8; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const float ox = __shfl_xor_sync(kFull, x, j);
                const uint32_t oid = __shfl_xor_sync(kFull, id, j);
                const bool lower = (lane & j) == 0;
                const bool asc = (lane & k) == 0;
                const bool ob = better(ox, oid, x, id);
                if ((lower == asc) ? !ob : ob) { x = ox; id = oid; }
            }
        }
        if constexpr (SLOTS == 1) merge_top_rev<8>(L.x[0], L.id[0], x, id, lane);
        cnt = 0;
    }
    // Append the elements of one ring block flagged in mk: bit 4u+k is element k of the
    // lane's vector u, whose value sits at slot_f[128u + 4 lane + k] and whose id is
    // idb + 128u + k. Warp-uniform call, one ballot round per element a lane appends
    // (usually one). An element stays flagged if a flush raises the threshold meanwhile:
    // below the threshold it is only extra work for the next merge.
    __device__ __forceinline__ void append_block(const float* slot_f, uint32_t mk, uint32_t idb, int lane) {
        const uint32_t lt = (1u << lane) - 1u;
        unsigned any = __ballot_sync(kFull, mk != 0);
        while (any) {
            if (mk) {
                const uint32_t e = (uint32_t)(__ffs(mk) - 1);
                mk &= mk - 1;
                const uint32_t off = 128u * (e >> 2) + (e & 3u);
                const int slot = cnt + __popc(any & lt);
                cx[slot] = slot_f[off + 4u * (uint32_t)lane];
                ci[slot] = idb + off;
            }
            cnt += __popc(any);
            if (cnt >= 32) flush(lane);
            any = __ballot_sync(kFull, mk != 0);
        }
    }
    // Append the elements of v flagged in pm (bit k: element k, id id0 + k).
    // Warp-uniform call; the threshold may rise while appending.
    __device__ __forceinline__ void append(const float4& v, uint32_t id0, uint32_t pm, int lane) {
        unsigned any = __ballot_sync(kFull, pm != 0);
        while (any) {
            if (pm) {
                const int k = __ffs(pm) - 1;
                pm &= pm - 1;
                const int slot = cnt + __popc(any & ((1u << lane) - 1u));
                cx[slot] = pick(v, k);
                ci[slot] = id0 + (uint32_t)k;
            }
            cnt += __popc(any);
            if (cnt >= 32) {
                flush(lane);
                pm &= ge_mask(v, thr);
            }
            any = __ballot_sync(kFull, pm != 0);
        }
    }
};

// Load one checked vector: elements outside [0, V) are -inf and masked out.
__device__ __forceinline__ float4 load_checked(const float* rowp, const float* vbase, int64_t q, int a, uint32_t V,
                                               uint32_t qf, uint32_t nfull, uint32_t& vm) {
    if ((uint64_t)(q - qf) < nfull) {
        vm = 0xFu;
        return ldg_stream(vbase + 4 * q);
    }
    float t[4];
    vm = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t e = 4 * q - a + k;
        t[k] = neg_inf();
        if (e >= 0 && e < (int64_t)V) { t[k] = rowp[e]; vm |= 1u << k; }
    }
    return make_float4(t[0], t[1], t[2], t[3]);
}

// Threshold refreshes: blocks 0, 1, 2, 4, then every kThrEvery blocks.
__device__ __forceinline__ bool refresh_due(uint32_t blk) {
    return (blk & (kThrEvery - 1)) == 0 || (blk < kThrEvery && (blk & (blk - 1)) == 0);
}
#ifndef LP_Q_REFRESH
#define LP_Q_REFRESH 1  // row-queue refresh schedule for K <= 7: blocks 0, 4, 8, then every 8
#endif
// Refreshes of the row-queue warps (a CTA-wide table of lane maxima) for K <= 7.
__device__ __forceinline__ bool refresh_due_q(uint32_t blk, int w) {
    if (LP_Q_REFRESH == 1) return (blk & 3u) == 0 && (blk <= 8u || (blk & 7u) == 0);
    if (LP_Q_REFRESH == 2) return blk == 0 || blk == 2 || (blk & 7u) == 4u;
    if (LP_Q_REFRESH == 3) return blk == 0 || blk == 2 || blk == 4 || (blk >= 8u && ((blk + (uint32_t)w) & 7u) == 0);
    return refresh_due(blk);
}

// Candidate mask of one block: bit 4u+k set when element k of vector u is >= thr.
template <int U>
__device__ __forceinline__ uint32_t block_mask(const float4 (&v)[U], float thr) {
    uint32_t mk = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) mk |= ge_mask(v[u], thr) << (4 * u);
    return mk;
}
// Elements of a block that are not ring padding (ids below id_end): all but in a piece's
// partial last block.
template <int U>
__device__ __forceinline__ uint32_t live_mask(uint32_t idb, uint32_t id_end) {
    uint32_t mk = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) mk |= ids_below(idb + 128u * u, id_end) << (4 * u);
    return mk;
}

// Top-k work of one block (U vectors per lane) whose largest element in this lane is
// bm: threshold refreshes on the schedule of refresh_due, then the block's elements
// at or above the threshold go to the candidate buffer. `partial`: the block holds
// ring padding (ids from id_end on), which must not become candidates. slot_f is
// the block's values in shared memory (all lanes), read back by the append.
template <int SLOTS, bool TOPK, int U, int TABW>
__device__ __forceinline__ void select_block(const float4 (&v)[U], float bm, uint32_t blk, bool partial,
                                             uint32_t idb, uint32_t id_end, const float* slot_f, const LaneSum& ls,
                                             Selector<SLOTS>& sel, int lane, uint32_t* shared_thr, float* lane_tab,
                                             int w) {
    if constexpr (TOPK && SLOTS == 1) {
        // The K-th largest of the 32 lanes' running maxima is the value of K distinct
        // elements already seen, so no element below it can be in the top-k: a
        // threshold that follows the warp's true K-th best at the cost of one float
        // sort, refreshed on blocks 0, 1, 2 and 4 (it rises fastest early) and then
        // every kThrEvery blocks (row queue at K <= 7: see refresh_due_q).
        if ((TABW > 0 && sel.K <= 7u) ? refresh_due_q(blk, w) : refresh_due(blk)) {
            float lm = ls.m;
            uint32_t kk = sel.K;
            if constexpr (TABW > 0) {
                volatile float* tab = lane_tab;
                tab[w * 32 + lane] = lm;
                if (kk <= 15u || blk < kThrEvery) {
#pragma unroll
                    for (int j = 0; j < TABW; ++j) lm = fmaxf(lm, tab[j * 32 + lane]);
                } else {
                    // K = 16..31: the K-th of 32 column maxima is nearly their minimum.
                    // Each lane position's second best across the warps instead: the
                    // k-th largest of those stands above 2k distinct elements (the k
                    // second bests and the k bests above them), so k = ceil(K/2). Not on
                    // the first blocks, while few warps have published their maxima
                    // (the second bests are then mostly -inf).
                    float hi = neg_inf(), lo = neg_inf();
#pragma unroll
                    for (int j = 0; j < TABW; ++j) {
                        const float v2 = tab[j * 32 + lane];
                        lo = fmaxf(lo, fminf(hi, v2));
                        hi = fmaxf(hi, v2);
                    }
                    lm = lo;
                    kk = (kk + 1u) >> 1;
                }
            }
            sel.thr = fmaxf(sel.thr, kth_largest32(lm, kk, lane));
            if (shared_thr != nullptr) {  // warps on the same row share their thresholds
                if (lane == 0 && sel.thr != neg_inf()) atomicMax(shared_thr, f2ord(sel.thr));
                sel.thr = fmaxf(sel.thr, ord2f(*(volatile uint32_t*)shared_thr));
            }
        }
        if (__any_sync(kFull, bm >= sel.thr)) {
            uint32_t mk = block_mask<U>(v, sel.thr);
            if (partial) mk &= live_mask<U>(idb, id_end);
            sel.append_block(slot_f, mk, idb, lane);
        }
    }
    if constexpr (TOPK && SLOTS == 2) {
        // K = 63 > 32 lanes: a bound needs 64 distinct elements. With TABW warps on the
        // row, each lane position takes the two best of the warps' lane maxima (elements
        // of two different (warp, lane) streams); the 63rd largest of those 64 values
        // (their second smallest) bounds the top-63. (Tracking a second maximum per lane
        // in the warp-range kernel costs more than it saves.)
        if (TABW > 0 && blk != 0 && refresh_due(blk)) {
            float hi = neg_inf(), lo = neg_inf();
            volatile float* tab = lane_tab;
            tab[w * 32 + lane] = ls.m;
#pragma unroll
            for (int j = 0; j < TABW; ++j) {
                const float v2 = tab[j * 32 + lane];
                lo = fmaxf(lo, fminf(hi, v2));
                hi = fmaxf(hi, v2);
            }
            // two smallest of the 64 values (lo <= hi in every lane)
#pragma unroll
            for (int d2 = 16; d2 > 0; d2 >>= 1) {
                const float olo = __shfl_xor_sync(kFull, lo, d2), ohi = __shfl_xor_sync(kFull, hi, d2);
                const float nhi = fminf(fmaxf(lo, olo), fminf(hi, ohi));
                lo = fminf(lo, olo);
                hi = nhi;
            }
            sel.thr = fmaxf(sel.thr, hi);
            if (shared_thr != nullptr) {
                if (lane == 0 && sel.thr != neg_inf()) atomicMax(shared_thr, f2ord(sel.thr));
                sel.thr = fmaxf(sel.thr, ord2f(*(volatile uint32_t*)shared_thr));
            }
        }
        if (blk == 0 && sel.cnt == 0 && sel.thr == neg_inf()) {
            // Seed the list with each lane's best (and second best) element of this
            // block, scanned in id order, so the threshold is useful at once.
            float b1 = neg_inf(), b2 = neg_inf();
            int p1 = -1, p2 = -1;
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float x = pick(v[u], k);
                    if (x > b1) {
                        b2 = b1; p2 = p1;
                        b1 = x; p1 = u * 4 + k;
                    } else if (SLOTS == 2 && x > b2) {
                        b2 = x; p2 = u * 4 + k;
                    }
                }
            }
            const uint32_t i1 = p1 >= 0 ? idb + 128u * (uint32_t)(p1 >> 2) + (uint32_t)(p1 & 3) : kPadId;
            sel.L.insert32(b1, i1, lane);
            if constexpr (SLOTS == 2) {
                const uint32_t i2 = p2 >= 0 ? idb + 128u * (uint32_t)(p2 >> 2) + (uint32_t)(p2 & 3) : kPadId;
                sel.L.insert32(b2, i2, lane);
            }
            sel.thr = sel.L.kth(sel.K);
            if (__any_sync(kFull, bm >= sel.thr)) {
                uint32_t ex = 0;  // the seeded elements are already in the list
                if (p1 >= 0) ex |= 1u << p1;
                if (SLOTS == 2 && p2 >= 0) ex |= 1u << p2;
                uint32_t mk = block_mask<U>(v, sel.thr) & ~ex;
                if (partial) mk &= live_mask<U>(idb, id_end);
                sel.append_block(slot_f, mk, idb, lane);
            }
        } else if (__any_sync(kFull, bm >= sel.thr)) {
            uint32_t mk = block_mask<U>(v, sel.thr);
            if (partial) mk &= live_mask<U>(idb, id_end);
            sel.append_block(slot_f, mk, idb, lane);
        }
    }
}

// Stream vectors [q0, q1) of one row: running sum per lane, top-k per warp.
// Full blocks (U vectors per lane, 512*U contiguous bytes per warp) go through a ring
// of STAGES blocks in shared memory filled by cp.async, so STAGES-1 blocks stay in
// flight while one is reduced; each lane reads back only what it copied itself.
//
// TABW > 0 (row-queue kernel: TABW warps stream parts of the same row): at each
// threshold refresh the warp publishes its lanes' running maxima in lane_tab[w][lane]
// and bounds the top-k by the K-th largest over lanes of max_j lane_tab[j][lane]. Each
// of those 32 values is an element of a different (warp, lane) stream of the row, so K
// of them are K distinct elements, and with TABW times more elements behind each value
// the bound sits much closer to the row's true K-th best than one warp's own.
template <int SLOTS, bool TOPK, int U, int STAGES, int TABW = 0, int IL = 1>
__device__ __forceinline__ void stream_piece(const float* rowp, uint32_t V, uint32_t q0, uint32_t q1, int lane,
                                             LaneSum& ls, Selector<SLOTS>& sel, bool& t_here, uint32_t t,
                                             float& xt, float4* ring, uint32_t* shared_thr = nullptr,
                                             float* lane_tab = nullptr, int w = 0) {
    const int a = (int)(((uintptr_t)rowp >> 2) & 3u);
    const float* vbase = rowp - a;  // 16-byte aligned
    const uint32_t qf = a ? 1u : 0u;
    const uint32_t qe = (V + (uint32_t)a) >> 2;
    const uint32_t nfull = qe > qf ? qe - qf : 0u;
    // [qa, qb): the piece's whole 16-byte vectors, streamed through the ring; before and
    // after them at most the row's partial first and last vectors (unaligned rows only).
    const uint32_t qa = max(q0, qf);
    const uint32_t qb = max(min(q1, qe), qa);
    // IL > 1: the IL warps of a CTA share the piece block by block, warp w taking blocks
    // w, w + IL, w + 2 IL, ... (each warp's bytes spread over the whole piece, so the warps
    // meet the same HBM and the same share of large values); IL = 1: the warp streams all.
    const uint32_t wi = IL > 1 ? (uint32_t)w : 0u;
    const uint32_t nb_all = (qb - qa + 32u * U - 1u) / (32u * U);
    const uint32_t nblk = nb_all > wi ? (nb_all - wi + IL - 1u) / IL : 0u;
    // vectors in the warp's last block when it is the piece's partial last block
    const uint32_t rem = (nb_all != 0u && (nb_all - 1u) % IL == wi) ? (qb - qa) % (32u * U) : 0u;

    // ---- bulk: U vectors per lane per block ---------------------------------------------
    // The issue side walks the source and the ring slots by running offsets (no index
    // arithmetic per block); the U copies of a block use immediate address offsets. In a
    // partial last block a lane copies only its vectors below qb and fills the others'
    // ring slots with -inf (no term, no maximum; the top-k keeps ids below id_end), so
    // the piece's tail streams through the ring like the rest.
    constexpr uint32_t kStage = U * 512u;  // ring bytes per block and warp
    const float* src = vbase + 4 * ((size_t)qa + 32u * U * wi + lane);
    const uint32_t ring_lane = (uint32_t)__cvta_generic_to_shared(ring + lane);
    uint32_t put = 0, get = 0;  // ring offsets of the next block to issue / to reduce
    uint32_t unissued = nblk;
    auto issue = [&]() {
        if (unissued) {
            if (unissued == 1u && rem != 0u) cp_async16_run_pad<U>(ring_lane + put, src, (int)rem - lane);
            else cp_async16_run<U>(ring_lane + put, src);
            src += 128 * U * IL;
            put = put == (STAGES - 1) * kStage ? 0u : put + kStage;
            --unissued;
        }
        cp_async_commit();
    };
    if (nblk) {
#pragma unroll
        for (int s0 = 0; s0 < STAGES - 1; ++s0) issue();
    }
    // Whether this piece holds the target column (t, the column in this row): decided
    // after the first copies are in flight, so the wait for the token id overlaps them.
    const int64_t e_lo = 4 * (int64_t)q0 - a, e_hi = 4 * (int64_t)q1 - a;
    t_here = t < V && (int64_t)t >= e_lo && (int64_t)t < e_hi;
    if (IL > 1 && t_here) {  // the warp of the target's block; warp 0 for the row's edges
        const uint32_t qt = (t + (uint32_t)a) >> 2;
        t_here = (qt >= qa && qt < qb) ? ((qt - qa) / (32u * U)) % IL == wi : wi == 0u;
    }
    bool xt_pending = t_here;
    uint32_t idb = 4u * (qa + 32u * U * wi + (uint32_t)lane) - (uint32_t)a;
    const uint32_t id_end = 4u * qb - (uint32_t)a;  // ids of the ring's padding start here
    for (uint32_t blk = 0; blk < nblk; ++blk) {
        issue();
        cp_async_wait<STAGES - 1>();
        float4 v[U];
        const float4* stage = ring + lane + get / 16u;
        const float* slot_f = reinterpret_cast<const float*>(ring + get / 16u);  // the block, all lanes
        get = get == (STAGES - 1) * kStage ? 0u : get + kStage;
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = stage[32 * u];
        if (xt_pending) {  // the target id has arrived by now
            if (lane == 0) xt = rowp[t];
            xt_pending = false;
        }
        float mu[U];
#pragma unroll
        for (int u = 0; u < U; ++u) mu[u] = max4(v[u]);
        float bm = mu[0];
#pragma unroll
        for (int u = 1; u + 1 < U; u += 2) bm = max3(bm, mu[u], mu[u + 1]);
        if ((U & 1) == 0) bm = fmaxf(bm, mu[U - 1]);
        ls.add_block<U>(v, bm);

        select_block<SLOTS, TOPK, U, TABW>(v, bm, blk, blk + 1u == nblk && rem != 0u, idb, id_end, slot_f, ls, sel,
                                           lane, shared_thr, lane_tab, w);
        idb += 128u * U * IL;
    }
    if (xt_pending && lane == 0) xt = rowp[t];

    // ---- edges: the row's partial first and last vectors (rows that do not start or end
    // on a 16-byte boundary), one checked vector per lane; warp 0 of an interleaved piece
#pragma unroll 1
    for (int part = 0; part < (wi == 0u ? 2 : 0); ++part) {
        const uint32_t lo = part ? qb : q0;
        const uint32_t hi = part ? q1 : min(qa, q1);
        for (uint32_t qs = lo; qs < hi; qs += 32) {
            const uint32_t q = qs + (uint32_t)lane;
            float4 v = make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
            uint32_t vm = 0;
            if (q < hi) v = load_checked(rowp, vbase, q, a, V, qf, nfull, vm);
            const float mx = max4(v);
            ls.note(mx);
            ls.add4(v);
            if constexpr (TOPK) {
                if (__any_sync(kFull, mx >= sel.thr))
                    sel.append(v, 4u * q - (uint32_t)a, ge_mask(v, sel.thr) & vm, lane);
            }
        }
    }
    if constexpr (TOPK) {
        // The row-queue kernel reads only the first K entries after this (its tree merges
        // 8 wide for K <= 8); the warp-range kernel merges whole lists.
        if (SLOTS == 1 && TABW > 0 && sel.K <= 8u && sel.cnt > 0 && sel.cnt <= 8) sel.flush_top8(lane);
        else if (sel.cnt > 0) sel.flush(lane);
    }
    // Leave the reference at the lane's maximum (c = m * k), the form the merges and the
    // row tuples use.
    if (ls.m != neg_inf()) ls.rebase(ls.m);
}

// 1 / fp32(log2(e)): the reference's scale factor of the plain path (tau = 1).
constexpr double kInvLog2eF = 1.0 / (double)kLog2e;

// Write one finished row: K top columns and the target column. (C, S) are the row's
// reference and sum in the log2 domain of scale kk = fp32(log2(e)/tau); a logprob is
// x/tau - (C/(kk*tau) + ln(S)), formed in fp64 (see the sum-exp note at the top).
template <int SLOTS, bool TOPK>
__device__ __forceinline__ void write_row(const RowsParams& p, uint32_t o, const WarpList<SLOTS>& L, float C,
                                          float S, uint32_t t, bool has_xt, float xt, float kk, float tau,
                                          int lane) {
    const bool unit = tau == 1.f && kk == kLog2e;
    const double inv_tau = unit ? 1.0 : 1.0 / (double)tau;
    const double lse = (unit ? (double)C * kInvLog2eF : (double)C / ((double)kk * (double)tau)) + (double)logf(S);
    const size_t ro = (size_t)o * p.W;
    if constexpr (TOPK) {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const uint32_t i = (uint32_t)lane + 32u * k;
            if (i < p.K) {
                p.out_lp[ro + i] = (float)((double)L.x[k] * inv_tau - lse);
                p.out_tok[ro + i] = L.id[k];
            }
        }
    }
    if (lane == 0) {
        float lpt = __int_as_float(0x7fc00000);
        if (t < p.V && has_xt) lpt = (float)((double)xt * inv_tau - lse);
        if (t >= p.V) atomicOr(p.status, kStatusTokenRange);
        p.out_lp[ro + p.K] = lpt;
        p.out_tok[ro + p.K] = t;
    }
}

// An invalid row gets NaN logprobs and padding ids; its status bit is raised.
__device__ __forceinline__ void write_invalid_row(const RowsParams& p, uint32_t o, uint32_t err, int lane) {
    for (uint32_t col = (uint32_t)lane; col < p.W; col += 32) {
        p.out_lp[(size_t)o * p.W + col] = __int_as_float(0x7fc00000);
        p.out_tok[(size_t)o * p.W + col] = kPadId;
    }
    if (lane == 0) atomicOr(p.status, err);
}

// Vocab shard mode: store a finished row's tuple (ids offset to global ids).
template <int SLOTS, bool TOPK>
__device__ __forceinline__ void store_row_tuple(const RowsParams& p, uint32_t o, const WarpList<SLOTS>& L, float C,
                                                float S, uint32_t t, bool has_xt, float xt, int lane) {
    uint32_t* pw = reinterpret_cast<uint32_t*>(p.tuple_out + (size_t)o * p.stride);
    if (lane == 0) {
        pw[0] = __float_as_uint(C);
        pw[1] = __float_as_uint(S);
        pw[2] = __float_as_uint(has_xt ? xt : 0.f);
        pw[3] = (t < kTupleHolds ? t : kTupleHolds - 1u) | (has_xt ? kTupleHolds : 0u);
    }
    if constexpr (TOPK) {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const uint32_t i = (uint32_t)lane + 32u * k;
            if (i < p.K) {
                pw[4 + i] = __float_as_uint(L.x[k]);
                pw[4 + p.K + i] = L.id[k] == kPadId ? kPadId : L.id[k] + p.vocab_base;
            }
        }
    }
}

// An invalid row: NaN logprobs and padding ids (or, in vocab shard mode, a tuple whose
// reference is NaN); its status bit is raised.
template <bool EXT>
__device__ __forceinline__ void emit_invalid(const RowsParams& p, uint32_t o, uint32_t err, int lane) {
    if (EXT && p.tuple_out != nullptr) {
        uint32_t* pw = reinterpret_cast<uint32_t*>(p.tuple_out + (size_t)o * p.stride);
        for (uint32_t i = (uint32_t)lane; i < 4u + 2u * p.K; i += 32)
            pw[i] = (i < 4u + p.K) ? 0x7fc00000u : kPadId;
        if (lane == 0) atomicOr(p.status, err);
    } else {
        write_invalid_row(p, o, err, lane);
    }
}

// Partial tuple of piece j of a row whose first piece belongs to warp w0. A warp
// stores the piece of its first row in slot 0 and that of its last row in slot 1;
// only piece 0 can be its warp's last row.
__device__ __forceinline__ uint32_t* piece_slot(const RowsParams& p, uint64_t w0, uint32_t j, bool tail0) {
    return reinterpret_cast<uint32_t*>(p.partials + (size_t)(2 * (w0 + j) + ((j == 0 && tail0) ? 1 : 0)) * p.stride);
}

template <int SLOTS, bool TOPK>
__device__ __forceinline__ void store_piece(uint32_t* pw, uint32_t K, const WarpList<SLOTS>& L, float C, float S,
                                            bool has_xt, float xt, int lane) {
    if (lane == 0) {
        pw[0] = __float_as_uint(C);
        pw[1] = __float_as_uint(S);
        pw[2] = __float_as_uint(xt);
        pw[3] = has_xt ? 1u : 0u;
    }
    if constexpr (TOPK) {
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const uint32_t i = (uint32_t)lane + 32u * k;
            if (i < K) { pw[4 + i] = __float_as_uint(L.x[k]); pw[4 + K + i] = L.id[k]; }
        }
    }
}

template <int SLOTS>
__device__ __forceinline__ void load_piece_list(const uint32_t* pw, uint32_t K, int lane, float (&x)[SLOTS],
                                                uint32_t (&id)[SLOTS]) {
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        const uint32_t i = (uint32_t)lane + 32u * k;
        x[k] = neg_inf();
        id[k] = kPadId;
        if (i < K) {
            x[k] = __uint_as_float(__ldcg(pw + 4 + i));
            id[k] = __ldcg(pw + 4 + K + i);
        }
    }
}

// Merge all pieces of a split row (called by the warp that took the last ticket):
// (reference, sum) and the target logit from the headers, the top-k by sequential
// bitonic merges of the pieces' sorted lists (next list prefetched).
template <int SLOTS, bool TOPK>
__device__ __forceinline__ void merge_pieces(const RowsParams& p, uint64_t w0, uint32_t pieces, bool tail0, int lane,
                                             WarpList<SLOTS>& L, float& C, float& S, bool& has_xt, float& xt) {
    C = neg_inf();
    S = 0.f;
    has_xt = false;
    xt = 0.f;
    for (uint32_t j = (uint32_t)lane; j < pieces; j += 32) {
        const uint32_t* hw = piece_slot(p, w0, j, tail0);
        const float hc = __uint_as_float(__ldcg(hw)), hs = __uint_as_float(__ldcg(hw + 1));
        const float hx = __uint_as_float(__ldcg(hw + 2));
        const uint32_t hh = __ldcg(hw + 3);
        lse2_combine(C, S, hc, hs);
        if (hh) { xt = hx; has_xt = true; }
    }
    L.reset();
    if constexpr (TOPK) {
        float nx[SLOTS];
        uint32_t ni[SLOTS];
        load_piece_list<SLOTS>(piece_slot(p, w0, 0, tail0), p.K, lane, nx, ni);
        for (uint32_t j = 0; j < pieces; ++j) {
            float cx[SLOTS];
            uint32_t ci[SLOTS];
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) { cx[k] = nx[k]; ci[k] = ni[k]; }
            if (j + 1 < pieces) load_piece_list<SLOTS>(piece_slot(p, w0, j + 1, tail0), p.K, lane, nx, ni);
            merge_lists<SLOTS>(L.x, L.id, cx, ci, lane);
        }
    }
    warp_lse2_reduce(C, S);
    const unsigned hb = __ballot_sync(kFull, has_xt);
    has_xt = hb != 0;
    xt = __shfl_sync(kFull, xt, hb ? __ffs(hb) - 1 : 0);
}

// Publish a piece and take a ticket; true for the warp that arrives last.
__device__ __forceinline__ bool take_ticket(uint32_t* counters, uint64_t w0, uint32_t pieces, int lane) {
    __threadfence();
    __syncwarp();
    uint32_t ticket = 0;
    if (lane == 0) ticket = atomicAdd(counters + w0, 1u);
    ticket = __shfl_sync(kFull, ticket, 0);
    const bool last = ticket == pieces - 1;
    if (last) __threadfence();
    return last;
}

// Batch of output row o: the last b < B with out_off[b] <= o (out_off[0] = 0 and the
// offsets increase: every batch has at least one output row). With the offsets in shared
// memory the warp looks at 32 evenly spaced entries, then at the entries of the stride the
// first round chose (at most 64 for B <= 2047): two dependent loads, against ~log2(B) for a
// binary search. Warp-uniform: every lane calls it with the same o.
__device__ __forceinline__ uint32_t batch_of_row(const uint32_t* out_off, uint32_t B, uint32_t o, bool staged,
                                                 int lane) {
    if (!staged) {
        uint32_t lo = 0, hi = B;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (out_off[mid] <= o) lo = mid; else hi = mid;
        }
        return lo;
    }
    const uint32_t step = (B + 31u) >> 5;
    const uint32_t i = (uint32_t)lane * step;
    const unsigned first = __ballot_sync(kFull, i < B && out_off[i] <= o);  // lanes 0.. (lane 0 always)
    const uint32_t base = (31u - (uint32_t)__clz(first | 1u)) * step;
    uint32_t best = base;
    for (uint32_t j0 = 0; j0 < step; j0 += 32u) {
        const uint32_t j = base + j0 + (uint32_t)lane;
        const unsigned hit = __ballot_sync(kFull, j0 + (uint32_t)lane < step && j < B && out_off[j] <= o);
        if (hit) best = base + j0 + (31u - (uint32_t)__clz(hit));
    }
    return best;
}

// Where one output row reads and what it scores. Output row o of batch b is the
// (o - out_off[b])-th of the batch's last cnt positions; position r scores token r+1
// of the same sequence, the last position the batch's sampled token. Its logits row
// counts back from the end of the batch's logits rows, which must hold cnt rows at
// least (all positions of a sequence, or only its last ones).
// EXT = false compiles the plain path (every position has its logits row, raw logits):
// loff is off and k is the constant log2(e).
struct RowDesc {
    const float* rowp;  // logits row
    uint32_t t;         // target token
    float k;            // log2(e) / tau, rounded to fp32
    float tau;          // the batch's temperature (1 without temperatures)
    uint32_t err;       // status bit, 0 if the row is valid
};

template <bool EXT>
__device__ __forceinline__ RowDesc describe_row(const RowsParams& p, const uint32_t* off, const uint32_t* loff,
                                                const uint32_t* out_off, const uint8_t* echo, uint32_t b,
                                                uint32_t o) {
    RowDesc d;
    const uint32_t ob = out_off[b], oe = out_off[b + 1];
    const uint32_t sb = off[b], eb = off[b + 1];
    const uint32_t lb = EXT ? loff[b] : sb, le = EXT ? loff[b + 1] : eb;
    const uint32_t cnt = oe - ob, len = eb - sb;
    const bool layout_ok = (o >= ob) && (o < oe) && (eb > sb) && (eb <= p.T) && (cnt == (echo[b] ? len : 1u)) &&
                           (!EXT || ((le >= lb) && (le - lb >= cnt) && (le <= p.T_logits)));
    // tau must be positive and finite (NaN fails the first test) with log2(e)/tau finite
    d.k = kLog2e;
    d.tau = 1.f;
    bool tau_ok = true;
    if (EXT && p.tau != nullptr) {
        const float tau = p.tau[b];
        d.tau = tau;
        d.k = __fdiv_rn(kLog2e, tau);  // fp32: its rounding is covered by the logprob form
        tau_ok = tau > 0.f && tau <= 3.4028234663852886e38f && d.k <= 3.4028234663852886e38f;
    }
    d.err = !layout_ok ? kStatusOffsets : (!tau_ok ? kStatusTemperature : 0u);
    d.t = 0;
    d.rowp = p.logits;
    if (d.err == 0) {
        const uint32_t r = eb - cnt + (o - ob);
        d.t = (r + 1 < eb) ? p.tokens[r + 1] : p.sampled[b];
        d.rowp = p.logits + (size_t)(le - cnt + (o - ob)) * p.V;
    }
    return d;
}


// Stage the per-batch arrays in shared memory: [off][out_off][loff if distinct][echo].
template <bool EXT>
__device__ __forceinline__ void stage_batch_arrays(const RowsParams& p, uint32_t* s_dyn, int tid, int nthreads,
                                                   const uint32_t*& off, const uint32_t*& loff,
                                                   const uint32_t*& out_off, const uint8_t*& echo) {
    const uint32_t B = p.B;
    const bool var = EXT && p.loff != p.off;
    uint32_t* s_l = var ? s_dyn + 2 * (B + 1) : s_dyn;
    uint8_t* s_e = reinterpret_cast<uint8_t*>(s_dyn + (var ? 3u : 2u) * (B + 1));
    for (uint32_t i = (uint32_t)tid; i <= B; i += (uint32_t)nthreads) {
        const uint32_t a0 = p.off[i], a1 = p.out_off[i];
        const uint32_t a2 = var ? p.loff[i] : 0u;
        const uint8_t e = i < B ? p.echo[i] : 0;
        s_dyn[i] = a0;
        s_dyn[B + 1 + i] = a1;
        if (var) s_l[i] = a2;
        if (i < B) s_e[i] = e;
    }
    off = s_dyn;
    out_off = s_dyn + B + 1;
    loff = s_l;
    echo = s_e;
}

// The same arrays staged from the inputs alone, with the output rows derived in place: an
// exclusive scan of (echo ? positions : 1) per batch and the plan's checks (a batch
// range that is empty, decreasing or past T makes the offsets bad), so that nothing
// written by lp_ragged_plan is read. Every thread of the CTA must call it; R is the
// row count (the plan's), bad whether the plan rejects the offsets.
template <bool EXT>
__device__ __forceinline__ void stage_and_scan(const RowsParams& p, uint32_t* s_dyn, int tid, int nthreads,
                                               const uint32_t*& off, const uint32_t*& loff, const uint32_t*& out_off,
                                               const uint8_t*& echo, uint32_t& R, bool& bad) {
    __shared__ __align__(128) uint32_t s_aux[64];  // per-warp sums, then [32]: bad flag (128-byte multiple)
    const uint32_t B = p.B;
    const bool var = EXT && p.loff != p.off;
    uint32_t* s_off = s_dyn;
    uint32_t* s_out = s_dyn + B + 1;
    uint32_t* s_l = var ? s_dyn + 2 * (B + 1) : s_dyn;
    uint8_t* s_e = reinterpret_cast<uint8_t*>(s_dyn + (var ? 3u : 2u) * (B + 1));
    if (tid == 0) s_aux[32] = 0u;
    for (uint32_t i = (uint32_t)tid; i <= B; i += (uint32_t)nthreads) {
        s_off[i] = p.off[i];
        if (var) s_l[i] = p.loff[i];
        if (i < B) s_e[i] = p.echo[i];
    }
    __syncthreads();
    // each thread scans a contiguous chunk of batches
    const uint32_t per = (B + (uint32_t)nthreads - 1u) / (uint32_t)nthreads;
    const uint32_t b0 = min((uint32_t)tid * per, B), b1 = min(b0 + per, B);
    uint32_t sum = 0;
    bool bd = false;
    for (uint32_t b = b0; b < b1; ++b) {
        const uint32_t sb = s_off[b], eb = s_off[b + 1];
        if (eb <= sb || eb > p.T) bd = true;
        else sum += s_e[b] ? eb - sb : 1u;
    }
    const int lane = tid & 31, w = tid >> 5, nw = nthreads >> 5;
    uint32_t x = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_aux[w] = x;
    if (bd) atomicOr(&s_aux[32], 1u);
    __syncthreads();
    if (w == 0) {
        uint32_t v = lane < nw ? s_aux[lane] : 0u;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, v, d);
            if (lane >= d) v += y;
        }
        s_aux[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    uint32_t run = x - sum + (w ? s_aux[w - 1] : 0u);
    for (uint32_t b = b0; b < b1; ++b) {
        s_out[b] = run;
        const uint32_t sb = s_off[b], eb = s_off[b + 1];
        if (!(eb <= sb || eb > p.T)) run += s_e[b] ? eb - sb : 1u;
    }
    if (b1 == B && b0 < b1) s_out[B] = run;
    R = s_aux[nw - 1];
    bad = s_aux[32] != 0u;
    __syncthreads();
    off = s_off;
    out_off = s_out;
    loff = s_l;
    echo = s_e;
}

// Dynamic shared memory: the warps' rings, then the staged offsets. It starts where the
// static shared memory ends, so every static shared array of the row kernels is a
// multiple of 128 bytes: the rings then start on a 128-byte boundary and a warp's
// 512-byte copies and 16-byte reads touch four 128-byte rows each, not five (a test
// checks the kernels' static sizes).
template <int U, int STAGES>
__host__ __device__ constexpr uint32_t ring_bytes() { return (uint32_t)kWarps * STAGES * U * 512u; }

template <int SLOTS, bool TOPK, int U, int STAGES, bool EXT>
__global__ void __launch_bounds__(kThreads, LP_MIN_BLOCKS) k_rows(RowsParams p) {
    extern __shared__ __align__(128) unsigned char s_raw[];
    trigger_dependents();
    float4* rings = reinterpret_cast<float4*>(s_raw);
    uint32_t* s_dyn = reinterpret_cast<uint32_t*>(s_raw + ring_bytes<U, STAGES>());
    __shared__ float s_cx[kWarps][64];
    __shared__ uint32_t s_ci[kWarps][64];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t B = p.B, V = p.V, K = p.K;

    const uint32_t* off = p.off;
    const uint32_t* loff = p.loff;
    const uint32_t* out_off = p.out_off;
    const uint8_t* echo = p.echo;
    uint32_t status, R;
    const bool early = p.early && p.stage_offsets;
    if (early) {
        // rows derived here: the plan may still be running (see RowsParams::early)
        bool bad;
        stage_and_scan<EXT>(p, s_dyn, threadIdx.x, kThreads, off, loff, out_off, echo, R, bad);
        status = bad ? kStatusOffsets : 0u;
    } else {
        pdl_wait();  // plan's outputs (status, output offsets, cleared counters) are visible
        // Status, row count and the offsets are fetched in one round trip.
        status = __ldcg(p.plan_status);
        R = __ldcg(p.out_off + B);
        if (p.stage_offsets) {
            stage_batch_arrays<EXT>(p, s_dyn, threadIdx.x, kThreads, off, loff, out_off, echo);
            __syncthreads();
        }
    }
    if (status & kStatusOffsets) return;  // the plan rejects the offsets
    if (R == 0) return;
    if (R > p.T || (EXT && p.tuple_out != nullptr && R > p.tuple_rows) || (p.out_rows && R > p.out_rows)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            pdl_wait();
            atomicOr(p.status, kStatusOffsets);
        }
        return;
    }
    const uint64_t Q = (uint64_t)R * p.nq;
    // pieces of at least min_piece vectors, but at least one warp per row: short rows
    // would otherwise queue up behind a few warps, each paying a row's fixed costs
    uint64_t G = (Q + p.min_piece - 1) / p.min_piece;
    if (G < R) G = R;
    const uint64_t G_launch = (uint64_t)gridDim.x * kWarps;
    if (G > G_launch) G = G_launch;
    if (G == 0) G = 1;
    // No CTA-wide barrier after this point: every warp runs on its own.
    const uint64_t gw = (uint64_t)blockIdx.x * kWarps + w;
    if (gw >= G) return;

    const uint64_t g0 = sk_start(gw, Q, G), g1 = sk_start(gw + 1, Q, G);
    uint32_t o = (uint32_t)(g0 / p.nq);
    const uint32_t o_first = o;
    uint32_t q0 = (uint32_t)(g0 - (uint64_t)o * p.nq);
    uint32_t b = batch_of_row(out_off, B, o, p.stage_offsets != 0u, lane);  // batch of row o
    float4* ring = rings + (size_t)w * STAGES * U * 32;

    for (uint64_t g = g0; g < g1;) {
        const uint32_t q1 = (uint32_t)min((uint64_t)p.nq, (uint64_t)q0 + (g1 - g));
        const bool full = (q0 == 0) && (q1 == p.nq);

        // ---- row descriptor (identical in every lane) ---------------------------------
        const RowDesc d = describe_row<EXT>(p, off, loff, out_off, echo, b, o);
        if (d.err) {
            if (early) pdl_wait();  // before any status write
            if (q0 == 0) emit_invalid<EXT>(p, o, d.err, lane);
        } else {
            const uint32_t t = d.t;
            const uint32_t t_loc = EXT ? t - p.vocab_base : t;  // column of the target in this shard
            const float* rowp = d.rowp;
            bool t_here;

            LaneSum ls;
            ls.init(d.k);
            Selector<SLOTS> sel;
            sel.init(s_cx[w], s_ci[w], K);
            float xt = 0.f;
            stream_piece<SLOTS, TOPK, U, STAGES>(rowp, V, q0, q1, lane, ls, sel, t_here, t_loc, xt, ring);
            if (early) pdl_wait();  // the plan has finished before a piece's tickets or the status are touched

            float C = (ls.m == neg_inf()) ? neg_inf() : ls.ref(), S = ls.sum();
            warp_lse2_reduce(C, S);
            bool has_xt = t_here;
            float xt_row = __shfl_sync(kFull, xt, 0);

            bool emit = full;
            if (!full) {
                // ---- publish this piece; the warp taking the last ticket merges --------
                const uint64_t gr = (uint64_t)o * p.nq;
                const uint64_t w0 = sk_owner(gr, Q, G), w1 = sk_owner(gr + p.nq - 1, Q, G);
                const uint32_t pieces = (uint32_t)(w1 - w0 + 1);
                store_piece<SLOTS, TOPK>(reinterpret_cast<uint32_t*>(
                                             p.partials + (size_t)(2 * gw + (o == o_first ? 0 : 1)) * p.stride),
                                         K, sel.L, C, S, has_xt, xt_row, lane);
                emit = take_ticket(p.counters, w0, pieces, lane);
                if (emit) {
                    const bool tail0 = sk_start(w0, Q, G) != gr;
                    merge_pieces<SLOTS, TOPK>(p, w0, pieces, tail0, lane, sel.L, C, S, has_xt, xt_row);
                    if (lane == 0) p.counters[w0] = 0u;  // ready for the next call
                }
            }
            if (emit) {
                if (EXT && p.tuple_out != nullptr)
                    store_row_tuple<SLOTS, TOPK>(p, o, sel.L, C, S, t, has_xt, xt_row, lane);
                else
                    write_row<SLOTS, TOPK>(p, o, sel.L, C, S, t, has_xt, xt_row, d.k, d.tau, lane);
            }
        }

        // ---- next piece -----------------------------------------------------------
        g += q1 - q0;
        q0 = 0;
        ++o;
        while (b + 1 < B && out_off[b + 1] <= o) ++b;
    }
}

// ---------------------------------------------------------------------------------
// Few rows (up to three per SM; e.g. next-token logits for a decode batch): CTAs of NW
// warps take tasks; a task is a whole row, or, when there are fewer rows than twice the
// SMs, one of S contiguous pieces of a row (split-vocab, chosen on the host: S = min(2*SMs
// / rows, row length / 42 KB, 64) for rows of 192 KB or more). The CTA's warps take the
// task's 2 KB blocks in turn (warp w: blocks w, w + NW, ...) and merge their results in
// shared memory; a whole row is written at once, a piece is published to the workspace
// and the CTA that takes the row's last ticket merges the S pieces with all its warps
// (each warp merges every NW-th piece, then the shared-memory tree). The first CTA on each
// SM starts on a task of its own without an atomic, every later task comes from one queue
// counter (in a next-token step with at most one task per CTA, from a fixed map instead),
// so all SMs stream from the start. The warps of a CTA share their lanes' running maxima
// for the top-k threshold (see stream_piece). The request that comes last resets the
// queue for the next call; the merging CTA resets its row's ticket.
template <int NW>
struct __align__(128) CtaMerge {
    float list_x[NW][64];
    uint32_t list_i[NW][64];
    float red_c[NW];
    float red_s[NW];
    float xt;
    uint32_t has_xt;
    uint32_t row;
    uint32_t thr;  // threshold shared by the warps of the CTA for the current row
    uint32_t last;  // this CTA took the last ticket of its split row
    uint32_t status, rows;  // the status word and R, read once for the whole CTA
    uint32_t fast_ok;  // next-token start: 2 unchecked, 1 the layout is valid, 0 it is not
    uint32_t chk[2];   // next-token start: output_row_offsets[o], [o + 1] of the current task
    float lane_max[NW][32];  // running lane maxima of the current row (-inf between rows)
};

// Next-token logits (one logits row per batch: output row o reads logits row o). Warp w
// of CTA i < B * S prefetches into L2 the first vectors of its part of task i (8 or
// 16 KB), before the dependency wait or the offsets: HBM already works meanwhile. Task i is
// the CTA's own for i < min(B * S, SMs), and for a later CTA the task the queue hands
// out i-th; whichever CTA takes a task, every task is streamed, so no prefetched line
// goes unread. The range is computed as in stream_piece and lies inside logits row
// o (o < B = rows of logits); the prefetch is a hint and changes no result, even when
// the offsets turn out to be bad.
constexpr uint32_t kPrefetchVec = 1024;  // 16 KB per warp

template <int NW>
__device__ __forceinline__ void prefetch_own_task(const RowsParams& p, int w) {
    const uint32_t S = p.split, ntask = p.B * S;
    if (blockIdx.x >= ntask) return;
    const uint32_t o = blockIdx.x / S, piece = blockIdx.x - o * S;
    const uint32_t pq0 = (uint32_t)(((uint64_t)p.nq * piece) / S);
    const uint32_t pq1 = (uint32_t)(((uint64_t)p.nq * (piece + 1)) / S);
    const float* rowp = p.logits + (size_t)o * p.V;
    const int a = (int)(((uintptr_t)rowp >> 2) & 3u);
    const uint32_t qf = a ? 1u : 0u, qe = (p.V + (uint32_t)a) >> 2;
    const uint32_t qa = max(pq0, qf), qb = max(min(pq1, qe), qa);
    // 16 KB per warp for a CTA's own first task when the launch has at most two tasks per
    // SM and a small top-k (cheap blocks: the prefetch is consumed soon), else 8 KB. The
    // warps take the piece block by block, so together they start on its first NW * n
    // vectors: warp w prefetches the w-th n of them.
    const bool big = blockIdx.x < p.num_sms && p.K <= 7u && ntask <= 2u * p.num_sms;
    const uint32_t n = big ? kPrefetchVec : kPrefetchVec / 2u;
    const uint32_t c0 = min(qa + (uint32_t)w * n, qb), c1 = min(c0 + n, qb);
    if (c1 > c0) prefetch_l2_bulk(rowp - a + 4 * (size_t)c0, 16u * (c1 - c0));
}

constexpr int kQueueWarps = LP_QUEUE_WARPS;
constexpr int kQueueStages = LP_QUEUE_STAGES;
constexpr int kQueueUnroll = LP_QUEUE_UNROLL;

template <int SLOTS, bool TOPK, int U, int STAGES, int NW, bool EXT, bool STEP>
__global__ void __launch_bounds__(NW * 32, 24 / NW) k_rows_cta(RowsParams p) {
    extern __shared__ __align__(128) unsigned char s_raw[];
    trigger_dependents();
    float4* rings = reinterpret_cast<float4*>(s_raw);
    uint32_t* s_dyn = reinterpret_cast<uint32_t*>(s_raw + (size_t)NW * STAGES * U * 512u);
    __shared__ float s_cx[NW][64];
    __shared__ uint32_t s_ci[NW][64];
    __shared__ CtaMerge<NW> cm;
    constexpr int kT = NW * 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t B = p.B, V = p.V, K = p.K;

    const uint32_t* off = p.off;
    const uint32_t* loff = p.loff;
    const uint32_t* out_off = p.out_off;
    const uint8_t* echo = p.echo;
    const bool fast = LP_NEXT_TOKEN_FAST && p.next_token != 0u;
    const bool early = STEP && p.early && (fast || p.stage_offsets);  // STEP: lp_ragged_step's launch
    uint32_t status, R;
    if (fast && early) {
        // A step on next-token logits: the plan, which let this launch start only once all
        // earlier work had finished, may still be running; the tasks are known without the
        // offsets (see RowsParams::next_token), so the first rows stream at once. The plan's
        // status and the row offsets are read after the stream's wait for the plan.
        status = 0u;
        R = B;
    } else if (early) {
        // The logits are complete (the plan, launched after all earlier work, is running).
        if (p.T_logits == B && lane == 0) prefetch_own_task<NW>(p, w);
        // rows derived here: the plan may still be running (see RowsParams::early)
        bool bad;
        stage_and_scan<EXT>(p, s_dyn, threadIdx.x, kT, off, loff, out_off, echo, R, bad);
        status = bad ? kStatusOffsets : 0u;
    } else if (fast) {
        // An L2 prefetch of the CTA's first task is a hint with no effect on any result, so it
        // may come before the dependency wait: should an earlier kernel still write these
        // logits, its writes update the lines in L2 (the point of coherence); when this
        // launch's CTAs become resident during the previous launch's tail, HBM serves them
        // meanwhile.
        if (LP_PREFETCH_BEFORE_WAIT && lane == 0) prefetch_own_task<NW>(p, w);
        pdl_wait();  // plan's outputs (status, output offsets, cleared counters) are visible
        // Next-token logits: the tasks are known without the offsets (see
        // RowsParams::next_token). The plan's status and the caller's row count arrive in
        // shared memory while the first task streams and are checked before any row is
        // written (a rejected layout writes nothing, as below).
        status = 0u;
        R = B;
        if (threadIdx.x == 0) {
            cp_async4((uint32_t)__cvta_generic_to_shared(&cm.status), p.plan_status);
            cp_async4((uint32_t)__cvta_generic_to_shared(&cm.rows), out_off + B);
        }
    } else {
        pdl_wait();  // plan's outputs (status, output offsets, cleared counters) are visible
        // one read for the whole CTA: other CTAs may set status bits meanwhile, and every
        // thread must leave the task loop below on the same task count
        if (threadIdx.x == 0) {
            cm.status = __ldcg(p.plan_status);
            cm.rows = __ldcg(p.out_off + B);
        }
        if (p.stage_offsets) stage_batch_arrays<EXT>(p, s_dyn, threadIdx.x, kT, off, loff, out_off, echo);
        __syncthreads();
        status = cm.status;
        R = cm.rows;
    }
    cm.lane_max[w][lane] = neg_inf();
    // Tasks: piece `task % S` of row `task / S` (S = p.split pieces per row). The launch
    // holds two CTAs per SM and the first min(tasks, SMs) CTAs (one per SM in the
    // hardware's dispatch order) start on task blockIdx.x without an atomic; every later
    // task comes from a queue: [0] next task of [nA, R*S) ([1] unused); with S > 1, one
    // arrival ticket per row from [2]. Any CTA may take any task, so the result does not
    // depend on where CTAs land, only the balance does.
    const uint32_t S = p.split;
    uint32_t* queue = p.counters;
    uint32_t* tickets = queue + 2;
    const bool too_many = R > p.T || (EXT && p.tuple_out != nullptr && R > p.tuple_rows) ||
                          (S > 1 && R > p.split_rows) || (p.out_rows && R > p.out_rows);
    const bool bad = (status & kStatusOffsets) || too_many;
    const uint32_t ntask = bad ? 0u : R * S;
    // In a step on next-token logits (spread_first) the CTAs after the first SMs take the
    // remaining tasks by a fixed map instead of the queue, which the plan clears: CTA
    // SMs + j takes task SMs + k for the j = floor(k * (CTAs - SMs) / (tasks - SMs)), so
    // the second tasks spread evenly over the CTAs in dispatch order (and thus over the
    // SMs); every CTA then holds at most one task and nA = tasks.
    const bool spread = STEP && p.spread_first != 0u && ntask > p.num_sms && ntask <= gridDim.x;
    const uint32_t nA = spread ? ntask : (ntask < p.num_sms ? ntask : p.num_sms);
    // Task -> row o, piece of the row, pieces of the row, partial slot of its piece 0.
    struct TaskRef {
        uint32_t o, piece, n, slot0;
    };
    auto task_ref = [&](uint32_t task) -> TaskRef {
        const uint32_t oo = S == 1u ? task : task / S;
        return TaskRef{oo, task - oo * S, S, oo * S};
    };
    // A CTA without a task of its own goes to the queue (counters): after the plan.
    if (early && !spread && blockIdx.x >= nA) pdl_wait();
    // Every CTA asks the queue after each task (and a CTA without a task of its own once at
    // its start) until it is told there is none: one request per queued task, one refusal
    // per CTA that asks. Every CTA sees the same task count, so the number of requests is
    // known, and the request that comes last resets the queue for the next call (no CTA
    // touches it afterwards), so no CTA has to count itself out at its end.
    const uint32_t requests = ntask > nA ? ntask - nA + gridDim.x : nA;
    auto next_task = [&]() -> uint32_t {  // thread 0 only
        const uint32_t r = atomicAdd(queue, 1u);
        if (r == requests - 1u) queue[0] = 0u;
        const uint32_t rb = nA + r;
        return rb < ntask ? rb : ntask;
    };
    if (threadIdx.x == 0) {
        cm.has_xt = 0u;
        cm.thr = 0u;
        cm.fast_ok = 2u;
        uint32_t task = ntask;
        if (spread) {
            const uint32_t f = p.num_sms, g2 = gridDim.x - f, rest = ntask - f;
            if (blockIdx.x < f) {
                task = blockIdx.x;
            } else {
                const uint32_t j = blockIdx.x - f;
                const uint32_t k = (uint32_t)(((uint64_t)j * rest + g2 - 1u) / g2);
                if (k < rest && (uint32_t)(((uint64_t)k * g2) / rest) == j) task = f + k;
            }
        } else if (blockIdx.x < nA) {
            task = blockIdx.x;
        } else if (ntask > nA) {
            task = next_task();
        }
        cm.row = task;
        if (blockIdx.x == 0 && too_many && !(status & kStatusOffsets)) atomicOr(p.status, kStatusOffsets);
    }
    float4* ring = rings + (size_t)w * STAGES * U * 32;
    __syncthreads();

    // The warps' sorted lists (in cm.list_*) merged into warp 0's list by a shared-memory tree.
    // Only the first K entries are read after the merge, so with one slot per lane the tree
    // merges the first 8 or 16 entries when K fits (fewer stages per round).
    const int tree_width = K <= 8u ? 8 : (K <= 16u ? 16 : 32);
    auto tree_merge = [&](WarpList<SLOTS>& L) {
        if constexpr (TOPK) {
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                cm.list_x[w][lane + 32 * k] = L.x[k];
                cm.list_i[w][lane + 32 * k] = L.id[k];
            }
        }
        __syncthreads();
        if constexpr (TOPK) {
#pragma unroll
            for (int st = 1; st < NW; st <<= 1) {
                if ((w & (2 * st - 1)) == 0 && w + st < NW) {
                    if constexpr (SLOTS == 1) {
                        // the partner's list read reversed within each group of tree_width
                        const int g = tree_width - 1;
                        const int src = (lane & ~g) | (g - (lane & g));
                        const float rx = cm.list_x[w + st][src];
                        const uint32_t ri = cm.list_i[w + st][src];
                        if (tree_width == 8) merge_top_rev<8>(L.x[0], L.id[0], rx, ri, lane);
                        else if (tree_width == 16) merge_top_rev<16>(L.x[0], L.id[0], rx, ri, lane);
                        else merge_top_rev<32>(L.x[0], L.id[0], rx, ri, lane);
                    } else {
                        float bx[SLOTS];
                        uint32_t bi[SLOTS];
#pragma unroll
                        for (int k = 0; k < SLOTS; ++k) {
                            bx[k] = cm.list_x[w + st][lane + 32 * k];
                            bi[k] = cm.list_i[w + st][lane + 32 * k];
                        }
                        merge_lists<SLOTS>(L.x, L.id, bx, bi, lane);
                    }
#pragma unroll
                    for (int k = 0; k < SLOTS; ++k) {
                        cm.list_x[w][lane + 32 * k] = L.x[k];
                        cm.list_i[w][lane + 32 * k] = L.id[k];
                    }
                }
                __syncthreads();
            }
        }
    };

    for (;;) {
        const uint32_t task = cm.row;
        if (task >= ntask) break;
        const TaskRef tr = task_ref(task);
        const uint32_t o = tr.o, piece = tr.piece, Sr = tr.n;
        RowDesc d;
        if (fast) {
            d.rowp = p.logits + (size_t)o * V;
            d.t = p.sampled[o];
            d.k = kLog2e;
            d.tau = 1.f;
            d.err = 0u;  // the row's checks come before its write
            if (EXT && p.tau != nullptr) {
                d.tau = p.tau[o];
                d.k = __fdiv_rn(kLog2e, d.tau);
            }
            if (threadIdx.x == 0 && !early) {  // the caller's output offsets of row o, fetched meanwhile
                cp_async4((uint32_t)__cvta_generic_to_shared(&cm.chk[0]), out_off + o);
                cp_async4((uint32_t)__cvta_generic_to_shared(&cm.chk[1]), out_off + o + 1);
                cp_async_commit();
            }
        } else {
            const uint32_t lo = batch_of_row(out_off, B, o, p.stage_offsets != 0u, lane);
            d = describe_row<EXT>(p, off, loff, out_off, echo, lo, o);
        }
        if (d.err) {
            if (early) pdl_wait();  // before any status write or queue access
            if (w == 0 && piece == 0) emit_invalid<EXT>(p, o, d.err, lane);
            __syncthreads();  // every thread has read cm.row
            if (threadIdx.x == 0) cm.row = next_task();
            __syncthreads();
            continue;
        }
        const uint32_t t = d.t;
        const uint32_t t_loc = EXT ? t - p.vocab_base : t;  // column of the target in this shard
        const float* rowp = d.rowp;
        const uint32_t pq0 = Sr == 1u ? 0u : (uint32_t)(((uint64_t)p.nq * piece) / Sr);
        const uint32_t pq1 = Sr == 1u ? p.nq : (uint32_t)(((uint64_t)p.nq * (piece + 1)) / Sr);
        bool t_here;

        LaneSum ls;
        ls.init(d.k);
        Selector<SLOTS> sel;
        sel.init(s_cx[w], s_ci[w], K);
        float xt = 0.f;
        stream_piece<SLOTS, TOPK, U, STAGES, NW, NW>(rowp, V, pq0, pq1, lane, ls, sel, t_here, t_loc, xt, ring,
                                                     &cm.thr, &cm.lane_max[0][0], w);
        if (early) pdl_wait();  // the plan has finished before the queue, tickets or status are touched
        if (fast && early && threadIdx.x == 0) {
            // the plan's outputs this task's checks need, read during the merges below
            if (cm.fast_ok == 2u) {
                cp_async4((uint32_t)__cvta_generic_to_shared(&cm.status), p.plan_status);
                cp_async4((uint32_t)__cvta_generic_to_shared(&cm.rows), out_off + B);
            }
            cp_async4((uint32_t)__cvta_generic_to_shared(&cm.chk[0]), out_off + o);
            cp_async4((uint32_t)__cvta_generic_to_shared(&cm.chk[1]), out_off + o + 1);
            cp_async_commit();
        }
        // The CTA's next task is asked for now, so the round trip overlaps the merges.
        uint32_t next = 0;
        if (threadIdx.x == 0) next = next_task();

        float C = (ls.m == neg_inf()) ? neg_inf() : ls.ref(), Sm = ls.sum();
        warp_lse2_reduce(C, Sm);
        if (lane == 0) {
            cm.red_c[w] = C;
            cm.red_s[w] = Sm;
            if (t_here) { cm.xt = xt; cm.has_xt = 1u; }
        }
        tree_merge(sel.L);
        if (w == 0) {
            C = neg_inf();
            Sm = 0.f;
            for (int j = lane; j < NW; j += 32) lse2_combine(C, Sm, cm.red_c[j], cm.red_s[j]);
            warp_lse2_reduce(C, Sm);
            uint32_t last = 0u;
            bool write = true;       // fast start: the layout is valid
            uint32_t row_err = 0u;   // fast start: this row's own check
            if (fast) {
                uint32_t ok = 0u, c0 = 0u, c1 = 0u;
                if (lane == 0) {
                    cp_async_wait<0>();
                    if (cm.fast_ok == 2u) {  // first task: the plan's check and the caller's row count
                        const bool st_ok = (cm.status & kStatusOffsets) == 0u;
                        cm.fast_ok = (st_ok && cm.rows == B) ? 1u : 0u;
                        if (st_ok && cm.rows != B) atomicOr(p.status, kStatusOffsets);
                    }
                    ok = cm.fast_ok;
                    c0 = cm.chk[0];
                    c1 = cm.chk[1];
                }
                write = __shfl_sync(kFull, ok, 0) == 1u;
                c0 = __shfl_sync(kFull, c0, 0);
                c1 = __shfl_sync(kFull, c1, 0);
                if (!(c0 == o && c1 == o + 1u)) row_err = kStatusOffsets;
                else if (EXT && p.tau != nullptr &&
                         !(d.tau > 0.f && d.tau <= 3.4028234663852886e38f && d.k <= 3.4028234663852886e38f))
                    row_err = kStatusTemperature;
            }
            if (!write) {
                // a layout the plan rejects: nothing written, nothing published
            } else if (row_err) {
                if (piece == 0) emit_invalid<EXT>(p, o, row_err, lane);
            } else if (Sr == 1) {
                if (EXT && p.tuple_out != nullptr)
                    store_row_tuple<SLOTS, TOPK>(p, o, sel.L, C, Sm, t, cm.has_xt != 0, cm.xt, lane);
                else
                    write_row<SLOTS, TOPK>(p, o, sel.L, C, Sm, t, cm.has_xt != 0, cm.xt, d.k, d.tau, lane);
            } else {
                // a piece of a split row: publish it; the CTA that takes the row's last
                // ticket merges all pieces
                store_piece<SLOTS, TOPK>(
                    reinterpret_cast<uint32_t*>(p.partials + (size_t)(tr.slot0 + piece) * p.stride), K, sel.L, C,
                    Sm, cm.has_xt != 0, cm.xt, lane);
                last = take_ticket(tickets, o, Sr, lane) ? 1u : 0u;
            }
            __syncwarp();
            if (lane == 0) {
                cm.has_xt = 0u;
                cm.thr = 0u;
                cm.last = last;
                cm.row = next;  // every thread read cm.row before the merge barriers
            }
        }
        cm.lane_max[w][lane] = neg_inf();  // every warp is past this task's stream
        __syncthreads();
        if (Sr > 1 && cm.last) {
            // ---- merge the row's Sr pieces with the whole CTA ----------------------------
            const unsigned char* base = p.partials + (size_t)tr.slot0 * p.stride;
            C = neg_inf();
            Sm = 0.f;
            bool has = false;
            float xr = 0.f;
            for (uint32_t j = threadIdx.x; j < Sr; j += kT) {
                const uint32_t* hw = reinterpret_cast<const uint32_t*>(base + (size_t)j * p.stride);
                lse2_combine(C, Sm, __uint_as_float(__ldcg(hw)), __uint_as_float(__ldcg(hw + 1)));
                if (__ldcg(hw + 3)) { xr = __uint_as_float(__ldcg(hw + 2)); has = true; }
            }
            warp_lse2_reduce(C, Sm);
            if (lane == 0) {
                cm.red_c[w] = C;
                cm.red_s[w] = Sm;
            }
            if (has) { cm.xt = xr; cm.has_xt = 1u; }  // one piece holds the target
            sel.L.reset();
            if constexpr (TOPK) {
                for (uint32_t j = (uint32_t)w; j < Sr; j += NW) {
                    float cx[SLOTS];
                    uint32_t ci[SLOTS];
                    load_piece_list<SLOTS>(reinterpret_cast<const uint32_t*>(base + (size_t)j * p.stride), K, lane,
                                           cx, ci);
                    merge_lists<SLOTS>(sel.L.x, sel.L.id, cx, ci, lane);
                }
            }
            tree_merge(sel.L);
            if (w == 0) {
                C = neg_inf();
                Sm = 0.f;
                for (int j = lane; j < NW; j += 32) lse2_combine(C, Sm, cm.red_c[j], cm.red_s[j]);
                warp_lse2_reduce(C, Sm);
                if (EXT && p.tuple_out != nullptr)
                    store_row_tuple<SLOTS, TOPK>(p, o, sel.L, C, Sm, t, cm.has_xt != 0, cm.xt, lane);
                else
                    write_row<SLOTS, TOPK>(p, o, sel.L, C, Sm, t, cm.has_xt != 0, cm.xt, d.k, d.tau, lane);
                __syncwarp();
                if (lane == 0) {
                    tickets[o] = 0u;  // ready for the next call
                    cm.has_xt = 0u;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------------
// Vocab shard merge: P row tuples per output row (one per vocab shard, as gathered from
// the ranks) -> the row's logprobs. One warp per row: the shards' (reference, sum)
// pairs combine in the log2 domain, their sorted top-k lists merge in shard order
// under (logit desc, global id asc), and the target logit comes from the shard that
// holds it.
constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 8;  // shard lists loaded together (the first batch before the headers)

template <int SLOTS, bool TOPK>
__global__ void __launch_bounds__(kMergeWarps * 32) k_shard_merge(RowsParams p, const unsigned char* tuples,
                                                                  uint32_t P, uint32_t rows_capacity) {
    const int lane = threadIdx.x & 31;
    const uint32_t R = __ldg(p.out_off + p.B);
    if (R > rows_capacity) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusOffsets);
        return;
    }
    const size_t shard_bytes = (size_t)rows_capacity * p.stride;
    const uint32_t nw = gridDim.x * kMergeWarps;
    for (uint32_t o = blockIdx.x * kMergeWarps + (threadIdx.x >> 5); o < R; o += nw) {
        const unsigned char* row0 = tuples + (size_t)o * p.stride;
        // The shards' sorted lists do not depend on the headers: the first batch is loaded
        // now, so the row costs about one memory latency for up to kMergeBatch shards.
        float bx[kMergeBatch][SLOTS];
        uint32_t bi[kMergeBatch][SLOTS];
        if constexpr (TOPK) {
#pragma unroll
            for (int q = 0; q < kMergeBatch; ++q)
                if ((uint32_t)q < P)
                    load_piece_list<SLOTS>(reinterpret_cast<const uint32_t*>(row0 + q * shard_bytes), p.K, lane, bx[q],
                                           bi[q]);
        }
        float C = neg_inf(), S = 0.f, xt = 0.f;
        bool has_xt = false, bad = false;
        uint32_t t = 0;
        for (uint32_t j = (uint32_t)lane; j < P; j += 32) {
            const uint32_t* hw = reinterpret_cast<const uint32_t*>(row0 + j * shard_bytes);
            const float hc = __uint_as_float(__ldg(hw)), hs = __uint_as_float(__ldg(hw + 1));
            const uint32_t w3 = __ldg(hw + 3);
            if (hc != hc) bad = true;
            else lse2_combine(C, S, hc, hs);
            if (w3 & kTupleHolds) { xt = __uint_as_float(__ldg(hw + 2)); has_xt = true; }
            t = w3 & ~kTupleHolds;
        }
        if (__any_sync(kFull, bad)) {
            write_invalid_row(p, o, 0u, lane);
            continue;
        }
        warp_lse2_reduce(C, S);
        const unsigned hb = __ballot_sync(kFull, has_xt);
        has_xt = hb != 0;
        xt = __shfl_sync(kFull, xt, hb ? __ffs(hb) - 1 : 0);
        t = __shfl_sync(kFull, t, 0);
        WarpList<SLOTS> L;
        L.reset();
        if constexpr (TOPK) {
            for (uint32_t j0 = 0; j0 < P; j0 += kMergeBatch) {
                if (j0 != 0) {
#pragma unroll
                    for (int q = 0; q < kMergeBatch; ++q)
                        if (j0 + q < P)
                            load_piece_list<SLOTS>(reinterpret_cast<const uint32_t*>(row0 + (j0 + q) * shard_bytes),
                                                   p.K, lane, bx[q], bi[q]);
                }
#pragma unroll
                for (int q = 0; q < kMergeBatch; ++q)
                    if (j0 + q < P) merge_lists<SLOTS>(L.x, L.id, bx[q], bi[q], lane);
            }
        }
        float kk = kLog2e, tau = 1.f;
        if (p.tau != nullptr) {  // same scale as the shards used (validated there)
            uint32_t lo = 0, hi = p.B;
            while (hi - lo > 1) {
                const uint32_t mid = (lo + hi) >> 1;
                if (__ldg(p.out_off + mid) <= o) lo = mid; else hi = mid;
            }
            tau = __ldg(p.tau + lo);
            kk = __fdiv_rn(kLog2e, tau);
        }
        write_row<SLOTS, TOPK>(p, o, L, C, S, t, has_xt, xt, kk, tau, lane);
    }
}

}  // namespace lpk
