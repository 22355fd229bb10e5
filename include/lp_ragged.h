/*
 * lp_ragged.h — C ABI of the GB300 ragged batched log-probability library.
 *
 * The operation (from "MAX Python SDK 中 log_probabilities 模块解析", sections
 * "两个核心函数的 API 契约", "ragged 数据编排：从输入缓冲到 kernel 调用" and
 * "top-k 语义：堆式 kernel 与「采样 token 兜底」"; the logprob definition from
 * "logprob、finish reason 与 output processing", section "logprob 的数值形态"):
 *
 *   batch b owns logits rows [off[b], off[b+1]) of an fp32 [T, V] matrix;
 *   it emits len_b output rows when echo[b] is set, else one row (its last
 *   position); output_row_offsets = [0, cumsum(counts)], R = output_row_offsets[B].
 *   For every output row o scoring logits row r:
 *     lse            = log(sum_v exp(x[r, v]))
 *     columns 0..K-1 = the K = 2^levels - 1 best tokens of the row under
 *                      (logit descending, token id ascending), as
 *                      (x[r, id] - lse, id), padded with (-inf, 0xFFFFFFFF)
 *                      when V < K;
 *     column K       = (x[r, t] - lse, t), t = tokens[r+1] when r+1 is still in
 *                      the sequence, else sampled_tokens[b].
 *   W = out_per_token = 2^levels (1 when levels == 0) columns per row.
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer (device memory, the workspace, the
 *     host words) and the stream. The library allocates nothing, keeps no state
 *     between calls apart from a per-device launch-shape cache, and may be called
 *     from several host threads on different workspaces.
 *   - Asynchrony: all device work is enqueued on `stream`; a return of LP_OK means
 *     "validated and enqueued", not "finished".
 *   - Host-checked errors are returned at once and nothing is enqueued.
 *   - Device-detected errors never trap: they set bits in the workspace status
 *     word (bit c set <=> error code c seen), read with lp_ragged_read_status.
 *   - Integers are uint32; echo flags are one byte each (0 = off).
 *   - Logits must be finite or -inf. -inf tokens have probability 0; a row of only
 *     -inf yields NaN logprobs. NaN or +inf logits give unspecified values (no fault).
 */
#ifndef LP_RAGGED_H
#define LP_RAGGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; 0 is the legacy default stream. */
typedef struct CUstream_st *lp_stream_t;

typedef enum lp_status {
    LP_OK = 0,
    LP_ERR_NULL = 1,         /* a required pointer is NULL                                  */
    LP_ERR_LEVELS = 2,       /* levels > LP_MAX_LEVELS                                      */
    LP_ERR_SHAPE = 3,        /* B, T or V is 0 or too large, or logits not 4-byte aligned   */
    LP_ERR_OFFSETS = 4,      /* device: empty or decreasing batch range, a range past T, or
                                output offsets that disagree with the echo flags           */
    LP_ERR_TOKEN_RANGE = 5,  /* device: an actual or sampled token >= V                     */
    LP_ERR_WORKSPACE = 6,    /* workspace NULL or smaller than lp_ragged_workspace_size     */
    LP_ERR_CUDA = 7,         /* a CUDA launch or copy failed                                */
    LP_ERR_TEMPERATURE = 8   /* device: a temperature that is not a positive finite number  */
} lp_status;

#define LP_MAX_LEVELS 6u
#define LP_PAD_TOKEN 0xFFFFFFFFu

/*
 * Bytes of scratch the two calls need on the CURRENT device (it depends on the
 * device's SM count and on levels only; B, T and V are accepted for forward
 * compatibility). Returns 0 when levels > LP_MAX_LEVELS or no device is usable.
 * The workspace holds the status word, per-CTA arrival counters and the split-row
 * partial tuples (max, sum-exp, top-K). One workspace per concurrently running call.
 */
size_t lp_ragged_workspace_size(uint32_t B, uint32_t T, uint32_t V, uint32_t levels);

/*
 * Step 1 — output-row plan (MAX page, "ragged 数据编排"): one device prefix sum of
 * count_b = echo[b] ? len_b : 1.
 *   logit_row_offsets   device, uint32[B+1], the input row offsets (next-token
 *                       logits: 0..B)
 *   echo                device, uint8[B]
 *   B, T                batches, logits rows
 *   output_row_offsets  device out, uint32[B+1]
 *   host_rows_and_status  optional host out (pinned for a truly async copy), two
 *                       words {R, status bits}; valid after the stream reaches this
 *                       point. Pass NULL to skip the copy.
 *   workspace           device, >= lp_ragged_workspace_size bytes; plan clears its
 *                       status word and arrival counters, so call plan before the
 *                       first compute on a workspace.
 * Device checks: len_b >= 1, off[b+1] <= T  (LP_ERR_OFFSETS bit).
 */
lp_status lp_ragged_plan(const uint32_t *logit_row_offsets, const uint8_t *echo, uint32_t B, uint32_t T,
                         uint32_t *output_row_offsets, uint32_t *host_rows_and_status,
                         void *workspace, size_t workspace_bytes, lp_stream_t stream);

/*
 * Step 2 — the streaming reduction (MAX page, "top-k 语义：堆式 kernel 与「采样
 * token 兜底」"): one pass over each scored logits row computing the online max and
 * sum-exp, the top-K under (logit desc, id asc), and the target token's logit.
 *   logits              device, float[T][V] row-major (any 4-byte alignment)
 *   logit_row_offsets   device, uint32[B+1]
 *   tokens              device, uint32[T], flat input tokens
 *   sampled_tokens      device, uint32[B]
 *   output_row_offsets  device, uint32[B+1], as written by lp_ragged_plan
 *   echo                device, uint8[B]
 *   levels              0..LP_MAX_LEVELS; K = 2^levels - 1, W = 2^levels (1 if 0)
 *   out_logprobs        device out, float[R][W]
 *   out_tokens          device out, uint32[R][W]
 *   R = output_row_offsets[B] is read on the device; the outputs must hold R*W
 *   entries each. Rows are split across CTAs when R is small (decode); the CTA that
 *   finishes a row's last piece merges the pieces, so there is a single launch.
 * Device checks: the offsets checks of plan (a bad batch is skipped), and
 *   tokens/sampled < V (LP_ERR_TOKEN_RANGE; that row's column K gets logprob NaN).
 */
lp_status lp_ragged_compute(const float *logits, uint32_t T, uint32_t V,
                            const uint32_t *logit_row_offsets, uint32_t B,
                            const uint32_t *tokens, const uint32_t *sampled_tokens,
                            const uint32_t *output_row_offsets, const uint8_t *echo, uint32_t levels,
                            float *out_logprobs, uint32_t *out_tokens,
                            void *workspace, size_t workspace_bytes, lp_stream_t stream);

/*
 * Step 2, extended: the same reduction for two variants of the caller's input.
 *
 * VARIABLE logits ("MAX Python SDK 中 log_probabilities 模块解析", section "echo 的
 * 前置条件：ReturnLogits 枚举": the model returns logits for only some positions).
 * Positions and logits rows are described separately:
 *   input_row_offsets   device, uint32[B+1]: batch b's positions [ioff[b], ioff[b+1])
 *                       of the T flat tokens; the output layout (plan) follows these.
 *   logit_row_offsets   device, uint32[B+1]: batch b's rows [loff[b], loff[b+1]) of
 *                       the T_logits logits rows, holding the LAST loff[b+1]-loff[b]
 *                       positions of the sequence. They must cover the positions the
 *                       batch scores (all of them with echo, the last one without);
 *                       otherwise the batch's rows get NaN / 0xFFFFFFFF and the
 *                       LP_ERR_OFFSETS bit is set.
 *   input_row_offsets == NULL means every position has its logits row (T == T_logits
 *   required, else LP_ERR_SHAPE), which is lp_ragged_compute.
 *   Call lp_ragged_plan with input_row_offsets and T first.
 *
 * Temperature (SGLang page "logprob、finish reason 与 output processing", section
 * "第二步：采样层选出 token_id，同时计算 logprob": the sampler scales the logits by
 * the request's temperature and the logprobs reuse that softmax):
 *   temperatures        device, float[B], or NULL for raw logits (tau = 1). Batch b's
 *                       logprobs are those of x / tau_b: column c holds
 *                       x[r, id] / tau_b - log(sum_v exp(x[r, v] / tau_b)). The top-K
 *                       ids still rank the raw fp32 logits (the same order for
 *                       tau_b > 0, and the ids stay exact). tau_b must be positive and
 *                       finite, else the batch's rows get NaN / 0xFFFFFFFF and the
 *                       LP_ERR_TEMPERATURE bit is set. Logits with |x| / tau beyond
 *                       ~8.8e37 overflow the fp32 sum and give unspecified values.
 *
 * Other arguments, outputs, workspace and checks: as lp_ragged_compute, with
 * logits float[T_logits][V] and tokens uint32[T].
 */
lp_status lp_ragged_compute_ex(const float *logits, uint32_t T_logits, uint32_t V,
                               const uint32_t *logit_row_offsets, const uint32_t *input_row_offsets, uint32_t T,
                               uint32_t B, const uint32_t *tokens, const uint32_t *sampled_tokens,
                               const uint32_t *output_row_offsets, const uint8_t *echo,
                               const float *temperatures, uint32_t levels, float *out_logprobs,
                               uint32_t *out_tokens, void *workspace, size_t workspace_bytes,
                               lp_stream_t stream);

/*
 * Steps 1 and 2 in one call, for a serving step whose output buffers are sized ahead
 * (R <= T always): lp_ragged_plan on the positions offsets (input_row_offsets, or
 * logit_row_offsets when it is NULL), then the reduction of lp_ragged_compute_ex, both
 * enqueued on `stream` by the library. Because the reduction directly follows the plan,
 * it streams the logits while the plan is still running (it derives the output rows
 * from the offsets itself, with the plan's checks) and waits for the plan only before
 * it touches the workspace counters or the status word; the rows are identical to
 * lp_ragged_plan + lp_ragged_compute_ex. With next-token logits (T == B == T_logits,
 * input_row_offsets NULL) the plan itself starts on the device as soon as the previous
 * kernel on the stream has finished (no launch gap; it waits for that kernel before it
 * reads or writes anything), and the reduction streams row o from logits row o before
 * it reads any offset; a layout the plan rejects still writes no row.
 *   output_row_offsets   device out, uint32[B+1] (as lp_ragged_plan)
 *   host_rows_and_status pinned host out, uint32[2] or NULL: {R, status}, copied after
 *                        the reduction (so the status holds the plan's and the
 *                        reduction's bits); valid once the stream reaches that point
 *   out_logprobs         device out, float[out_rows][W]
 *   out_tokens           device out, uint32[out_rows][W]
 *   out_rows             rows the outputs hold, > 0; when R > out_rows nothing is
 *                        written and the LP_ERR_OFFSETS bit is set
 * Other arguments, workspace and checks: as lp_ragged_plan and lp_ragged_compute_ex.
 * Errors: those of both calls.
 */
lp_status lp_ragged_step(const float *logits, uint32_t T_logits, uint32_t V, const uint32_t *logit_row_offsets,
                         const uint32_t *input_row_offsets, uint32_t T, uint32_t B, const uint32_t *tokens,
                         const uint32_t *sampled_tokens, const uint8_t *echo, const float *temperatures,
                         uint32_t levels, uint32_t *output_row_offsets, uint32_t *host_rows_and_status,
                         float *out_logprobs, uint32_t *out_tokens, uint32_t out_rows, void *workspace,
                         size_t workspace_bytes, lp_stream_t stream);

/*
 * Vocab-parallel form (the forward pass runs on tensor-parallel workers, SGLang page
 * "logprob、finish reason 与 output processing", section "第一步：ModelRunner.forward()
 * 输出 logits"; with the lm_head split by vocabulary each rank holds a contiguous range
 * of columns). Three steps per rank, on the same inputs except the logits:
 *   1. lp_ragged_plan (as usual; positions offsets),
 *   2. lp_ragged_shard_partials: this rank's columns -> one row tuple per output row,
 *   3. gather all ranks' tuple buffers into one [P][rows_capacity][stride] buffer in
 *      shard order (e.g. an NCCL all-gather), then lp_ragged_shard_merge -> the rows,
 *      identical to lp_ragged_compute on the unsplit logits (ids exact; logprobs
 *      within rounding).
 *
 * Row tuple layout (u32 words, stride = lp_ragged_tuple_bytes(levels) bytes, a
 * multiple of 16):
 *   [0] c  fp32 reference in the log2 domain: max logit of the shard's row x log2(e)/tau
 *          (-inf when every column is -inf; NaN marks an invalid row)
 *   [1] s  fp32 sum over the shard's columns of 2^(x*log2(e)/tau - c)
 *   [2] fp32 logit of the target token when this shard holds it, else 0
 *   [3] target token id in bits 0-30 (ids >= 2^31 stored as 2^31-1); bit 31 set when
 *       this shard holds the target
 *   [4, 4+K)     the shard's K best fp32 logits, sorted (logit desc, global id asc),
 *                -inf padding
 *   [4+K, 4+2K)  their global token ids (vocab_base + column), 0xFFFFFFFF padding
 */
uint32_t lp_ragged_tuple_bytes(uint32_t levels);

/*
 *   logits          device, float[T_logits][V_shard]: this rank's columns
 *                   [vocab_base, vocab_base + V_shard) of the full vocabulary
 *   vocab_base      global id of column 0 (vocab_base + V_shard < 2^31 - 1)
 *   tuples          device out, rows_capacity x lp_ragged_tuple_bytes(levels) bytes,
 *                   16-byte aligned; rows_capacity >= R, else nothing is written and
 *                   the LP_ERR_OFFSETS bit is set
 *   other arguments as lp_ragged_compute_ex (temperatures: the same on every rank).
 * A token id is not range-checked here (only the merge knows the full vocabulary).
 * An invalid row (bad offsets or temperature) sets its status bit and gets a tuple
 * with c = NaN.
 */
lp_status lp_ragged_shard_partials(const float *logits, uint32_t T_logits, uint32_t V_shard, uint32_t vocab_base,
                                   const uint32_t *logit_row_offsets, const uint32_t *input_row_offsets, uint32_t T,
                                   uint32_t B, const uint32_t *tokens, const uint32_t *sampled_tokens,
                                   const uint32_t *output_row_offsets, const uint8_t *echo,
                                   const float *temperatures, uint32_t levels, void *tuples,
                                   uint32_t rows_capacity, void *workspace, size_t workspace_bytes,
                                   lp_stream_t stream);

/*
 *   tuples          device, [P][rows_capacity][stride] bytes: shard p's tuple of output
 *                   row o at byte (p * rows_capacity + o) * stride. The P shards must
 *                   cover the vocabulary [0, V) exactly (a target no shard holds gets
 *                   logprob NaN). rows_capacity >= R, else LP_ERR_OFFSETS bit.
 *   V               full vocabulary size: targets >= V set LP_ERR_TOKEN_RANGE and get
 *                   logprob NaN
 *   output_row_offsets, B   as written by lp_ragged_plan
 *   temperatures    the same array the shards used, or NULL
 *   out_logprobs, out_tokens  device out, R x W, as lp_ragged_compute
 *   workspace       only its status word is used (set bits; plan clears it)
 * A row any of whose tuples is invalid gets NaN / 0xFFFFFFFF (the shard call set the
 * status bit). One warp per row; no allocation.
 */
lp_status lp_ragged_shard_merge(const void *tuples, uint32_t P, uint32_t rows_capacity, uint32_t V,
                                const uint32_t *output_row_offsets, uint32_t B, const float *temperatures,
                                uint32_t levels, float *out_logprobs, uint32_t *out_tokens, void *workspace,
                                size_t workspace_bytes, lp_stream_t stream);

/*
 * Allocation-free form of lp_ragged_compute (no counterpart on the pages; it exists
 * for callers that cannot allocate device memory: a serving engine whose HBM is
 * reserved up front by its own pool and that forbids cudaMalloc on the request
 * path, where cudaMalloc may synchronise the device; or a binding with no device
 * allocator of its own).
 *   Same arguments and host checks as lp_ragged_compute, minus the workspace. The
 *   scratch is a static device array of LP_NOALLOC_SCRATCH_BYTES inside this
 *   library, held by every GPU that loads it until the process exits.
 *   output_row_offsets  the plan's output (device, uint32[B+1]). lp_ragged_plan needs
 *                a workspace of at least 256 + 4 x (SMs x 32) bytes rounded up to
 *                256 (its status word and counters); a caller that has none can
 *                compute the same values on the host (an exclusive running sum of
 *                echo[b] ? len_b : 1) and copy them in.
 *   host_status  optional host word (pinned for an async copy): the status bits of
 *                this call, valid once the stream reaches this point; NULL skips.
 *                They include the plan's offsets check: the call validates the
 *                offsets itself first, and on a layout lp_ragged_plan rejects it
 *                writes no row and sets the LP_ERR_OFFSETS bit.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture. Every host check runs before anything is enqueued; then the call
 *   clears the status word and arrival counters itself (two launches: the
 *   validation, then the reduction), and no allocating routine (cudaMalloc,
 *   cudaFree, a library allocator) is called.
 *   Returns LP_ERR_WORKSPACE when this GPU needs more scratch than the array holds
 *   (more than ~245 SMs at levels 6). All calls share the array: calls that overlap
 *   on the GPU (other streams, other host threads) race; serialise them.
 */
#define LP_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
lp_status lp_ragged_compute_noalloc(const float *logits, uint32_t T, uint32_t V,
                                    const uint32_t *logit_row_offsets, uint32_t B,
                                    const uint32_t *tokens, const uint32_t *sampled_tokens,
                                    const uint32_t *output_row_offsets, const uint8_t *echo, uint32_t levels,
                                    float *out_logprobs, uint32_t *out_tokens, uint32_t *host_status,
                                    lp_stream_t stream);

/* Enqueue a copy of the workspace status word (bit c <=> lp_status c) to host. */
lp_status lp_ragged_read_status(const void *workspace, uint32_t *host_status, lp_stream_t stream);

/*
 * Which row kernel lp_ragged_compute / lp_ragged_compute_ex / lp_ragged_step launch for
 * this shape on the current device (diagnostics; no counterpart on the pages): *kind = 1
 * for the row queue (CTAs of 12 warps take whole rows or row pieces), 0 for warp-owned
 * ranges of the row space. T_logits, T, V, levels as in lp_ragged_compute_ex. The two
 * kernels give the same rows. Errors: LP_ERR_NULL, LP_ERR_LEVELS, LP_ERR_CUDA (no device).
 */
lp_status lp_ragged_row_kernel(uint32_t T_logits, uint32_t T, uint32_t V, uint32_t levels, int *kind);

/* Static, NUL-terminated description of a status code. */
const char *lp_ragged_strerror(lp_status status);

#ifdef __cplusplus
}
#endif

#endif /* LP_RAGGED_H */
