/*
 * dspark.h - C ABI of the DSpark draft-and-schedule step for NVIDIA GB300
 * (sm_103a).  One shared library, libdspark.so.
 *
 * The step has two stages.
 *
 *   Chaining  ("DSpark on MAX", section "What DSpark is", item 3; "How DSpark
 *   Speeds Up LLM Inference", section "Draft better"): a parallel drafter
 *   emits backbone logits for K draft positions at once; a rank-r Markov
 *   head adjusts position k's logits by bias[v] = U[prev] . V[v], prev being
 *   the token chosen at k-1 (the request's last committed token at k = 0),
 *   and an argmax over the vocabulary picks the token.
 *
 *   Confidence-scheduled verification ("Adaptive Verification in vLLM",
 *   sections "Scheduling the budget" and "The cost model"): survival is the
 *   running product of the per-position confidences; the best B slots over
 *   all requests are verified, B maximising
 *       (N_sampling + sum of the best B survivals) / cost[T + B]
 *   over a profiled step-cost table forced monotone; every request receives
 *   a contiguous prefix of its draft and the verify list is flattened across
 *   requests with per-request offsets ("How DSpark Speeds Up LLM Inference",
 *   appendix Part B: tokens flattened across requests plus a marker tensor).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is caller-owned memory.  Unless stated otherwise
 *     it is DEVICE memory of the current CUDA device.  The library never
 *     allocates, frees or synchronises, and copies to the host only in
 *     dspark_read_status().  Every call is asynchronous on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns DSPARK_ERR_INVALID_ARG or DSPARK_ERR_UNSUPPORTED
 *     and launches nothing.  A launch error returns DSPARK_ERR_CUDA.
 *   - Data anomalies found on the device never trap: the kernel writes a
 *     defined value and ORs a DSPARK_DEV_* bit into a uint32 status word that
 *     lives at offset 0 of the caller's workspace.  The word is sticky: it is
 *     cleared only by dspark_clear_status().  A workspace must be zero-filled
 *     once before its first use.
 *   - Every wait inside a kernel is bounded (about one second); a wait that
 *     gives up sets DSPARK_DEV_TIMEOUT and the kernel returns.
 *   - Calls that share a workspace must not overlap on the GPU.
 *   - Index arrays are int32; slot ids are n*K + k.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st *dspark_stream_t;

typedef int32_t dspark_status;
#define DSPARK_OK              0
#define DSPARK_ERR_INVALID_ARG 1   /* NULL pointer, bad size, stride or alignment */
#define DSPARK_ERR_UNSUPPORTED 2   /* valid but outside what this build handles */
#define DSPARK_ERR_CUDA        3   /* a CUDA call or launch failed */
#define DSPARK_ERR_WORKSPACE   4   /* workspace NULL or smaller than required */

/* logits element types */
#define DSPARK_BF16 0
#define DSPARK_F32  1

/* device status bits (status word at offset 0 of a workspace) */
#define DSPARK_DEV_TOKEN_OOR   1u   /* last_token outside [0, vocab): 0 used instead */
#define DSPARK_DEV_NAN_LOGIT   2u   /* an adjusted logit was NaN; it won its row */
#define DSPARK_DEV_CONF_OOR    4u   /* confidence NaN or outside [0,1]: clamped, NaN -> 0 */
#define DSPARK_DEV_TABLE_SHORT 8u   /* T outside [0, cost_len): B = 0 */
#define DSPARK_DEV_COST_NONPOS 16u  /* a cost (+ draft_cost) in use was <= 0 or NaN */
#define DSPARK_DEV_TIMEOUT     32u  /* a bounded wait gave up; outputs undefined */

/* scheduler flags */
#define DSPARK_COST_FORCE_MONOTONE   1u  /* use cost'[n] = max_{m<=n} cost[m] */
#define DSPARK_COST_FORCE_SUFFIX_MIN 2u  /* use cost'[n] = min_{m>=n} cost[m] */
#define DSPARK_BUDGET_GREEDY_STOP    4u  /* admit slots while the objective strictly rises */

/* ------------------------------------------------------------------------
 * Chaining.  "DSpark on MAX", "What DSpark is", item 3: a low-rank bias keyed
 * on the previous chosen token, then an argmax.
 *
 * logits       [N, K, vocab] of logits_dtype; element (n, k, v) at
 *              n*stride_n + k*stride_k + v (elements).  vocab, stride_n and
 *              stride_k must be multiples of 16 bytes / element size, and
 *              the base 16-byte aligned.
 * U, V         bf16 [vocab, rank] row-major each, 16-byte aligned.
 * last_token   [N] int32: the token before draft position 0.  Values outside
 *              [0, vocab) are replaced by 0 and flag DSPARK_DEV_TOKEN_OOR.
 * draft_tokens out [N, K] int32, row-major.  draft[n,k] is the first index of
 *              the maximum of logits[n,k,:] + U[prev] . V^T (fp32 arithmetic,
 *              bf16 products accumulated in fp32); a NaN ranks above every
 *              number, so the first NaN wins and DSPARK_DEV_NAN_LOGIT is set.
 *              An index outside [0, vocab) is never written.
 * draft_score  optional out [N, K] fp32: the adjusted value at draft[n,k];
 *              NULL to skip.
 * workspace    >= dspark_chain_workspace_size(N, K) bytes, 256-byte aligned,
 *              zero-filled before its first use.  Word 1 (bytes 4..7) is a
 *              test hook: nonzero makes every barrier between positions wait
 *              for one arrival more than can come, so the wait runs out after
 *              its time limit and the call ends with DSPARK_DEV_TIMEOUT and
 *              undefined drafts.  It exists to exercise the timeout path;
 *              keep it zero.
 * Limits: 1 <= N <= 128 * (SM count), 1 <= K <= 32, 8 <= vocab < 2^31,
 * rank a multiple of 16 in [16, 256].
 * ------------------------------------------------------------------------ */
DSPARK_API size_t dspark_chain_workspace_size(int32_t N, int32_t K);

DSPARK_API dspark_status dspark_chain_draft(
    const void *logits, int32_t logits_dtype,
    int64_t logits_stride_n, int64_t logits_stride_k,
    const void *U, const void *V,
    const int32_t *last_token,
    int32_t N, int32_t K, int32_t vocab, int32_t rank,
    int32_t *draft_tokens, float *draft_score,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * Probabilistic drafting.  "Adaptive Verification in vLLM", "Appendix:
 * reproducing": the drafter runs with draft_sample_method "probabilistic",
 * drawing each draft token from the adjusted distribution instead of taking
 * its argmax.  Same chain, same arguments and limits as dspark_chain_draft,
 * except that draft[n,k] ~ softmax(adj[n,k,:] / temperature) given the
 * earlier tokens, drawn in two steps over blocks of 16 vocabulary entries
 * (block j = entries 16j .. 16j+15): the block with the largest
 *     key_j = log sum_{v in j} exp(adj[n,k,v] / temperature) + g_j,
 * g_j = -ln(-ln u_j) (the Gumbel-max rule over blocks: block j wins with
 * probability Z_j / sum Z), then the first entry of that block whose
 * cumulative weight exp(adj / temperature) exceeds c_j times the block's
 * total (entry v wins with probability exp(adj_v / temperature) / Z_j).  A
 * block holding a NaN has key NaN, NaN ranks highest, and its entry is its
 * first NaN; ties go to the lower index.  u_j and c_j come from a
 * counter-based generator: words 2 (j % 2) and 2 (j % 2) + 1 of
 * Philox4x32-10 (Salmon et al., SC 2011) with counter (j / 2, n, k, offset)
 * and key (seed low 32 bits, seed high 32 bits), u = (2 (x >> 9) + 1) / 2^24
 * for a word x; the keys are fp32.  The same (seed, offset) reproduces the
 * same drafts; a caller advances offset every decoding step.
 * temperature  > 0 and finite with a finite reciprocal, else
 *              DSPARK_ERR_INVALID_ARG.
 * draft_score  optional out [N, K]: the winning block's key key_j.
 * ------------------------------------------------------------------------ */
DSPARK_API dspark_status dspark_chain_sample(
    const void *logits, int32_t logits_dtype,
    int64_t logits_stride_n, int64_t logits_stride_k,
    const void *U, const void *V,
    const int32_t *last_token,
    int32_t N, int32_t K, int32_t vocab, int32_t rank,
    uint64_t seed, uint32_t offset, float temperature,
    int32_t *draft_tokens, float *draft_score,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused output projection.  "DSpark on MAX", "What DSpark is", items 2-3:
 * the block drafter scores all K positions in one pass and the chain adds
 * the low-rank bias before the argmax.  This call takes the drafter's hidden
 * states and output projection instead of its logits and computes
 *     adj[n,k,v] = h[n,k,:] . W[v,:] + U[prev] . V[v,:]
 * as one product with inner dimension d + rank (bf16 operands, fp32
 * accumulation), so the backbone logits are never written to memory.  The
 * chain, argmax rule, status bits, workspace and limits are those of
 * dspark_chain_draft.
 * h           bf16 [N, K, d]; element (n, k, j) at n*h_stride_n +
 *             k*h_stride_k + j (elements); strides multiples of 8, base
 *             16-byte aligned.
 * W           bf16 [vocab, d] row-major, 16-byte aligned.
 * d           a multiple of 64 in [64, 65536]; vocab a multiple of 8.
 * draft_score optional out [N, K]: adj at draft[n,k].
 * ------------------------------------------------------------------------ */
DSPARK_API dspark_status dspark_chain_lmhead(
    const void *h, int64_t h_stride_n, int64_t h_stride_k,
    const void *W, const void *U, const void *V,
    const int32_t *last_token,
    int32_t N, int32_t K, int32_t vocab, int32_t d, int32_t rank,
    int32_t *draft_tokens, float *draft_score,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * dspark_chain_draft for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is an interface convenience, not part of
 * the method.  Serving engines that reserve the whole device memory at
 * start-up and allow no later allocation, plugins running under a host
 * runtime that owns every allocation, and latency-critical code where
 * cudaMalloc (which may synchronise the device) is not permitted cannot hand
 * out the chain workspace; this call takes its scratch from a fixed array in
 * the library's own device memory instead, and allocates nothing (no
 * cudaMalloc, cudaFree or allocating library call).
 *
 * Arguments and results are those of dspark_chain_draft, without the
 * workspace.  device_status: optional device pointer to a uint32 that
 * receives this call's DSPARK_DEV_* bits (overwritten, not ORed); NULL to
 * discard them.
 * Limit: 256 + N*K*8 + K*ceil(N/128)*4 <= 262144 bytes of scratch (N = 1024,
 * K = 15 fits); larger sizes return DSPARK_ERR_UNSUPPORTED.  Every argument
 * check (those of dspark_chain_draft and this limit) runs before the first
 * CUDA call, so a rejected call enqueues nothing.  The scratch array
 * (256 KiB) stays allocated on every GPU that loaded the library until the
 * process exits.  The first call on each device looks up the array's device
 * address with cudaGetSymbolAddress (that device must be current), and so
 * does the first call after the device's context was replaced (for example
 * by cudaDeviceReset).
 * Every call shares the one array and keeps the last call's contents (each
 * call clears what must start at zero), so calls that overlap on the GPU
 * race: order them on one stream or with events.
 * ------------------------------------------------------------------------ */
DSPARK_API dspark_status dspark_chain_draft_noalloc(
    const void *logits, int32_t logits_dtype,
    int64_t logits_stride_n, int64_t logits_stride_k,
    const void *U, const void *V,
    const int32_t *last_token,
    int32_t N, int32_t K, int32_t vocab, int32_t rank,
    int32_t *draft_tokens, float *draft_score,
    uint32_t *device_status, dspark_stream_t stream);

/* ------------------------------------------------------------------------
 * Scheduler workspace: dspark_select_workspace_size() bytes, 256-byte
 * aligned, zero-filled before first use (status word at offset 0).
 * Limits of every scheduler call: 1 <= N, 1 <= K <= 32, N*K <= 16384,
 * 1 <= cost_len <= 2^30.
 * ------------------------------------------------------------------------ */
DSPARK_API size_t dspark_select_workspace_size(int32_t N, int32_t K, int32_t cost_len);

/* Survival and global order.  "Adaptive Verification in vLLM", "Scheduling
 * the budget": survival is the running product of confidences along each
 * request; slots compete globally on it.
 *
 * conf          [N, K] fp32.  Clamped into [0,1] (NaN -> 0, DSPARK_DEV_CONF_OOR).
 * sampling_mask [N] uint8, 1 = request samples this step; NULL = all sample.
 * survival      out [N, K] fp32: prod_{j<=k} conf[n,j] computed left to right
 *               in fp64 and rounded once; 0 for non-sampling requests.
 * sorted_slots  out [N*K] int32: the S = N_sampling*K eligible slot ids by
 *               survival descending, slot id ascending on ties; entries past S
 *               are left untouched.
 * prefix_sum    out [N*K+1] fp64: prefix_sum[b] = the exact sum of the first b
 *               sorted survivals (as fp64 values) rounded once to fp64, for
 *               b = 0..S.
 * n_eligible    out device scalar: S.   n_sampling out device scalar.
 */
DSPARK_API dspark_status dspark_survival_topb(
    const float *conf, const uint8_t *sampling_mask, int32_t N, int32_t K,
    float *survival, int32_t *sorted_slots, double *prefix_sum,
    int32_t *n_eligible, int32_t *n_sampling,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Budget.  "Adaptive Verification in vLLM", "Scheduling the budget" (the
 * paragraph after the formula) and "The cost model".
 *
 * prefix_sum, n_eligible, n_sampling: as written by dspark_survival_topb.
 * cost      [cost_len] fp32 microseconds, indexed by the step's token count.
 * T_dev     device scalar: tokens of the step that are not drafts.
 * draft_cost  host fp32 added to every cost (the drafter table's entry).
 * flags     DSPARK_COST_FORCE_* (forcing applied on the fly, the table is not
 *           written) and DSPARK_BUDGET_GREEDY_STOP.
 * B         out device scalar: for b = 0..b_max, b_max = min(S, cost_len-1-T),
 *           f(b) = fl(fl(N_sampling + prefix_sum[b]) / fl(cost'[T+b] + draft_cost))
 *           in fp64; B is the first maximiser (NaN ranks highest).  T outside
 *           [0, cost_len) gives B = 0 and DSPARK_DEV_TABLE_SHORT.
 * objective out device scalar fp64: f(B) (0 when the table is short).
 */
DSPARK_API dspark_status dspark_choose_budget(
    const double *prefix_sum, const int32_t *n_eligible,
    const int32_t *n_sampling, const float *cost, int32_t cost_len,
    const int32_t *T_dev, float draft_cost, uint32_t flags,
    int32_t *B, double *objective,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Allocation.  "Adaptive Verification in vLLM", "Scheduling the budget": the
 * B best slots give every request a contiguous prefix of its draft.
 * draft_len out [N] int32: number of request n's slots among sorted_slots[0..B).
 */
DSPARK_API dspark_status dspark_allocate_prefix(
    const int32_t *sorted_slots, const int32_t *B, int32_t N, int32_t K,
    int32_t *draft_len,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Compaction.  "How DSpark Speeds Up LLM Inference", appendix Part B; "Adaptive
 * Verification in vLLM", "Limitations" (logits compacted after the forward).
 * cu_len     out [N+1] int32: exclusive prefix sum of draft_len (the marker).
 * verify_idx out [N*K] int32: slot ids n*K+k for k < draft_len[n], request-
 *            major; the first cu_len[N] entries are written.
 * verify_tok optional out [N*K] int32: draft_tokens[verify_idx[j]]; needs
 *            draft_tokens [N, K]; either may be NULL (then nothing is written).
 */
DSPARK_API dspark_status dspark_compact_verify(
    const int32_t *draft_len, const int32_t *draft_tokens, int32_t N, int32_t K,
    int32_t *cu_len, int32_t *verify_idx, int32_t *verify_tok,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* The four scheduler calls above fused into one single-CTA launch that keeps
 * every intermediate on chip and never reads back to the host ("Adaptive
 * Verification in vLLM", "Scheduling the budget", last paragraph).  Outputs
 * are identical to the four calls in sequence; any of survival, sorted_slots,
 * prefix_sum, n_eligible, n_sampling, objective, verify_tok may be NULL. */
DSPARK_API dspark_status dspark_select_step(
    const float *conf, const uint8_t *sampling_mask, int32_t N, int32_t K,
    const float *cost, int32_t cost_len, const int32_t *T_dev,
    float draft_cost, uint32_t flags, const int32_t *draft_tokens,
    float *survival, int32_t *sorted_slots, double *prefix_sum,
    int32_t *n_eligible, int32_t *n_sampling,
    int32_t *B, double *objective,
    int32_t *draft_len, int32_t *cu_len, int32_t *verify_idx,
    int32_t *verify_tok,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Stale sizing.  "Adaptive Verification in vLLM", "Scheduling the budget",
 * last paragraph: B is sized from a double-buffered confidence array that is
 * one step old, while handing the B slots to requests uses current
 * confidences; "How DSpark Speeds Up LLM Inference", appendix Part B: the
 * capacity comes from confidences two steps earlier.
 * conf_size in [N, K] fp32: the older buffer, aligned slot by slot with the
 *           current batch (the caller keeps it); must not be NULL.
 * conf      in [N, K] fp32: the current confidences.
 * Every other argument is as for dspark_select_step, with the current
 * sampling_mask and T applying to both buffers.  B, objective and prefix_sum
 * come from conf_size (survival, order, exact prefix sums, f(b)); survival,
 * sorted_slots, n_eligible, n_sampling, draft_len, cu_len, verify_idx and
 * verify_tok come from conf, whose B best slots are allocated (B never
 * exceeds the eligible slot count, which both buffers share).  Status bits
 * from either buffer are raised.  One single-CTA launch, which sorts twice.
 */
DSPARK_API dspark_status dspark_select_step_stale(
    const float *conf_size, const float *conf, const uint8_t *sampling_mask,
    int32_t N, int32_t K, const float *cost, int32_t cost_len,
    const int32_t *T_dev, float draft_cost, uint32_t flags,
    const int32_t *draft_tokens, float *survival, int32_t *sorted_slots,
    double *prefix_sum, int32_t *n_eligible, int32_t *n_sampling,
    int32_t *B, double *objective,
    int32_t *draft_len, int32_t *cu_len, int32_t *verify_idx,
    int32_t *verify_tok,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Verify tokens of the compacted list: verify_tok[j] = draft_tokens[
 * verify_idx[j]] for j < *B (B and verify_idx as written by the scheduler).
 * The scheduler does not depend on the draft except for these tokens, so a
 * caller can run dspark_select_step (with draft_tokens = NULL) on a second
 * stream while dspark_chain_draft runs, join the streams, then call this;
 * dspark_chain_draft always leaves at least one SM idle for that.  Limits
 * as for the scheduler calls. */
DSPARK_API dspark_status dspark_gather_verify_tokens(
    const int32_t *verify_idx, const int32_t *B, const int32_t *draft_tokens,
    int32_t N, int32_t K, int32_t *verify_tok, dspark_stream_t stream);

/* Greedy verification of the compacted list.  "DSpark on MAX", "The kernel
 * pass", item 2: under greedy sampling a draft token is accepted iff it
 * equals the target's best token; "How DSpark Speeds Up LLM Inference",
 * "Context": the longest matching run is kept and the target adds its next
 * token.
 *
 * target_logits [R, vocab] (logits_dtype), row r at r*row_stride elements
 *               (16-byte aligned rows): each sampling request n has
 *               draft_len[n] + 1 consecutive rows, request-major (the target's
 *               outputs after the last committed token and after each of the
 *               draft_len[n] verified draft tokens); R = cu_len[N] + N_sampling.
 * draft_tokens [N, K], draft_len [N], cu_len [N+1], sampling_mask [N] (NULL =
 *               all sample): as used and written by the scheduler.
 * target_argmax out [N*(K+1)]: first-index argmax of each row (NaN ranks
 *               highest; DSPARK_DEV_NAN_LOGIT is set in the workspace status).
 * accepted, bonus out [N]: leading draft tokens equal to the target's argmax,
 *               and the target's argmax after them; -1 for non-sampling
 *               requests.
 * workspace: a scheduler workspace (status word at offset 0). */
DSPARK_API dspark_status dspark_greedy_verify(
    const void *target_logits, int32_t logits_dtype, int64_t row_stride,
    int32_t vocab, const int32_t *draft_tokens, const int32_t *draft_len,
    const int32_t *cu_len, const uint8_t *sampling_mask, int32_t N, int32_t K,
    int32_t *target_argmax, int32_t *accepted, int32_t *bonus,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Cost-table preparation.  "Adaptive Verification in vLLM", "The cost model":
 * profiling noise is removed by forcing the curve monotone; run once per
 * table.  mode = DSPARK_COST_FORCE_MONOTONE (running max from the left) or
 * DSPARK_COST_FORCE_SUFFIX_MIN (running min from the right); NaN propagates.
 * cost_in and cost_out may alias. */
DSPARK_API dspark_status dspark_force_monotone(
    const float *cost_in, float *cost_out, int32_t cost_len, uint32_t mode,
    dspark_stream_t stream);

/* Copies the workspace's status word to *host_out (host memory) and waits
 * for the copy; the only call that synchronises. */
DSPARK_API dspark_status dspark_read_status(const void *workspace, uint32_t *host_out,
                                 dspark_stream_t stream);

/* Zeroes the workspace's status word (asynchronous). */
DSPARK_API dspark_status dspark_clear_status(void *workspace, dspark_stream_t stream);

/* Number of SMs the library plans its grids for (device attribute), and the
 * library's version as major*10000 + minor*100 + patch. */
DSPARK_API int32_t dspark_sm_count(void);
DSPARK_API int32_t dspark_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H_ */
