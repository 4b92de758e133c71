// C entry points of libdspark.so: host-side validation, then the launches.
// Nothing here allocates device memory or synchronises, except
// dspark_read_status(), which copies the status word to the host.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "dspark_internal.h"

namespace dspark {

static std::mutex g_sm_mu;
static int g_sm_count[128];

int device_sm_count(int dev) {
  if (dev < 0 || dev >= 128) return -1;
  std::lock_guard<std::mutex> lk(g_sm_mu);
  if (g_sm_count[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return -1;
    g_sm_count[dev] = v;
  }
  return g_sm_count[dev];
}

static bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

static dspark_status check_select_dims(int32_t N, int32_t K) {
  if (N <= 0 || K <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K > kMaxK) return DSPARK_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(N) * K > kMaxSlots) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

static dspark_status check_ws(const void *ws, size_t bytes, size_t need) {
  if (ws == nullptr || bytes < need || !aligned(ws, 256))
    return DSPARK_ERR_WORKSPACE;
  return DSPARK_OK;
}

dspark_status check_chain_inputs(const void *logits, int32_t logits_dtype,
                                 int64_t logits_stride_n,
                                 int64_t logits_stride_k, const void *U,
                                 const void *V, const int32_t *last_token,
                                 int32_t N, int32_t K, int32_t vocab,
                                 int32_t rank, const int32_t *draft_tokens,
                                 const float *draft_score) {
  if (!logits || !U || !V || !last_token || !draft_tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (logits_dtype != DSPARK_BF16 && logits_dtype != DSPARK_F32)
    return DSPARK_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || vocab <= 0 || rank <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K > kMaxK) return DSPARK_ERR_UNSUPPORTED;
  if (rank % 16 != 0 || rank > 256) return DSPARK_ERR_UNSUPPORTED;
  const int esz = logits_dtype == DSPARK_BF16 ? 2 : 4;
  const int vec = 16 / esz;  // elements per 16 bytes
  if (vocab < vec || vocab % vec != 0) return DSPARK_ERR_UNSUPPORTED;
  if (logits_stride_n < vocab || logits_stride_n % vec != 0)
    return DSPARK_ERR_INVALID_ARG;
  if (K > 1 && (logits_stride_k < vocab || logits_stride_k % vec != 0))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || !aligned(U, 16) || !aligned(V, 16))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(last_token, 4) || !aligned(draft_tokens, 4) ||
      (draft_score && !aligned(draft_score, 4)))
    return DSPARK_ERR_INVALID_ARG;
  return DSPARK_OK;
}

static dspark_status fill_chain_args(
    ChainArgs &a, const void *logits, int32_t logits_dtype,
    int64_t logits_stride_n, int64_t logits_stride_k, const void *U,
    const void *V, const int32_t *last_token, int32_t N, int32_t K,
    int32_t vocab, int32_t rank, int32_t *draft_tokens, float *draft_score,
    void *workspace, size_t workspace_bytes) {
  dspark_status s = check_chain_inputs(
      logits, logits_dtype, logits_stride_n, logits_stride_k, U, V,
      last_token, N, K, vocab, rank, draft_tokens, draft_score);
  if (s != DSPARK_OK) return s;
  s = check_ws(workspace, workspace_bytes, chain_workspace_bytes(N, K));
  if (s != DSPARK_OK) return s;
  a.logits = logits;
  a.logits_dtype = logits_dtype;
  a.stride_n = logits_stride_n;
  a.stride_k = logits_stride_k;
  a.U = U;
  a.V = V;
  a.last_token = last_token;
  a.N = N;
  a.K = K;
  a.vocab = vocab;
  a.rank = rank;
  a.draft = draft_tokens;
  a.score = draft_score;
  a.workspace = workspace;
  return DSPARK_OK;
}

static SelectArgs empty_select_args(void *ws) {
  SelectArgs a = {};
  a.status = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                          kStatusOffset);
  return a;
}

static bool flags_ok(uint32_t flags) {
  return (flags & ~(DSPARK_COST_FORCE_MONOTONE | DSPARK_COST_FORCE_SUFFIX_MIN |
                    DSPARK_BUDGET_GREEDY_STOP)) == 0;
}

static dspark_status select_step_common(
    const float *conf_size, const float *conf, const uint8_t *sampling_mask,
    int32_t N, int32_t K, const float *cost, int32_t cost_len,
    const int32_t *T_dev, float draft_cost, uint32_t flags,
    const int32_t *draft_tokens, float *survival, int32_t *sorted_slots,
    double *prefix_sum, int32_t *n_eligible, int32_t *n_sampling, int32_t *B,
    double *objective, int32_t *draft_len, int32_t *cu_len,
    int32_t *verify_idx, int32_t *verify_tok, void *workspace,
    size_t workspace_bytes, dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!conf || !cost || !T_dev || !B || !draft_len || !cu_len || !verify_idx)
    return DSPARK_ERR_INVALID_ARG;
  if (cost_len <= 0 || cost_len > (1 << 30)) return DSPARK_ERR_INVALID_ARG;
  if (!flags_ok(flags)) return DSPARK_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes)) !=
      DSPARK_OK)
    return s;
  SelectArgs a = empty_select_args(workspace);
  a.conf = conf;
  a.conf_size = conf_size;
  a.mask = sampling_mask;
  a.N = N;
  a.K = K;
  a.cost = cost;
  a.L = cost_len;
  a.T_dev = T_dev;
  a.draft_cost = draft_cost;
  a.flags = flags;
  a.draft = draft_tokens;
  a.survival = survival;
  a.sorted_slots = sorted_slots;
  a.prefix_sum = prefix_sum;
  a.n_eligible = n_eligible;
  a.n_sampling = n_sampling;
  a.B = B;
  a.objective = objective;
  a.draft_len = draft_len;
  a.cu_len = cu_len;
  a.verify_idx = verify_idx;
  a.verify_tok = verify_tok;
  return select_launch(a,
                       kStageSurvival | kStageBudget | kStageAllocate |
                           kStageCompact,
                       reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace dspark

using namespace dspark;

extern "C" {

int32_t dspark_version(void) { return 100; }

int32_t dspark_sm_count(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return device_sm_count(dev);
}

size_t dspark_chain_workspace_size(int32_t N, int32_t K) {
  if (N <= 0 || K <= 0) return 0;
  return chain_workspace_bytes(N, K);
}

dspark_status dspark_chain_draft(const void *logits, int32_t logits_dtype,
                                 int64_t logits_stride_n,
                                 int64_t logits_stride_k, const void *U,
                                 const void *V, const int32_t *last_token,
                                 int32_t N, int32_t K, int32_t vocab,
                                 int32_t rank, int32_t *draft_tokens,
                                 float *draft_score, void *workspace,
                                 size_t workspace_bytes,
                                 dspark_stream_t stream) {
  ChainArgs a;
  const dspark_status s = fill_chain_args(
      a, logits, logits_dtype, logits_stride_n, logits_stride_k, U, V,
      last_token, N, K, vocab, rank, draft_tokens, draft_score, workspace,
      workspace_bytes);
  if (s != DSPARK_OK) return s;
  return chain_draft_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_chain_sample(const void *logits, int32_t logits_dtype,
                                  int64_t logits_stride_n,
                                  int64_t logits_stride_k, const void *U,
                                  const void *V, const int32_t *last_token,
                                  int32_t N, int32_t K, int32_t vocab,
                                  int32_t rank, uint64_t seed, uint32_t offset,
                                  float temperature, int32_t *draft_tokens,
                                  float *draft_score, void *workspace,
                                  size_t workspace_bytes,
                                  dspark_stream_t stream) {
  if (!(temperature > 0.0f) || !std::isfinite(temperature) ||
      !std::isfinite(1.0f / temperature))
    return DSPARK_ERR_INVALID_ARG;
  ChainArgs a;
  const dspark_status s = fill_chain_args(
      a, logits, logits_dtype, logits_stride_n, logits_stride_k, U, V,
      last_token, N, K, vocab, rank, draft_tokens, draft_score, workspace,
      workspace_bytes);
  if (s != DSPARK_OK) return s;
  a.sample = 1;
  a.seed_lo = static_cast<uint32_t>(seed);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  a.offset = offset;
  a.inv_tau = 1.0f / temperature;
  return chain_draft_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_chain_lmhead(const void *h, int64_t h_stride_n,
                                  int64_t h_stride_k, const void *W,
                                  const void *U, const void *V,
                                  const int32_t *last_token, int32_t N,
                                  int32_t K, int32_t vocab, int32_t d,
                                  int32_t rank, int32_t *draft_tokens,
                                  float *draft_score, void *workspace,
                                  size_t workspace_bytes,
                                  dspark_stream_t stream) {
  if (!h || !W || !U || !V || !last_token || !draft_tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || vocab <= 0 || d <= 0 || rank <= 0)
    return DSPARK_ERR_INVALID_ARG;
  if (K > kMaxK) return DSPARK_ERR_UNSUPPORTED;
  if (rank % 16 != 0 || rank > 256) return DSPARK_ERR_UNSUPPORTED;
  if (d % 64 != 0 || d > 65536) return DSPARK_ERR_UNSUPPORTED;
  if (vocab < 8 || vocab % 8 != 0) return DSPARK_ERR_UNSUPPORTED;
  if (h_stride_n < d || h_stride_n % 8 != 0) return DSPARK_ERR_INVALID_ARG;
  if (K > 1 && (h_stride_k < d || h_stride_k % 8 != 0)) return DSPARK_ERR_INVALID_ARG;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(U, 16) || !aligned(V, 16))
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned(last_token, 4) || !aligned(draft_tokens, 4) ||
      (draft_score && !aligned(draft_score, 4)))
    return DSPARK_ERR_INVALID_ARG;
  const dspark_status s =
      check_ws(workspace, workspace_bytes, chain_workspace_bytes(N, K));
  if (s != DSPARK_OK) return s;
  LmheadArgs a;
  a.h = h;
  a.stride_n = h_stride_n;
  a.stride_k = h_stride_k;
  a.W = W;
  a.U = U;
  a.V = V;
  a.last_token = last_token;
  a.N = N;
  a.K = K;
  a.vocab = vocab;
  a.d = d;
  a.rank = rank;
  a.draft = draft_tokens;
  a.score = draft_score;
  a.workspace = workspace;
  return lmhead_chain_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t dspark_select_workspace_size(int32_t N, int32_t K, int32_t cost_len) {
  if (N <= 0 || K <= 0 || cost_len <= 0) return 0;
  return kSelectWorkspaceBytes;
}

dspark_status dspark_survival_topb(const float *conf,
                                   const uint8_t *sampling_mask, int32_t N,
                                   int32_t K, float *survival,
                                   int32_t *sorted_slots, double *prefix_sum,
                                   int32_t *n_eligible, int32_t *n_sampling,
                                   void *workspace, size_t workspace_bytes,
                                   dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!conf || !survival || !sorted_slots || !prefix_sum || !n_eligible ||
      !n_sampling)
    return DSPARK_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes)) !=
      DSPARK_OK)
    return s;
  SelectArgs a = empty_select_args(workspace);
  a.conf = conf;
  a.mask = sampling_mask;
  a.N = N;
  a.K = K;
  a.survival = survival;
  a.sorted_slots = sorted_slots;
  a.prefix_sum = prefix_sum;
  a.n_eligible = n_eligible;
  a.n_sampling = n_sampling;
  return select_launch(a, kStageSurvival, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_choose_budget(const double *prefix_sum,
                                   const int32_t *n_eligible,
                                   const int32_t *n_sampling, const float *cost,
                                   int32_t cost_len, const int32_t *T_dev,
                                   float draft_cost, uint32_t flags,
                                   int32_t *B, double *objective,
                                   void *workspace, size_t workspace_bytes,
                                   dspark_stream_t stream) {
  if (!prefix_sum || !n_eligible || !n_sampling || !cost || !T_dev || !B)
    return DSPARK_ERR_INVALID_ARG;
  if (cost_len <= 0 || cost_len > (1 << 30)) return DSPARK_ERR_INVALID_ARG;
  if (!flags_ok(flags)) return DSPARK_ERR_INVALID_ARG;
  dspark_status s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes);
  if (s != DSPARK_OK) return s;
  SelectArgs a = empty_select_args(workspace);
  // N*K is only used to clamp the eligible count read from the device
  a.N = kMaxSlots;
  a.K = 1;
  a.prefix_in = prefix_sum;
  a.n_eligible_in = n_eligible;
  a.n_sampling_in = n_sampling;
  a.cost = cost;
  a.L = cost_len;
  a.T_dev = T_dev;
  a.draft_cost = draft_cost;
  a.flags = flags;
  a.B = B;
  a.objective = objective;
  return select_launch(a, kStageBudget, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_allocate_prefix(const int32_t *sorted_slots,
                                     const int32_t *B, int32_t N, int32_t K,
                                     int32_t *draft_len, void *workspace,
                                     size_t workspace_bytes,
                                     dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!sorted_slots || !B || !draft_len) return DSPARK_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes)) !=
      DSPARK_OK)
    return s;
  SelectArgs a = empty_select_args(workspace);
  a.N = N;
  a.K = K;
  a.sorted_in = sorted_slots;
  a.B_in = B;
  a.draft_len = draft_len;
  return select_launch(a, kStageAllocate, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_compact_verify(const int32_t *draft_len,
                                    const int32_t *draft_tokens, int32_t N,
                                    int32_t K, int32_t *cu_len,
                                    int32_t *verify_idx, int32_t *verify_tok,
                                    void *workspace, size_t workspace_bytes,
                                    dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!draft_len || !cu_len || !verify_idx) return DSPARK_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes)) !=
      DSPARK_OK)
    return s;
  SelectArgs a = empty_select_args(workspace);
  a.N = N;
  a.K = K;
  a.len_in = draft_len;
  a.draft = draft_tokens;
  a.cu_len = cu_len;
  a.verify_idx = verify_idx;
  a.verify_tok = verify_tok;
  return select_launch(a, kStageCompact, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_select_step(
    const float *conf, const uint8_t *sampling_mask, int32_t N, int32_t K,
    const float *cost, int32_t cost_len, const int32_t *T_dev,
    float draft_cost, uint32_t flags, const int32_t *draft_tokens,
    float *survival, int32_t *sorted_slots, double *prefix_sum,
    int32_t *n_eligible, int32_t *n_sampling, int32_t *B, double *objective,
    int32_t *draft_len, int32_t *cu_len, int32_t *verify_idx,
    int32_t *verify_tok, void *workspace, size_t workspace_bytes,
    dspark_stream_t stream) {
  return dspark::select_step_common(
      nullptr, conf, sampling_mask, N, K, cost, cost_len, T_dev, draft_cost,
      flags, draft_tokens, survival, sorted_slots, prefix_sum, n_eligible,
      n_sampling, B, objective, draft_len, cu_len, verify_idx, verify_tok,
      workspace, workspace_bytes, stream);
}

dspark_status dspark_select_step_stale(
    const float *conf_size, const float *conf, const uint8_t *sampling_mask,
    int32_t N, int32_t K, const float *cost, int32_t cost_len,
    const int32_t *T_dev, float draft_cost, uint32_t flags,
    const int32_t *draft_tokens, float *survival, int32_t *sorted_slots,
    double *prefix_sum, int32_t *n_eligible, int32_t *n_sampling, int32_t *B,
    double *objective, int32_t *draft_len, int32_t *cu_len,
    int32_t *verify_idx, int32_t *verify_tok, void *workspace,
    size_t workspace_bytes, dspark_stream_t stream) {
  if (!conf_size) return DSPARK_ERR_INVALID_ARG;
  return dspark::select_step_common(
      conf_size, conf, sampling_mask, N, K, cost, cost_len, T_dev, draft_cost,
      flags, draft_tokens, survival, sorted_slots, prefix_sum, n_eligible,
      n_sampling, B, objective, draft_len, cu_len, verify_idx, verify_tok,
      workspace, workspace_bytes, stream);
}

dspark_status dspark_gather_verify_tokens(const int32_t *verify_idx,
                                         const int32_t *B,
                                         const int32_t *draft_tokens, int32_t N,
                                         int32_t K, int32_t *verify_tok,
                                         dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!verify_idx || !B || !draft_tokens || !verify_tok)
    return DSPARK_ERR_INVALID_ARG;
  return gather_verify_launch(verify_idx, B, draft_tokens, N * K, verify_tok,
                              reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_greedy_verify(
    const void *target_logits, int32_t logits_dtype, int64_t row_stride,
    int32_t vocab, const int32_t *draft_tokens, const int32_t *draft_len,
    const int32_t *cu_len, const uint8_t *sampling_mask, int32_t N, int32_t K,
    int32_t *target_argmax, int32_t *accepted, int32_t *bonus,
    void *workspace, size_t workspace_bytes, dspark_stream_t stream) {
  dspark_status s = check_select_dims(N, K);
  if (s != DSPARK_OK) return s;
  if (!target_logits || !draft_tokens || !draft_len || !cu_len ||
      !target_argmax || !accepted || !bonus)
    return DSPARK_ERR_INVALID_ARG;
  if (logits_dtype != DSPARK_BF16 && logits_dtype != DSPARK_F32)
    return DSPARK_ERR_INVALID_ARG;
  const int vec = logits_dtype == DSPARK_BF16 ? 8 : 4;
  if (vocab <= 0 || vocab % vec != 0) return DSPARK_ERR_UNSUPPORTED;
  if (row_stride < vocab || row_stride % vec != 0 || !aligned(target_logits, 16))
    return DSPARK_ERR_INVALID_ARG;
  if ((s = check_ws(workspace, workspace_bytes, kSelectWorkspaceBytes)) !=
      DSPARK_OK)
    return s;
  VerifyArgs a;
  a.target_logits = target_logits;
  a.logits_dtype = logits_dtype;
  a.row_stride = row_stride;
  a.vocab = vocab;
  a.draft = draft_tokens;
  a.draft_len = draft_len;
  a.cu_len = cu_len;
  a.mask = sampling_mask;
  a.N = N;
  a.K = K;
  a.target_argmax = target_argmax;
  a.accepted = accepted;
  a.bonus = bonus;
  a.status = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) +
                                          kStatusOffset);
  return greedy_verify_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_force_monotone(const float *cost_in, float *cost_out,
                                    int32_t cost_len, uint32_t mode,
                                    dspark_stream_t stream) {
  if (!cost_in || !cost_out || cost_len <= 0) return DSPARK_ERR_INVALID_ARG;
  if (mode != DSPARK_COST_FORCE_MONOTONE && mode != DSPARK_COST_FORCE_SUFFIX_MIN)
    return DSPARK_ERR_INVALID_ARG;
  return force_monotone_launch(cost_in, cost_out, cost_len, mode,
                               reinterpret_cast<cudaStream_t>(stream));
}

dspark_status dspark_read_status(const void *workspace, uint32_t *host_out,
                                 dspark_stream_t stream) {
  if (!workspace || !host_out) return DSPARK_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out,
                      static_cast<const uint8_t *>(workspace) + kStatusOffset,
                      sizeof(uint32_t), cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status dspark_clear_status(void *workspace, dspark_stream_t stream) {
  if (!workspace) return DSPARK_ERR_INVALID_ARG;
  return cudaMemsetAsync(static_cast<uint8_t *>(workspace) + kStatusOffset, 0,
                         sizeof(uint32_t),
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ERR_CUDA;
}

}  // extern "C"
