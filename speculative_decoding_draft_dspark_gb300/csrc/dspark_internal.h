// Internal interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dspark.h"

namespace dspark {

// workspace layout (bytes from the workspace base)
constexpr size_t kStatusOffset = 0;         // uint32 sticky status word
constexpr size_t kChainHangTestOffset = 4;  // uint32 test hook (see dspark.h)
constexpr size_t kChainAbortOffset = 8;     // uint32 chain abort flag
constexpr size_t kChainSlotsOffset = 256;   // uint64 [K][N] per-row winners,
                                            // then uint32 [K][N/128] counters
constexpr size_t kSelectWorkspaceBytes = 256;

inline size_t chain_counters_offset(int32_t N, int32_t K) {
  return kChainSlotsOffset + static_cast<size_t>(N) * K * 8;
}

constexpr int kMaxK = 32;
constexpr int kMaxSlots = 16384;  // N*K limit of the scheduler kernels

int device_sm_count(int dev);

struct ChainArgs {
  const void *logits;
  int32_t logits_dtype;
  int64_t stride_n, stride_k;
  const void *U, *V;
  const int32_t *last_token;
  int32_t N, K, vocab, rank;
  int32_t *draft;
  float *score;
  void *workspace;
  // probabilistic drafting (Gumbel-max with Philox4x32-10 noise)
  int32_t sample = 0;
  uint32_t seed_lo = 0, seed_hi = 0, offset = 0;
  float inv_tau = 1.0f;
};
size_t chain_workspace_bytes(int32_t N, int32_t K);
// Every host check of dspark_chain_draft except the workspace's (pointers,
// dtype, sizes, strides, alignment); touches no CUDA state.
dspark_status check_chain_inputs(const void *logits, int32_t logits_dtype,
                                 int64_t logits_stride_n,
                                 int64_t logits_stride_k, const void *U,
                                 const void *V, const int32_t *last_token,
                                 int32_t N, int32_t K, int32_t vocab,
                                 int32_t rank, const int32_t *draft_tokens,
                                 const float *draft_score);

struct LmheadArgs {
  const void *h;  // bf16 [N, K, d] (strides in elements)
  int64_t stride_n, stride_k;
  const void *W, *U, *V;  // bf16 [vocab, d], [vocab, rank], [vocab, rank]
  const int32_t *last_token;
  int32_t N, K, vocab, d, rank;
  int32_t *draft;
  float *score;
  void *workspace;
};
dspark_status lmhead_chain_launch(const LmheadArgs &a, cudaStream_t stream);
dspark_status chain_draft_launch(const ChainArgs &a, cudaStream_t stream);

struct SelectArgs {
  const float *conf;
  // optional older confidence buffer: when set (fused call only), the budget
  // is sized from it and the order and allocation use `conf`
  const float *conf_size;
  const uint8_t *mask;
  int32_t N, K;
  const float *cost;
  int32_t L;
  const int32_t *T_dev;
  float draft_cost;
  uint32_t flags;
  const int32_t *draft;
  // stage inputs for the separate calls
  const double *prefix_in;
  const int32_t *n_eligible_in;
  const int32_t *n_sampling_in;
  const int32_t *sorted_in;
  const int32_t *B_in;
  const int32_t *len_in;
  // outputs (any may be NULL where the header allows)
  float *survival;
  int32_t *sorted_slots;
  double *prefix_sum;
  int32_t *n_eligible;
  int32_t *n_sampling;
  int32_t *B;
  double *objective;
  int32_t *draft_len;
  int32_t *cu_len;
  int32_t *verify_idx;
  int32_t *verify_tok;
  uint32_t *status;
};

enum SelectStage : uint32_t {
  kStageSurvival = 1u,  // survival, order, exact prefix sums
  kStageBudget = 2u,    // budget argmax
  kStageAllocate = 4u,  // per-request prefix lengths
  kStageCompact = 8u,   // offsets and the flattened verify list
};

struct VerifyArgs {
  const void *target_logits;
  int32_t logits_dtype;
  int64_t row_stride;  // elements
  int32_t vocab;
  const int32_t *draft;
  const int32_t *draft_len;
  const int32_t *cu_len;
  const uint8_t *mask;
  int32_t N, K;
  int32_t *target_argmax;
  int32_t *accepted;
  int32_t *bonus;
  uint32_t *status;
};
dspark_status greedy_verify_launch(const VerifyArgs &a, cudaStream_t stream);

dspark_status select_launch(const SelectArgs &a, uint32_t stages,
                            cudaStream_t stream);
dspark_status gather_verify_launch(const int32_t *verify_idx,
                                   const int32_t *B_dev, const int32_t *draft,
                                   int32_t NK, int32_t *verify_tok,
                                   cudaStream_t stream);
dspark_status force_monotone_launch(const float *in, float *out, int32_t L,
                                    uint32_t mode, cudaStream_t stream);

}  // namespace dspark
