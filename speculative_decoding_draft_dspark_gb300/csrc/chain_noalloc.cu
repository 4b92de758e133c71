// dspark_chain_draft_noalloc: the chaining call for callers that cannot
// allocate device memory.
//
// Some callers have no way to provide the scratch workspace that
// dspark_chain_draft needs: code running while a CUDA graph is being
// captured (cudaMalloc is not a stream operation and is refused during
// capture), serving engines that reserve the whole device memory budget at
// start-up and allow no allocation afterwards, and plugins called from a
// host runtime that owns every allocation.  This entry point takes its
// scratch (per-row winner slots, barrier counters, abort flag, status word)
// from a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Host code cannot use the
// array's name as a device address: its device address is queried once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.  That first call should therefore come before
// any stream capture.  All calls share the one array and each call leaves
// its contents behind; the parts that must start at zero are cleared at the
// start of every call (the existing launch clears the per-call state, this
// file clears the status word).  Calls that overlap on the GPU would race
// on the array, so they must be ordered (one stream, or explicit events).
#include <cstdint>
#include <mutex>

#include "dspark_internal.h"

namespace dspark {

// Largest scratch this entry point supports: 256 + N*K*8 + K*ceil(N/128)*4
// bytes must not exceed it (N = 1024, K = 15 fits; N = 4096, K = 8 does not).
constexpr size_t kNoAllocScratchBytes = 256 * 1024;

static __device__ __align__(256) unsigned char g_chain_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[128];

// Device address of g_chain_scratch on the current device (queried once).
static cudaError_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_chain_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_chain_draft_noalloc(
    const void *logits, int32_t logits_dtype, int64_t logits_stride_n,
    int64_t logits_stride_k, const void *U, const void *V,
    const int32_t *last_token, int32_t N, int32_t K, int32_t vocab,
    int32_t rank, int32_t *draft_tokens, float *draft_score,
    uint32_t *device_status, dspark_stream_t stream) {
  if (N <= 0 || K <= 0) return DSPARK_ERR_INVALID_ARG;
  if (K > kMaxK) return DSPARK_ERR_UNSUPPORTED;
  const size_t need = dspark_chain_workspace_size(N, K);
  if (need == 0 || need > kNoAllocScratchBytes) return DSPARK_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // this call's status starts at zero (the array keeps the last call's)
  if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + kStatusOffset, 0,
                      sizeof(uint32_t), st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const dspark_status s = dspark_chain_draft(
      logits, logits_dtype, logits_stride_n, logits_stride_k, U, V, last_token,
      N, K, vocab, rank, draft_tokens, draft_score, scratch,
      kNoAllocScratchBytes, stream);
  if (s != DSPARK_OK) return s;
  if (device_status &&
      cudaMemcpyAsync(device_status,
                      static_cast<uint8_t *>(scratch) + kStatusOffset,
                      sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                      st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
