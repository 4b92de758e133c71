// dspark_chain_draft_noalloc: the chaining call for callers that cannot
// allocate device memory.
//
// Some callers have no way to provide the scratch workspace that
// dspark_chain_draft needs: serving engines that reserve the whole device
// memory budget at start-up and allow no allocation afterwards, plugins
// called from a host runtime that owns every allocation, and code on a
// latency-critical path where cudaMalloc (which may synchronise the device)
// is not permitted.  This entry point takes its scratch (per-row winner
// slots, barrier counters, abort flag, status word) from a fixed array in
// the library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Host code cannot use the
// array's name as a device address: its device address is queried with
// cudaGetSymbolAddress, with that device current, by the first call made on
// that device (and again by the first call after the device's context was
// replaced, e.g. by cudaDeviceReset).  All calls share the one array and
// each call leaves its contents behind; the parts that must start at zero
// are cleared at the start of every call (the chain launch clears the
// per-call state, this file clears the status word).  Calls that overlap on
// the GPU would race on the array, so they must be ordered (one stream, or
// explicit events).
//
// Every argument check runs before the first CUDA call, so a rejected call
// enqueues nothing.
#include <cstdint>
#include <mutex>

#include "chain_common.cuh"
#include "dspark_internal.h"

namespace dspark {

// Largest scratch this entry point supports: 256 + N*K*8 + K*ceil(N/128)*4
// bytes must not exceed it (N = 1024, K = 15 fits; N = 4096, K = 8 does not).
constexpr size_t kNoAllocScratchBytes = 256 * 1024;

static __device__ __align__(256) unsigned char g_chain_scratch[kNoAllocScratchBytes];

// cuCtxGetCurrent, looked up once through the runtime (the library does not
// link the driver library)
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

static CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

struct ScratchSlot {
  CUcontext ctx;
  void *ptr;
};
static std::mutex g_noalloc_mu;
static ScratchSlot g_noalloc_slot[128];

// Device address of g_chain_scratch in the current device's current
// context: looked up once per device and again whenever that device's
// context has changed since (a reset reloads the module, which may move the
// array).
static cudaError_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return cudaErrorNotSupported;
  // no context current on this thread yet: the symbol lookup below makes the
  // runtime bind the device's primary context first
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  ScratchSlot &slot = g_noalloc_slot[dev];
  if (ctx == nullptr || slot.ptr == nullptr || slot.ctx != ctx) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_chain_scratch);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return cudaErrorDeviceUninitialized;
    slot.ctx = ctx;
    slot.ptr = ptr;
  }
  *out = slot.ptr;
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
  // every check before the first CUDA call: a rejected call enqueues nothing
  dspark_status s = check_chain_inputs(
      logits, logits_dtype, logits_stride_n, logits_stride_k, U, V,
      last_token, N, K, vocab, rank, draft_tokens, draft_score);
  if (s != DSPARK_OK) return s;
  const size_t need = dspark_chain_workspace_size(N, K);
  if (need == 0 || need > kNoAllocScratchBytes) return DSPARK_ERR_UNSUPPORTED;

  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // this call's status starts at zero (the array keeps the last call's)
  if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + kStatusOffset, 0,
                      sizeof(uint32_t), st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  s = dspark_chain_draft(logits, logits_dtype, logits_stride_n,
                         logits_stride_k, U, V, last_token, N, K, vocab, rank,
                         draft_tokens, draft_score, scratch,
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
