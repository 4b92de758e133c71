// Greedy verification of the compacted verify list on sm_103a.
//
// "DSpark on MAX", section "The kernel pass", item 2: under greedy sampling
// acceptance is "does the guess equal the target's best token"; "How DSpark
// Speeds Up LLM Inference", section "Context": the target keeps the longest
// matching run of the guess and adds its own next token.
//
// row_argmax_kernel: the target's best token of every verify row (one row
// per verified draft token plus the bonus position of each sampling
// request).  A persistent grid, two CTAs per SM, streams rows through a
// 6-stage ring of 16 KB shared-memory buffers per CTA filled by 1-D bulk
// copies (one producer thread).  Each thread of the 16 consumer warps takes
// two 16-byte vectors of a stage, reduces their values with packed
// NaN-propagating bf16x2 max instructions and keeps only its running maximum
// and the first stage that held it: no index work per element (the "eight
// values per load" lesson of the same section, carried further).  At the end
// of a row the lanes holding their warp's maximum re-read their 32 bytes of
// that stage, which the row streamed moments earlier, to find its first
// position.  Ties keep the lowest
// index; the first NaN wins.
//
// greedy_accept_kernel: per sampling request, the leading draft tokens that
// equal the target's best tokens, and the target's token after them (bonus).
#include <climits>
#include <cuda_bf16.h>
#include <mutex>

#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int VA_CONSUMER_WARPS = 16;
constexpr int VA_THREADS = (VA_CONSUMER_WARPS + 1) * 32;
constexpr int VA_CHUNK = 16384;  // bytes per stage
constexpr int VA_STAGES = 6;
constexpr int VA_CTAS_PER_SM = 2;  // two rows in flight per SM
// 16-byte vectors per consumer thread in a full stage
constexpr int VA_VPT = VA_CHUNK / 16 / (VA_CONSUMER_WARPS * 32);
constexpr int VA_RING = VA_STAGES + 1;  // row-partial buffers in flight
constexpr int VA_SMEM_BYTES =
    VA_STAGES * VA_CHUNK + 2 * VA_STAGES * 8 +
    VA_RING * (VA_CONSUMER_WARPS * 8 + 8) + 64 + 128;

struct RowArgmaxParams {
  const uint8_t *logits;
  int64_t row_stride_bytes;
  int32_t vocab;
  const int32_t *cu_len;
  const uint8_t *mask;
  int32_t N;
  int32_t *out;
  uint32_t *status;
};

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// NaN-propagating max of two bf16 pairs
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int LDT>
__global__ void __launch_bounds__(VA_THREADS, VA_CTAS_PER_SM)
    row_argmax_kernel(const RowArgmaxParams p) {
  extern __shared__ __align__(128) uint8_t vsm[];
  uint8_t *stages = vsm;
  uint64_t *full = reinterpret_cast<uint64_t *>(vsm + VA_STAGES * VA_CHUNK);
  uint64_t *empty = full + VA_STAGES;
  unsigned long long *partial = reinterpret_cast<unsigned long long *>(empty + VA_STAGES);
  // partial[b * (VA_CONSUMER_WARPS + 1) + w]; the last entry of each buffer
  // is the warps-done counter
  volatile uint32_t *abort_flag =
      reinterpret_cast<uint32_t *>(partial + VA_RING * (VA_CONSUMER_WARPS + 1));
  __shared__ int sh_ns[33];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int ESZ = LDT == DSPARK_BF16 ? 2 : 4;
  constexpr int EPV = 16 / ESZ;  // elements per 16-byte vector

  // rows to verify: sum of draft lengths plus one per sampling request
  int my = 0;
  for (int n = tid; n < p.N; n += blockDim.x) my += (p.mask == nullptr || p.mask[n]) ? 1 : 0;
  for (int o = 16; o > 0; o >>= 1) my += __shfl_down_sync(0xFFFFFFFFu, my, o);
  if (lane == 0) sh_ns[warp] = my;
  if (tid == 0) {
    for (int i = 0; i < VA_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], VA_CONSUMER_WARPS);
    }
    for (int b = 0; b < VA_RING; ++b)
      reinterpret_cast<volatile unsigned long long *>(partial)[b * (VA_CONSUMER_WARPS + 1) + VA_CONSUMER_WARPS] = 0ull;
    *abort_flag = 0u;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (tid == 0) {
    int ns = 0;
    for (int w = 0; w < VA_THREADS / 32; ++w) ns += sh_ns[w];
    sh_ns[32] = ns;
  }
  __syncthreads();
  const int R = p.cu_len[p.N] + sh_ns[32];
  const uint32_t row_bytes = static_cast<uint32_t>(p.vocab) * ESZ;
  const int chunks = static_cast<int>((row_bytes + VA_CHUNK - 1) / VA_CHUNK);

  if (warp == VA_CONSUMER_WARPS) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int it = 0;
      int last_it[VA_STAGES];
      for (int s = 0; s < VA_STAGES; ++s) last_it[s] = -1;
      bool ok = true;
      for (int r = blockIdx.x; r < R && ok; r += gridDim.x) {
        const uint8_t *row = p.logits + static_cast<int64_t>(r) * p.row_stride_bytes;
        for (int c = 0; c < chunks; ++c, ++it) {
          const int s = it % VA_STAGES;
          const uint32_t ph = (it / VA_STAGES) & 1;
          if (!(ok = wait_bounded(&empty[s], ph ^ 1u, abort_flag, p.status))) break;
          const uint32_t off = static_cast<uint32_t>(c) * VA_CHUNK;
          const uint32_t bytes = min(static_cast<uint32_t>(VA_CHUNK), row_bytes - off);
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_copy_g2s(stages + s * VA_CHUNK, row + off, bytes, &full[s]);
          last_it[s] = it;
        }
      }
      if (!ok) {
        for (int s = 0; s < VA_STAGES; ++s) {
          if (last_it[s] < 0) continue;
          const uint32_t par = (last_it[s] / VA_STAGES) & 1;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&full[s], par) && global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- consumers
    const int ct = tid;  // 0 .. 8*32-1
    constexpr int NCT = VA_CONSUMER_WARPS * 32;
    // fill for vectors past the end of a ragged stage: -inf never beats a
    // real value and the index search below skips those vectors
    constexpr uint32_t NEG_INF_WORD = LDT == DSPARK_BF16 ? 0xFF80FF80u : 0xFF800000u;
    int it = 0, rl = 0;
    bool ok = true;
    for (int r = blockIdx.x; r < R && ok; r += gridDim.x, ++rl) {
      // per thread: its largest value in the row and the first stage holding
      // it; where in that stage is found once, at the end of the row
      float best = -INFINITY;
      int best_c = -1;
      for (int c = 0; c < chunks; ++c, ++it) {
        const int s = it % VA_STAGES;
        const uint32_t ph = (it / VA_STAGES) & 1;
        ok = __all_sync(0xFFFFFFFFu, wait_bounded(&full[s], ph, abort_flag, p.status));
        if (!ok) break;
        const uint32_t off = static_cast<uint32_t>(c) * VA_CHUNK;
        const int nvec = static_cast<int>(min(static_cast<uint32_t>(VA_CHUNK), row_bytes - off) / 16);
        const uint32_t base = smem_u32(stages + s * VA_CHUNK);
        uint4 w[VA_VPT];
#pragma unroll
        for (int u = 0; u < VA_VPT; ++u) {
          const int v = ct + u * NCT;  // ascending index with u
          w[u] = v < nvec ? ld_shared_v4(base + v * 16)
                          : make_uint4(NEG_INF_WORD, NEG_INF_WORD, NEG_INF_WORD, NEG_INF_WORD);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        float m;
        if constexpr (LDT == DSPARK_BF16) {
          uint32_t t[VA_VPT];
#pragma unroll
          for (int u = 0; u < VA_VPT; ++u)
            t[u] = bf16x2_max_nan(bf16x2_max_nan(w[u].x, w[u].y), bf16x2_max_nan(w[u].z, w[u].w));
#pragma unroll
          for (int h = VA_VPT / 2; h >= 1; h >>= 1)
#pragma unroll
            for (int u = 0; u < h; ++u) t[u] = bf16x2_max_nan(t[u], t[u + h]);
          m = fmax_nan(bf16_lo(t[0]), bf16_hi(t[0]));
        } else {
          float t[VA_VPT];
#pragma unroll
          for (int u = 0; u < VA_VPT; ++u)
            t[u] = fmax_nan(fmax_nan(__uint_as_float(w[u].x), __uint_as_float(w[u].y)),
                            fmax_nan(__uint_as_float(w[u].z), __uint_as_float(w[u].w)));
#pragma unroll
          for (int h = VA_VPT / 2; h >= 1; h >>= 1)
#pragma unroll
            for (int u = 0; u < h; ++u) t[u] = fmax_nan(t[u], t[u + h]);
          m = t[0];
        }
        // strictly larger (or the first NaN): earlier stages keep ties
        const bool better = ct < nvec && (best_c < 0 || m > best || (m != m && best == best));
        best = better ? m : best;
        best_c = better ? c : best_c;
      }
      if (!ok) break;
      // warp maximum; the lanes holding it find their first position in
      // their stage by re-reading those bytes (just streamed, so from L2)
      const uint32_t key = best_c >= 0 ? f32_key(best) : 0u;
      const uint32_t wkey = __reduce_max_sync(0xFFFFFFFFu, key);
      int idx = INT_MAX;
      if (best_c >= 0 && key == wkey) {
        const uint32_t off = static_cast<uint32_t>(best_c) * VA_CHUNK;
        const int nvec = static_cast<int>(min(static_cast<uint32_t>(VA_CHUNK), row_bytes - off) / 16);
        const uint8_t *src = p.logits + static_cast<int64_t>(r) * p.row_stride_bytes + off;
        const bool want_nan = best != best;
        for (int u = VA_VPT - 1; u >= 0; --u) {
          const int v = ct + u * NCT;
          if (v >= nvec) continue;
          const uint4 w = __ldg(reinterpret_cast<const uint4 *>(src + static_cast<size_t>(v) * 16));
          float vals[EPV];
          if constexpr (LDT == DSPARK_BF16) {
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              vals[2 * h] = bf16_lo(ww[h]);
              vals[2 * h + 1] = bf16_hi(ww[h]);
            }
          } else {
            vals[0] = __uint_as_float(w.x);
            vals[1] = __uint_as_float(w.y);
            vals[2] = __uint_as_float(w.z);
            vals[3] = __uint_as_float(w.w);
          }
#pragma unroll
          for (int e = EPV - 1; e >= 0; --e) {
            const bool hit = want_nan ? (vals[e] != vals[e]) : (vals[e] == best);
            idx = hit ? static_cast<int>(off / ESZ) + v * EPV + e : idx;
          }
        }
      }
      idx = __reduce_min_sync(0xFFFFFFFFu, idx);
      const uint32_t key_w = wkey;
      const int b = rl % VA_RING;
      volatile unsigned long long *pb =
          reinterpret_cast<volatile unsigned long long *>(partial) + b * (VA_CONSUMER_WARPS + 1);
      if (lane == 0) {
        pb[warp] = (static_cast<unsigned long long>(key_w) << 32) |
                   static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
        __threadfence_block();
        const unsigned long long done = atomicAdd(
            const_cast<unsigned long long *>(&pb[VA_CONSUMER_WARPS]), 1ull);
        if (done == VA_CONSUMER_WARPS - 1) {  // last warp of this row
          __threadfence_block();
          unsigned long long top = 0ull;
          for (int w = 0; w < VA_CONSUMER_WARPS; ++w) top = max(top, pb[w]);
          pb[VA_CONSUMER_WARPS] = 0ull;
          int ri = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(top));
          if (top == 0ull || ri < 0 || ri >= p.vocab) ri = 0;
          p.out[r] = ri;
          if ((top >> 32) == 0xFFFFFFFFull) raise_status(p.status, DSPARK_DEV_NAN_LOGIT);
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0) *abort_flag = 1u;
  }
  __syncthreads();
}

// one CTA: per-request row offsets, accepted lengths and bonus tokens
__global__ void __launch_bounds__(1024)
    greedy_accept_kernel(const int32_t *target, const int32_t *draft,
                         const int32_t *draft_len, const uint8_t *mask,
                         const int N, const int K, int32_t *accepted,
                         int32_t *bonus) {
  __shared__ int sh[33];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int NT = blockDim.x;
  const int C = (N + NT - 1) / NT;
  const int n0 = min(N, tid * C), n1 = min(N, n0 + C);
  auto rows_of = [&](int n) {
    const bool samp = mask == nullptr || mask[n] != 0;
    int ln = draft_len[n];
    ln = ln < 0 ? 0 : (ln > K ? K : ln);
    return samp ? ln + 1 : 0;
  };
  int loc = 0;
  for (int n = n0; n < n1; ++n) loc += rows_of(n);
  int x = loc;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    const int t = lane < (NT + 31) / 32 ? sh[lane] : 0;
    int s = t;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    sh[lane] = s - t;
  }
  __syncthreads();
  int off = sh[w] + x - loc;
  for (int n = n0; n < n1; ++n) {
    const int rows = rows_of(n);
    if (rows == 0) {
      accepted[n] = -1;
      bonus[n] = -1;
      continue;
    }
    const int ln = rows - 1;
    int a = 0;
    while (a < ln && draft[static_cast<size_t>(n) * K + a] == target[off + a]) ++a;
    accepted[n] = a;
    bonus[n] = target[off + a];
    off += rows;
  }
}

// ==========================================================================
// host side
// ==========================================================================
static std::mutex g_va_mu;
static bool g_va_attr[2][128];

dspark_status greedy_verify_launch(const VerifyArgs &a, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return DSPARK_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return DSPARK_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_va_mu);
    const int t = a.logits_dtype == DSPARK_BF16 ? 0 : 1;
    if (!g_va_attr[t][dev]) {
      cudaError_t e = t == 0
          ? cudaFuncSetAttribute(row_argmax_kernel<DSPARK_BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, VA_SMEM_BYTES)
          : cudaFuncSetAttribute(row_argmax_kernel<DSPARK_F32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, VA_SMEM_BYTES);
      if (e != cudaSuccess) return DSPARK_ERR_CUDA;
      g_va_attr[t][dev] = true;
    }
  }
  RowArgmaxParams p;
  p.logits = static_cast<const uint8_t *>(a.target_logits);
  p.row_stride_bytes = a.row_stride * (a.logits_dtype == DSPARK_BF16 ? 2 : 4);
  p.vocab = a.vocab;
  p.cu_len = a.cu_len;
  p.mask = a.mask;
  p.N = a.N;
  p.out = a.target_argmax;
  p.status = a.status;
  const int rows_max = a.N * (a.K + 1);
  const int grid = std::max(1, std::min(VA_CTAS_PER_SM * sms, rows_max));
  if (a.logits_dtype == DSPARK_BF16)
    row_argmax_kernel<DSPARK_BF16><<<grid, VA_THREADS, VA_SMEM_BYTES, stream>>>(p);
  else
    row_argmax_kernel<DSPARK_F32><<<grid, VA_THREADS, VA_SMEM_BYTES, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  greedy_accept_kernel<<<1, 1024, 0, stream>>>(a.target_argmax, a.draft, a.draft_len,
                                               a.mask, a.N, a.K, a.accepted, a.bonus);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
