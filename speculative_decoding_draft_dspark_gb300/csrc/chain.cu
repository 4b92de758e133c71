// Chaining stage of the DSpark draft step on sm_103a.
//
// "DSpark on MAX", section "What DSpark is", item 3: turning the parallel
// drafter's scores into a K-token chain is a low-rank bias keyed on the
// previous chosen token followed by an argmax.  "How DSpark Speeds Up LLM
// Inference", section "Draft better": the Markov head is a rank-256
// factorisation that adjusts each word's odds using only the word before it.
//
// One launch per draft position k.  Per launch, for the 128-request tile m
// and the vocabulary tiles a CTA owns:
//
//   A = U[prev_m]        128 x r   bf16, gathered into shared memory
//   B = V[v0 : v0+256]   256 x r   bf16, streamed by TMA
//   D = A B^T            128 x 256 fp32 in tensor memory (tcgen05.mma)
//   adj = D + logits[m, k, v0 : v0+256]   (logits streamed by TMA)
//   per row: running (max, first index) over the CTA's vocabulary range
//
// so the [N x vocab] bias never leaves the SM.  The per-CTA winners are
// combined with one 64-bit atomicMax per row on a key
// (orderable(value) << 32) | (0xFFFFFFFF - index): larger value wins, then
// smaller index; NaN maps to the largest key.  The last CTA to finish writes
// draft[:, k] (and the score), which the next position's launch gathers from
// after a programmatic-dependent-launch wait.
//
// Warp roles (256 threads, one CTA per SM, all 512 TMEM columns):
//   warp 0      TMA producer of V tiles (4 K-blocks of 64 per tile)
//   warp 1      TMEM allocation; one thread issues tcgen05.mma
//   warp 2      TMA producer of logits boxes
//   warp 3      idle
//   warps 4-7   gather of U rows, then the epilogue (TMEM lane quarter w%4)
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int BM = 128;  // requests per tile (MMA M)
constexpr int BN = 256;  // vocabulary entries per tile (MMA N)
constexpr int BK = 64;   // rank entries per K-block (128 bytes of bf16)
constexpr int MAX_KB = 4;
constexpr int NUM_B_STAGES = 3;
constexpr int NUM_L_STAGES = 4;
constexpr int A_KBLOCK_BYTES = BM * 128;
constexpr int A_BYTES = MAX_KB * A_KBLOCK_BYTES;
constexpr int B_STAGE_BYTES = BN * 128;
constexpr int L_STAGE_BYTES = BM * 128;
constexpr int SMEM_A_OFF = 0;
constexpr int SMEM_B_OFF = SMEM_A_OFF + A_BYTES;
constexpr int SMEM_L_OFF = SMEM_B_OFF + NUM_B_STAGES * B_STAGE_BYTES;
constexpr int SMEM_BAR_OFF = SMEM_L_OFF + NUM_L_STAGES * L_STAGE_BYTES;
constexpr int NUM_BARS = 20;
constexpr int SMEM_USED = SMEM_BAR_OFF + NUM_BARS * 8 + 16;
constexpr int CHAIN_SMEM_BYTES = SMEM_USED + 1024;  // 1 KB alignment slack
constexpr int CHAIN_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column fp32 accumulators
constexpr uint32_t IDESC = umma_idesc_bf16_f32(BM, BN);

static_assert(CHAIN_SMEM_BYTES <= 232448, "shared memory budget");

struct ChainParams {
  const uint16_t *U;
  const int32_t *last_token;
  int32_t *draft;
  float *score;
  unsigned long long *slots;  // [N] winners of this position
  uint32_t *counter;          // CTAs finished with this position
  uint32_t *status;
  int32_t N, K, vocab, rank, k_pos;
  int32_t n_mtiles, n_vgroups, n_vtiles;
  int32_t l_k_is_dim1;  // logits map: dim1 = K, dim2 = N (else swapped)
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  return wait_bounded(bar, parity, abort_flag, status);
}

// bounded wait that ignores the abort flag (teardown of copies in flight)
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity,
                                           uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_status(status, DSPARK_DEV_TIMEOUT);
      return;
    }
  }
}

template <int LDT>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    chain_position_kernel(const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmL,
                          const ChainParams p) {
  constexpr int LBOX_COLS = (LDT == DSPARK_BF16) ? 64 : 32;  // 128-byte rows
  constexpr int NBOX = BN / LBOX_COLS;
  constexpr int CHUNKS_PER_BOX = LBOX_COLS / 32;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SMEM_BAR_OFF);
  uint64_t *b_full = bars + 0;
  uint64_t *b_empty = bars + 3;
  uint64_t *l_full = bars + 6;
  uint64_t *l_empty = bars + 10;
  uint64_t *acc_full = bars + 14;
  uint64_t *acc_empty = bars + 16;
  uint64_t *a_full = bars + 18;
  uint64_t *mma_done = bars + 19;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  volatile uint32_t *last_flag = tmem_slot + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x % p.n_mtiles;
  const int grp = blockIdx.x / p.n_mtiles;
  const int m0 = m_tile * BM;
  const int t_begin =
      static_cast<int>((static_cast<long long>(grp) * p.n_vtiles) / p.n_vgroups);
  const int t_end = static_cast<int>(
      (static_cast<long long>(grp + 1) * p.n_vtiles) / p.n_vgroups);
  const int nt = t_end - t_begin;
  // alternate the sweep direction between positions: the V tiles touched
  // last by position k are the first ones position k+1 reads, while they
  // are still in L2
  const bool ascending = (p.k_pos & 1) == 0;
  const int KB = (p.rank + BK - 1) / BK;

  if (threadIdx.x == 0) {
    pdl_launch_dependents();
    for (int i = 0; i < NUM_B_STAGES; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < NUM_L_STAGES; ++i) {
      mbar_init(&l_full[i], 1);
      mbar_init(&l_empty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(a_full, 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0u;
    *last_flag = 0u;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 64) {
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmL);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ V tile producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int last_it[NUM_B_STAGES];
      for (int s = 0; s < NUM_B_STAGES; ++s) last_it[s] = -1;
      int it = 0;
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const int t = ascending ? t_begin + i : t_end - 1 - i;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NUM_B_STAGES;
          const uint32_t ph = (it / NUM_B_STAGES) & 1;
          if (!(ok = wait_or_abort(&b_empty[s], ph ^ 1u, abort_flag, p.status)))
            break;
          mbar_arrive_expect_tx(&b_full[s], B_STAGE_BYTES);
          tma_load_2d(smem + SMEM_B_OFF + s * B_STAGE_BYTES, &tmV, &b_full[s],
                      kb * BK, t * BN, pol);
          last_it[s] = it;
        }
      }
      if (!ok) {
        for (int s = 0; s < NUM_B_STAGES; ++s)
          if (last_it[s] >= 0)
            drain_wait(&b_full[s], (last_it[s] / NUM_B_STAGES) & 1, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_u32(smem + SMEM_A_OFF);
      const uint32_t b_base = smem_u32(smem + SMEM_B_OFF);
      bool ok = wait_or_abort(a_full, 0, abort_flag, p.status);
      if (ok) tc_fence_after();
      int it = 0;
      for (int i = 0; i < nt && ok; ++i) {
        const int buf = i & 1;
        const uint32_t aph = (i >> 1) & 1;
        if (!(ok = wait_or_abort(&acc_empty[buf], aph ^ 1u, abort_flag, p.status)))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NUM_B_STAGES;
          const uint32_t ph = (it / NUM_B_STAGES) & 1;
          if (!(ok = wait_or_abort(&b_full[s], ph, abort_flag, p.status))) break;
          tc_fence_after();
          const int nk = min(BK, p.rank - kb * BK) / 16;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t ad =
                sw128_kmajor_desc(a_base + kb * A_KBLOCK_BYTES + kk * 32);
            const uint64_t bd =
                sw128_kmajor_desc(b_base + s * B_STAGE_BYTES + kk * 32);
            umma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&b_empty[s]);  // stage free once these MMAs retire
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);  // accumulator ready for the epilogue
      }
      // every MMA has retired before the CTA frees tensor memory
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.status);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------ logits producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int last_it[NUM_L_STAGES];
      for (int s = 0; s < NUM_L_STAGES; ++s) last_it[s] = -1;
      const int c1 = p.l_k_is_dim1 ? p.k_pos : m0;
      const int c2 = p.l_k_is_dim1 ? m0 : p.k_pos;
      int it = 0;
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const int t = ascending ? t_begin + i : t_end - 1 - i;
        for (int j = 0; j < NBOX; ++j, ++it) {
          const int s = it % NUM_L_STAGES;
          const uint32_t ph = (it / NUM_L_STAGES) & 1;
          if (!(ok = wait_or_abort(&l_empty[s], ph ^ 1u, abort_flag, p.status)))
            break;
          mbar_arrive_expect_tx(&l_full[s], L_STAGE_BYTES);
          tma_load_3d(smem + SMEM_L_OFF + s * L_STAGE_BYTES, &tmL, &l_full[s],
                      t * BN + j * LBOX_COLS, c1, c2, pol);
          last_it[s] = it;
        }
      }
      if (!ok) {
        for (int s = 0; s < NUM_L_STAGES; ++s)
          if (last_it[s] >= 0)
            drain_wait(&l_full[s], (last_it[s] / NUM_L_STAGES) & 1, p.status);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------ gather + epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int m = m0 + row;
    const bool row_ok = m < p.N;
    // the previous position's tokens are final once its grid has completed
    pdl_wait_primary();
    int prev = 0;
    if (row_ok) {
      if (p.k_pos == 0) {
        prev = p.last_token[m];
        if (prev < 0 || prev >= p.vocab) {
          prev = 0;
          raise_status(p.status, DSPARK_DEV_TOKEN_OOR);
        }
      } else {
        prev = p.draft[static_cast<size_t>(m) * p.K + (p.k_pos - 1)];
      }
    }
    const uint16_t *urow = p.U + static_cast<size_t>(prev) * p.rank;
    const uint32_t a_base = smem_u32(smem + SMEM_A_OFF);
    for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t dst = a_base + kb * A_KBLOCK_BYTES + row * 128 +
                             ((c ^ (row & 7)) << 4);
        const int col = kb * BK + c * 8;
        if (row_ok && col < p.rank)
          cp_async_16(dst, urow + col);
        else
          st_shared_zero16(dst);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
    __syncwarp();
    if (lane == 0) mbar_arrive(a_full);

    uint32_t best_key = 0u;  // below every real key
    int best_idx = 0x7FFFFFFF;
    int lit = 0;
    bool ok = true;
    for (int i = 0; i < nt && ok; ++i) {
      const int t = ascending ? t_begin + i : t_end - 1 - i;
      const int buf = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      ok = __all_sync(0xFFFFFFFFu,
                      wait_or_abort(&acc_full[buf], aph, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const int v_tile0 = t * BN;
      for (int j = 0; j < NBOX; ++j, ++lit) {
        const int s = lit % NUM_L_STAGES;
        const uint32_t lph = (lit / NUM_L_STAGES) & 1;
        ok = __all_sync(0xFFFFFFFFu,
                        wait_or_abort(&l_full[s], lph, abort_flag, p.status));
        if (!ok) break;
        const uint32_t box =
            smem_u32(smem + SMEM_L_OFF + s * L_STAGE_BYTES) + row * 128;
#pragma unroll
        for (int c = 0; c < CHUNKS_PER_BOX; ++c) {
          const int col0 = j * LBOX_COLS + c * 32;
          uint32_t acc[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(buf * BN + col0),
                             acc);
          tmem_ld_wait(acc);
          float v[32];
          if constexpr (LDT == DSPARK_BF16) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int chunk = c * 4 + u;
              const uint4 w = ld_shared_v4(box + ((chunk ^ (row & 7)) << 4));
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                v[u * 8 + 2 * h] =
                    __uint_as_float(acc[u * 8 + 2 * h]) +
                    __uint_as_float(ww[h] << 16);
                v[u * 8 + 2 * h + 1] =
                    __uint_as_float(acc[u * 8 + 2 * h + 1]) +
                    __uint_as_float(ww[h] & 0xFFFF0000u);
              }
            }
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 w = ld_shared_v4(box + ((u ^ (row & 7)) << 4));
              v[u * 4 + 0] = __uint_as_float(acc[u * 4 + 0]) + __uint_as_float(w.x);
              v[u * 4 + 1] = __uint_as_float(acc[u * 4 + 1]) + __uint_as_float(w.y);
              v[u * 4 + 2] = __uint_as_float(acc[u * 4 + 2]) + __uint_as_float(w.z);
              v[u * 4 + 3] = __uint_as_float(acc[u * 4 + 3]) + __uint_as_float(w.w);
            }
          }
          const int vbase = v_tile0 + col0;
          if (vbase + 32 > p.vocab) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (vbase + e >= p.vocab) v[e] = -INFINITY;
          }
          float mx = v[0];
#pragma unroll
          for (int e = 1; e < 32; ++e) mx = fmax_nan(mx, v[e]);
          int ie = 0;
          if (mx != mx) {
#pragma unroll
            for (int e = 31; e >= 0; --e) ie = (v[e] != v[e]) ? e : ie;
          } else {
#pragma unroll
            for (int e = 31; e >= 0; --e) ie = (v[e] == mx) ? e : ie;
          }
          const uint32_t key = f32_key(mx);
          const int idx = vbase + ie;
          if (key > best_key || (key == best_key && idx < best_idx)) {
            best_key = key;
            best_idx = idx;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&l_empty[s]);
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (ok && row_ok) {
      const unsigned long long packed =
          (static_cast<unsigned long long>(best_key) << 32) |
          static_cast<unsigned long long>(0xFFFFFFFFu -
                                          static_cast<uint32_t>(best_idx));
      atomicMax(&p.slots[m], packed);
      __threadfence();
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);

  // the last CTA of the grid decodes the winners of every request
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t ticket = atomicAdd(p.counter, 1u);
    *last_flag = (ticket == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (*last_flag) {
    __threadfence();
    for (int n = threadIdx.x; n < p.N; n += blockDim.x) {
      const unsigned long long key =
          *reinterpret_cast<volatile unsigned long long *>(&p.slots[n]);
      const uint32_t kh = static_cast<uint32_t>(key >> 32);
      int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
      if (key == 0ull || idx < 0 || idx >= p.vocab) idx = 0;
      p.draft[static_cast<size_t>(n) * p.K + p.k_pos] = idx;
      if (p.score)
        p.score[static_cast<size_t>(n) * p.K + p.k_pos] = f32_from_key(kh);
      if (kh == 0xFFFFFFFFu) raise_status(p.status, DSPARK_DEV_NAN_LOGIT);
    }
  }
}

// ==========================================================================
// host side
// ==========================================================================
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

static std::mutex g_attr_mu;
static bool g_attr_done[2][128];

static cudaError_t ensure_kernel_attrs(int dev) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!g_attr_done[0][dev]) {
    cudaError_t e = cudaFuncSetAttribute(chain_position_kernel<DSPARK_BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CHAIN_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    g_attr_done[0][dev] = true;
  }
  if (!g_attr_done[1][dev]) {
    cudaError_t e = cudaFuncSetAttribute(chain_position_kernel<DSPARK_F32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CHAIN_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    g_attr_done[1][dev] = true;
  }
  return cudaSuccess;
}

size_t chain_workspace_bytes(int32_t N, int32_t K) {
  const size_t slots = static_cast<size_t>(N) * K * sizeof(unsigned long long);
  return ((kChainSlotsOffset + slots + 255) / 256) * 256;
}

dspark_status chain_draft_launch(const ChainArgs &a, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return DSPARK_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return DSPARK_ERR_CUDA;
  const int n_mtiles = (a.N + BM - 1) / BM;
  if (n_mtiles > sms) return DSPARK_ERR_UNSUPPORTED;
  if (ensure_kernel_attrs(dev) != cudaSuccess) return DSPARK_ERR_CUDA;

  const int n_vtiles = (a.vocab + BN - 1) / BN;
  const int n_vgroups = std::max(1, std::min(sms / n_mtiles, n_vtiles));
  const int grid = n_mtiles * n_vgroups;

  // V: dim0 = rank (contiguous), dim1 = vocab; 64 x 256 boxes, 128-B swizzle
  CUtensorMap tmV, tmL;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.rank),
                          static_cast<cuuint64_t>(a.vocab)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.rank) * 2};
    cuuint32_t box[2] = {BK, BN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.V),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSPARK_ERR_INVALID_ARG;
  }
  // logits: dim0 = vocab; dims 1, 2 = (K, N) ordered by stride; boxes of
  // 128 bytes x 128 requests x 1 position
  int l_k_is_dim1 = 1;
  {
    const int esz = a.logits_dtype == DSPARK_BF16 ? 2 : 4;
    const int64_t sk = a.K > 1 ? a.stride_k : a.stride_n;
    l_k_is_dim1 = (sk <= a.stride_n) ? 1 : 0;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    dims[0] = static_cast<cuuint64_t>(a.vocab);
    box[0] = 128 / esz;
    if (l_k_is_dim1) {
      dims[1] = a.K;  strides[0] = static_cast<cuuint64_t>(sk) * esz;  box[1] = 1;
      dims[2] = a.N;  strides[1] = static_cast<cuuint64_t>(a.stride_n) * esz;  box[2] = BM;
    } else {
      dims[1] = a.N;  strides[0] = static_cast<cuuint64_t>(a.stride_n) * esz;  box[1] = BM;
      dims[2] = a.K;  strides[1] = static_cast<cuuint64_t>(sk) * esz;  box[2] = 1;
    }
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmL,
            a.logits_dtype == DSPARK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
            3, const_cast<void *>(a.logits), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSPARK_ERR_INVALID_ARG;
  }

  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + kStatusOffset);
  uint32_t *counters = reinterpret_cast<uint32_t *>(ws + kChainCounterOffset);
  unsigned long long *slots =
      reinterpret_cast<unsigned long long *>(ws + kChainSlotsOffset);
  const size_t clear_bytes = kChainSlotsOffset - kChainCounterOffset +
                             static_cast<size_t>(a.N) * a.K * 8;
  if (cudaMemsetAsync(counters, 0, clear_bytes, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;

  ChainParams p;
  p.U = static_cast<const uint16_t *>(a.U);
  p.last_token = a.last_token;
  p.draft = a.draft;
  p.score = a.score;
  p.status = status;
  p.N = a.N;
  p.K = a.K;
  p.vocab = a.vocab;
  p.rank = a.rank;
  p.n_mtiles = n_mtiles;
  p.n_vgroups = n_vgroups;
  p.n_vtiles = n_vtiles;
  p.l_k_is_dim1 = l_k_is_dim1;

  for (int k = 0; k < a.K; ++k) {
    p.k_pos = k;
    p.slots = slots + static_cast<size_t>(k) * a.N;
    p.counter = counters + k;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CHAIN_THREADS);
    cfg.dynamicSmemBytes = CHAIN_SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = k > 0 ? 1 : 0;  // position 0 waits for all prior work
    cudaError_t e;
    if (a.logits_dtype == DSPARK_BF16)
      e = cudaLaunchKernelEx(&cfg, chain_position_kernel<DSPARK_BF16>, tmV, tmL, p);
    else
      e = cudaLaunchKernelEx(&cfg, chain_position_kernel<DSPARK_F32>, tmV, tmL, p);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

}  // namespace dspark
