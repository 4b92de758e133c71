// Fused drafter output projection + Markov bias + chain on sm_103a.
//
// "DSpark on MAX", section "What DSpark is", items 2-3: the block-parallel
// drafter scores all K positions in one forward pass; chaining then adds a
// low-rank bias keyed on the previous chosen token and takes the argmax.
// Here the drafter's last step, its output projection W, is fused with the
// bias into one score per position:
//
//   adj[n, k, :] = [h[n, k, :], U[prev]] . [W, V]^T      (K-dim d + r)
//
// so neither the backbone logits nor the bias are ever written to memory.
// One persistent, cooperative launch chains all K positions, like the chain
// kernel, with both operands streamed per 64-wide K-block:
//
//   A = h[m0 : m0+128, k, kb]    128 x 64 bf16 by TMA      (kb < d / 64)
//       U[prev_m]                gathered once per position (the last r/64)
//   B = W[v0 : v0+256, kb]       256 x 64 bf16 by TMA      (kb < d / 64)
//       V[v0 : v0+256, kb']                                 (the last r/64)
//
// The h . W^T part of a position does not depend on the chain, so the MMA
// issuer runs it for the position's first tile while the epilogue warps are
// still at the grid barrier and gathering U[prev]; only the last r/64
// K-blocks wait for the gathered rows.  That hides the per-position barrier
// latency behind tensor-core work.
//
// Warp roles (256 threads, one CTA per SM, all 512 TMEM columns):
//   warp 0      TMA producer of B (W then V K-blocks per tile)
//   warp 1      TMEM allocation; one thread issues tcgen05.mma
//   warp 2      TMA producer of A's h K-blocks
//   warp 3      idle
//   warps 4-7   grid barrier, winner decode and U gather, then the argmax
//               epilogue (TMEM lane quarter w % 4)
#include <algorithm>
#include <mutex>

#include "chain_common.cuh"
#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

namespace {

constexpr int LM_MAX_KU = 4;  // rank <= 256
constexpr int LM_B_STAGES = 4;  // W streams from DRAM: the deeper ring (measured 1660 -> 1520 us vs 3 + 4)
constexpr int LM_H_STAGES = 2;  // h is re-read from L2: a shallow ring suffices
constexpr int LM_A_KBLOCK_BYTES = BM * 128;
constexpr int LM_AU_BYTES = LM_MAX_KU * LM_A_KBLOCK_BYTES;
constexpr int LM_B_STAGE_BYTES = BN * 128;
constexpr int LM_B_BOX_BYTES = BQ * 128;
constexpr int LM_H_STAGE_BYTES = BM * 128;
constexpr int LM_AU_OFF = 0;
constexpr int LM_B_OFF = LM_AU_OFF + LM_AU_BYTES;
constexpr int LM_H_OFF = LM_B_OFF + LM_B_STAGES * LM_B_STAGE_BYTES;
constexpr int LM_BAR_OFF = LM_H_OFF + LM_H_STAGES * LM_H_STAGE_BYTES;
constexpr int LM_NUM_BARS = 2 * LM_B_STAGES + 2 * LM_H_STAGES + 2 + 2 + 1 + 1;
constexpr int LM_SMEM_BYTES = LM_BAR_OFF + LM_NUM_BARS * 8 + 16 + 1024;
constexpr int LM_THREADS = 256;
constexpr uint32_t LM_TMEM_COLS = 512;
constexpr double kLmL2KeepBytes = 40.0 * 1024 * 1024;

static_assert(LM_SMEM_BYTES <= 232448, "shared memory budget");

struct LmParams {
  const uint16_t *U;
  const int32_t *last_token;
  int32_t *draft;
  float *score;
  unsigned long long *slots;
  uint32_t *counters;
  uint32_t *g_abort;
  const uint32_t *hang_test;
  uint32_t *status;
  int32_t N, K, vocab, rank, d;
  int32_t n_mtiles, n_vgroups, n_quanta;
  int32_t h_k_is_dim1;  // h map: dim1 = K, dim2 = N (else swapped)
  int32_t v_keep_tenths;
};

__global__ void __launch_bounds__(LM_THREADS, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmH, const LmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LM_BAR_OFF);
  uint64_t *b_full = bars;
  uint64_t *b_empty = b_full + LM_B_STAGES;
  uint64_t *h_full = b_empty + LM_B_STAGES;
  uint64_t *h_empty = h_full + LM_H_STAGES;
  uint64_t *acc_full = h_empty + LM_H_STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *a_full = acc_empty + 2;
  uint64_t *mma_done = a_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + LM_NUM_BARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x % p.n_mtiles;
  const int grp = blockIdx.x / p.n_mtiles;
  const int m0 = m_tile * BM;
  const int qb = static_cast<int>((static_cast<long long>(grp) * p.n_quanta) /
                                  p.n_vgroups);
  const int qe = static_cast<int>(
      (static_cast<long long>(grp + 1) * p.n_quanta) / p.n_vgroups);
  const int nt = (qe - qb + QPT - 1) / QPT;  // tiles per position
  const int KH = p.d / BK;                    // h . W^T K-blocks
  const int KU = (p.rank + BK - 1) / BK;      // U . V^T K-blocks

  if (threadIdx.x == 0) {
    for (int i = 0; i < LM_B_STAGES; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < LM_H_STAGES; ++i) {
      mbar_init(&h_full[i], 1);
      mbar_init(&h_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(a_full, 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 64) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmH);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, LM_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ B producer (W, V)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_v = policy_keep_tenths(p.v_keep_tenths);
      int last_it[LM_B_STAGES];
      for (int s = 0; s < LM_B_STAGES; ++s) last_it[s] = -1;
      int it = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        for (int i = 0; i < nt && ok; ++i) {
          const TileGeom g = tile_geom(k, i, qb, qe);
          for (int kb = 0; kb < KH + KU; ++kb, ++it) {
            const int s = it % LM_B_STAGES;
            const uint32_t ph = (it / LM_B_STAGES) & 1;
            if (!(ok = wait_bounded(&b_empty[s], ph ^ 1u, abort_flag, p.status)))
              break;
            mbar_arrive_expect_tx(&b_full[s], g.nq * LM_B_BOX_BYTES);
            for (int j = 0; j < g.nq; ++j) {
              uint8_t *dst = smem + LM_B_OFF + s * LM_B_STAGE_BYTES + j * LM_B_BOX_BYTES;
              if (kb < KH)
                tma_load_2d(dst, &tmW, &b_full[s], kb * BK, (g.qa + j) * BQ, pol_w);
              else
                tma_load_2d(dst, &tmV, &b_full[s], (kb - KH) * BK, (g.qa + j) * BQ,
                            pol_v);
            }
            last_it[s] = it;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < LM_B_STAGES; ++s)
          if (last_it[s] >= 0)
            drain_wait(&b_full[s], (last_it[s] / LM_B_STAGES) & 1, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------ A producer (h)
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // re-read by every tile
      int last_it[LM_H_STAGES];
      for (int s = 0; s < LM_H_STAGES; ++s) last_it[s] = -1;
      int it = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        const int c1 = p.h_k_is_dim1 ? k : m0;
        const int c2 = p.h_k_is_dim1 ? m0 : k;
        for (int i = 0; i < nt && ok; ++i) {
          for (int kb = 0; kb < KH; ++kb, ++it) {
            const int s = it % LM_H_STAGES;
            const uint32_t ph = (it / LM_H_STAGES) & 1;
            if (!(ok = wait_bounded(&h_empty[s], ph ^ 1u, abort_flag, p.status)))
              break;
            mbar_arrive_expect_tx(&h_full[s], LM_H_STAGE_BYTES);
            tma_load_3d(smem + LM_H_OFF + s * LM_H_STAGE_BYTES, &tmH, &h_full[s],
                        kb * BK, c1, c2, pol);
            last_it[s] = it;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < LM_H_STAGES; ++s)
          if (last_it[s] >= 0)
            drain_wait(&h_full[s], (last_it[s] / LM_H_STAGES) & 1, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t au_base = smem_u32(smem + LM_AU_OFF);
      const uint32_t b_base = smem_u32(smem + LM_B_OFF);
      const uint32_t h_base = smem_u32(smem + LM_H_OFF);
      int ib = 0, ih = 0, ig = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        for (int i = 0; i < nt && ok; ++i, ++ig) {
          const TileGeom g = tile_geom(k, i, qb, qe);
          const uint32_t idesc =
              umma_idesc_bf16_f32(BM, static_cast<uint32_t>(g.nq * BQ));
          const int buf = ig & 1;
          const uint32_t aph = (ig >> 1) & 1;
          if (!(ok = wait_bounded(&acc_empty[buf], aph ^ 1u, abort_flag, p.status)))
            break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
          // h . W^T: independent of the chain
          for (int kb = 0; kb < KH && ok; ++kb, ++ib, ++ih) {
            const int sb = ib % LM_B_STAGES, sh = ih % LM_H_STAGES;
            ok = wait_bounded(&h_full[sh], (ih / LM_H_STAGES) & 1, abort_flag, p.status) &&
                 wait_bounded(&b_full[sb], (ib / LM_B_STAGES) & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad =
                  sw128_kmajor_desc(h_base + sh * LM_H_STAGE_BYTES + kk * 32);
              const uint64_t bd =
                  sw128_kmajor_desc(b_base + sb * LM_B_STAGE_BYTES + kk * 32);
              umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&h_empty[sh]);
            umma_commit(&b_empty[sb]);
          }
          if (!ok) break;
          // U[prev] . V^T: the position's gathered rows
          if (i == 0) {
            if (!(ok = wait_bounded(a_full, k & 1, abort_flag, p.status))) break;
            tc_fence_after();
          }
          for (int ku = 0; ku < KU && ok; ++ku, ++ib) {
            const int sb = ib % LM_B_STAGES;
            if (!(ok = wait_bounded(&b_full[sb], (ib / LM_B_STAGES) & 1, abort_flag,
                                    p.status)))
              break;
            tc_fence_after();
            const int nk = min(BK, p.rank - ku * BK) / 16;
            for (int kk = 0; kk < nk; ++kk) {
              const uint64_t ad =
                  sw128_kmajor_desc(au_base + ku * LM_A_KBLOCK_BYTES + kk * 32);
              const uint64_t bd =
                  sw128_kmajor_desc(b_base + sb * LM_B_STAGE_BYTES + kk * 32);
              umma_bf16(d_tmem, ad, bd, idesc, 1u);
            }
            umma_commit(&b_empty[sb]);
          }
          if (!ok) break;
          umma_commit(&acc_full[buf]);
        }
      }
      umma_commit(mma_done);
      drain_wait(mma_done, 0, p.status);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ----------------------------- grid barrier, gather, epilogue per k
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int m = m0 + row;
    const bool row_ok = m < p.N;
    const bool writer = (grp == 0) && row_ok;
    const uint32_t au_base = smem_u32(smem + LM_AU_OFF);
    int ig = 0;
    bool ok = true;
    for (int k = 0; k < p.K && ok; ++k) {
      int prev = 0;
      if (k == 0) {
        if (row_ok) {
          prev = p.last_token[m];
          if (prev < 0 || prev >= p.vocab) {
            prev = 0;
            raise_status(p.status, DSPARK_DEV_TOKEN_OOR);
          }
        }
      } else {
        if (!(ok = grid_wait(p, k - 1, m_tile, abort_flag, 4u))) break;
        if (row_ok) {
          const unsigned long long key = *reinterpret_cast<volatile unsigned long long *>(
              &p.slots[static_cast<size_t>(k - 1) * p.N + m]);
          prev = decode_index(key, p.vocab);
          if (writer) {
            const uint32_t kh = static_cast<uint32_t>(key >> 32);
            p.draft[static_cast<size_t>(m) * p.K + (k - 1)] = prev;
            if (p.score)
              p.score[static_cast<size_t>(m) * p.K + (k - 1)] = f32_from_key(kh);
            if (kh == 0xFFFFFFFFu) raise_status(p.status, DSPARK_DEV_NAN_LOGIT);
          }
        }
      }
      // gather U[prev] into the resident A K-blocks, one 512-byte row per
      // warp instruction; the U . V^T MMAs of position k-1 have retired
      // (their last accumulator was consumed)
      const int nchunk = KU * 8;
      for (int r = 0; r < 32; ++r) {
        const int rp = __shfl_sync(0xFFFFFFFFu, prev, r);
        const int rrow = q * 32 + r;
        const bool rok = (m0 + rrow) < p.N;
        if (lane < nchunk) {
          const int kb = lane >> 3, c = lane & 7;
          const uint32_t dst = au_base + kb * LM_A_KBLOCK_BYTES + rrow * 128 +
                               ((c ^ (rrow & 7)) << 4);
          if (rok && lane * 8 < p.rank)
            cp_async_16(dst, p.U + static_cast<size_t>(rp) * p.rank + lane * 8);
          else
            st_shared_zero16(dst);
        }
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full);

      uint32_t best_key = 0u;
      int best_idx = 0x7FFFFFFF;
      for (int i = 0; i < nt && ok; ++i, ++ig) {
        const TileGeom g = tile_geom(k, i, qb, qe);
        const int buf = ig & 1;
        const uint32_t aph = (ig >> 1) & 1;
        ok = __all_sync(0xFFFFFFFFu,
                        wait_bounded(&acc_full[buf], aph, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        for (int col0 = 0; col0 < g.nq * BQ; col0 += 32) {
          uint32_t acc[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(buf * BN + col0),
                             acc);
          tmem_ld_wait(acc);
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(acc[e]);
          const int vbase = g.qa * BQ + col0;
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      if (!ok) break;
      if (row_ok) {
        const unsigned long long packed =
            (static_cast<unsigned long long>(best_key) << 32) |
            static_cast<unsigned long long>(0xFFFFFFFFu -
                                            static_cast<uint32_t>(best_idx));
        atomicMax(&p.slots[static_cast<size_t>(k) * p.N + m], packed);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(&p.counters[k * p.n_mtiles + m_tile], 1u);
    }
    if (ok) {
      ok = grid_wait(p, p.K - 1, m_tile, abort_flag, 4u);
      if (ok && writer) {
        const unsigned long long key = *reinterpret_cast<volatile unsigned long long *>(
            &p.slots[static_cast<size_t>(p.K - 1) * p.N + m]);
        const uint32_t kh = static_cast<uint32_t>(key >> 32);
        p.draft[static_cast<size_t>(m) * p.K + (p.K - 1)] = decode_index(key, p.vocab);
        if (p.score)
          p.score[static_cast<size_t>(m) * p.K + (p.K - 1)] = f32_from_key(kh);
        if (kh == 0xFFFFFFFFu) raise_status(p.status, DSPARK_DEV_NAN_LOGIT);
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1u;
      atomicExch(p.g_abort, 1u);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, LM_TMEM_COLS);
}

std::mutex g_lm_mu;
bool g_lm_attr[128];

}  // namespace

dspark_status lmhead_chain_launch(const LmheadArgs &a, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return DSPARK_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return DSPARK_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return DSPARK_ERR_CUDA;
  const int n_mtiles = (a.N + BM - 1) / BM;
  if (n_mtiles > sms) return DSPARK_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_lm_mu);
    if (!g_lm_attr[dev]) {
      if (cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LM_SMEM_BYTES) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      g_lm_attr[dev] = true;
    }
  }
  const int n_quanta = (a.vocab + BQ - 1) / BQ;
  int groups = sms / n_mtiles;
  if (n_mtiles * groups > sms - 1 && groups > 1) groups = (sms - 1) / n_mtiles;
  const int n_vgroups = std::max(1, std::min(groups, n_quanta));
  const int grid = n_mtiles * n_vgroups;

  CUtensorMap tmW, tmV, tmH;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.d), static_cast<cuuint64_t>(a.vocab)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.d) * 2};
    cuuint32_t box[2] = {BK, BQ};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.W), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSPARK_ERR_INVALID_ARG;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.rank), static_cast<cuuint64_t>(a.vocab)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.rank) * 2};
    cuuint32_t box[2] = {BK, BQ};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.V), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSPARK_ERR_INVALID_ARG;
  }
  int h_k_is_dim1 = 1;
  {
    const int64_t sk = a.K > 1 ? a.stride_k : a.stride_n;
    h_k_is_dim1 = (sk <= a.stride_n) ? 1 : 0;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    dims[0] = static_cast<cuuint64_t>(a.d);
    box[0] = BK;
    if (h_k_is_dim1) {
      dims[1] = a.K;  strides[0] = static_cast<cuuint64_t>(sk) * 2;  box[1] = 1;
      dims[2] = a.N;  strides[1] = static_cast<cuuint64_t>(a.stride_n) * 2;  box[2] = BM;
    } else {
      dims[1] = a.N;  strides[0] = static_cast<cuuint64_t>(a.stride_n) * 2;  box[1] = BM;
      dims[2] = a.K;  strides[1] = static_cast<cuuint64_t>(sk) * 2;  box[2] = 1;
    }
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmH, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.h), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSPARK_ERR_INVALID_ARG;
  }

  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  const size_t clear_bytes = chain_counters_offset(a.N, a.K) +
                             static_cast<size_t>(n_mtiles) * a.K * 4 -
                             kChainAbortOffset;
  if (cudaMemsetAsync(ws + kChainAbortOffset, 0, clear_bytes, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;

  LmParams p;
  p.U = static_cast<const uint16_t *>(a.U);
  p.last_token = a.last_token;
  p.draft = a.draft;
  p.score = a.score;
  p.slots = reinterpret_cast<unsigned long long *>(ws + kChainSlotsOffset);
  p.counters = reinterpret_cast<uint32_t *>(ws + chain_counters_offset(a.N, a.K));
  p.g_abort = reinterpret_cast<uint32_t *>(ws + kChainAbortOffset);
  p.hang_test = reinterpret_cast<const uint32_t *>(ws + kChainHangTestOffset);
  p.status = reinterpret_cast<uint32_t *>(ws + kStatusOffset);
  p.N = a.N;
  p.K = a.K;
  p.vocab = a.vocab;
  p.rank = a.rank;
  p.d = a.d;
  p.n_mtiles = n_mtiles;
  p.n_vgroups = n_vgroups;
  p.n_quanta = n_quanta;
  p.h_k_is_dim1 = h_k_is_dim1;
  {
    const double v_bytes = static_cast<double>(a.vocab) * a.rank * 2;
    const int tenths = static_cast<int>(10.0 * kLmL2KeepBytes / v_bytes);
    p.v_keep_tenths = std::max(0, std::min(10, tenths));
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(LM_THREADS);
  cfg.dynamicSmemBytes = LM_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lmhead_kernel, tmW, tmV, tmH, p);
  if (e == cudaErrorCooperativeLaunchTooLarge) return DSPARK_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace dspark
