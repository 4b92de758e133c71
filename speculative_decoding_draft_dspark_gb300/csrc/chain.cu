// Chaining stage of the DSpark draft step on sm_103a.
//
// "DSpark on MAX", section "What DSpark is", item 3: turning the parallel
// drafter's scores into a K-token chain is a low-rank bias keyed on the
// previous chosen token followed by an argmax.  "How DSpark Speeds Up LLM
// Inference", section "Draft better": the Markov head is a rank-256
// factorisation that adjusts each word's odds using only the word before it.
//
// One persistent, cooperative launch chains all K positions.  For draft
// position k, the 128-request tile m and the vocabulary tiles a CTA owns:
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
// smaller index; NaN maps to the largest key.  Position k+1 needs every
// row's winner of position k, so the epilogue warps meet at a grid barrier
// (a counter per position, polled with a time limit; the cooperative launch
// keeps all CTAs resident) and then each warp decodes the winners of its own
// 32 rows and gathers their U rows.  The TMA producers do not depend on the winners and
// keep streaming V and logits across position boundaries.
//
// Probabilistic drafting ("Adaptive Verification in vLLM", section "Appendix:
// reproducing", draft_sample_method "probabilistic") is the same kernel with
// SAMPLE set: each token is a draw from the softmax of adj / tau, taken as a
// Gumbel-max over blocks of 16 vocabulary entries (keyed on each block's log
// partition function, noise from Philox4x32-10) and then the entry inside
// the winning block; the running (key, index) maximum is combined as above.
//
// Warp roles (one CTA per SM, all 512 TMEM columns):
//   warp 0      TMA producer of V tiles (4 K-blocks of 64 per tile)
//   warp 1      TMEM allocation; one thread issues tcgen05.mma
//   warp 2      TMA producer of logits boxes
//   warp 3      idle
//   warps 4-7   grid barrier, winner decode and U gather, then the epilogue
//               (TMEM lane quarter w % 4)
//   warps 8-11  more epilogue warps on the same lane quarters (warp w takes
//               quarter w % 4; the warps of a quarter split each tile's
//               32-column chunks; they also decode the winners and, with a
//               single tile per position, gather half of each U row);
//               sampling runs warps 8-19 with full request tiles, and only
//               warps 4-11 when the tile holds its requests several times
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "chain_common.cuh"
#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int MAX_KB = 4;
constexpr int NUM_B_STAGES = 3;
constexpr int NUM_L_STAGES = 4;
constexpr int A_KBLOCK_BYTES = BM * 128;
constexpr int A_BYTES = MAX_KB * A_KBLOCK_BYTES;
constexpr int B_STAGE_BYTES = BN * 128;
constexpr int B_BOX_BYTES = BQ * 128;  // one quantum of one K-block
constexpr int L_STAGE_BYTES = BM * 128;
constexpr int SMEM_A_OFF = 0;
constexpr int SMEM_B_OFF = SMEM_A_OFF + A_BYTES;
constexpr int SMEM_L_OFF = SMEM_B_OFF + NUM_B_STAGES * B_STAGE_BYTES;
constexpr int SMEM_BAR_OFF = SMEM_L_OFF + NUM_L_STAGES * L_STAGE_BYTES;
constexpr int NUM_BARS = 20;
constexpr int SMEM_USED = SMEM_BAR_OFF + NUM_BARS * 8 + 16;
constexpr int CHAIN_SMEM_BYTES = SMEM_USED + 1024;  // 1 KB alignment slack
// warps 0-3 have fixed roles; EPI epilogue warps follow: 8 for the argmax
// chain (4 / 8 / 12 measured at the headline: chain 311 / 295 / 301 us;
// Stress 2410 / 2176 / 2157 us); for sampling, whose epilogue does more
// arithmetic per element, 16 with full request tiles and 8 when requests
// are held several times (8 / 12 / 16 / 20 warps: headline 499 / 433 / 421
// / 440 us, Conc-64 234 / 245 / 263 / 286 us, Gemma4-12B 191 / 203 / 212 /
// 233 us)
constexpr int chain_threads(int epi) { return (4 + epi) * 32; }
constexpr int EPI_ARGMAX = 8;
constexpr int EPI_SAMPLE = 16;      // sampling, full request tiles
constexpr int EPI_SAMPLE_REP = 8;   // sampling, requests held 2 or 4 times
constexpr int SAMPLE_BLOCK = 16;  // vocabulary entries per block of the sampling draw
constexpr uint32_t TMEM_COLS = 512;  // two 256-column fp32 accumulators
// bytes of V worth protecting in L2 across positions (measured on GB300:
// with a 128 MiB V, protecting 6 tenths is fastest for batches of 8 to 256
// requests and neutral at 1024; 8 tenths or more and the logits stream
// evicts it anyway; a V that fits in L2, 63 MiB, is best protected whole)
constexpr double kL2KeepBytes = 80.0 * 1024 * 1024;

static_assert(CHAIN_SMEM_BYTES <= 232448, "shared memory budget");

struct ChainParams {
  const uint16_t *U;
  const int32_t *last_token;
  int32_t *draft;
  float *score;
  unsigned long long *slots;  // [K][N] per-row winners
  uint32_t *counters;         // [K][n_mtiles] epilogue warps done
  uint32_t *g_abort;          // set by any CTA that gives up
  const uint32_t *hang_test;  // nonzero: barriers wait for one arrival too many
  uint32_t *status;
  int32_t N, K, vocab, rank;
  int32_t n_mtiles, n_vgroups, n_quanta;
  int32_t l_k_is_dim1;  // logits map: dim1 = K, dim2 = N (else swapped)
  int32_t v_keep_tenths;
  uint32_t seed_lo, seed_hi, offset;  // sampling: Philox key, counter word 3
  float inv_tau;                       // sampling: 1 / temperature
};

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): 10 rounds of two 32 x 32 -> 64-bit products of
// counter words 0 and 2 with the round multipliers, the high halves mixed
// into the other words with the key, the key bumped by the Weyl constants.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// The round keys depend only on the seed: a thread computes them once.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys r;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    r.k0[i] = k0 + static_cast<uint32_t>(i) * kPhiloxW0;
    r.k1[i] = k1 + static_cast<uint32_t>(i) * kPhiloxW1;
  }
  return r;
}

// In a position's draws only counter word 0 varies (the vocabulary block);
// words 1-3 are the request, the position and the offset.  So the product of
// round 1 that involves word 2, and the product of round 2 that involves the
// round-1 output word 0, are the same for every draw of a (request,
// position): computed once per position, they leave 18 of the 20 products
// per block.  The words are those of the plain rounds, bit for bit.
struct PhiloxRow {
  uint32_t c0k;  // offset ^ round-1 key 1 (mixed into round-1 word 2)
  uint32_t c1k;  // low(M1 * position) ^ round-2 key 0
  uint32_t c2k;  // high(M0 * a0) ^ round-2 key 1, a0 = round-1 word 0
  uint32_t d;    // low(M0 * a0): round-2 word 3
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t n, uint32_t k, uint32_t offset,
                                                const PhiloxKeys &key) {
  const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * k;
  const uint32_t a0 = static_cast<uint32_t>(p1 >> 32) ^ n ^ key.k0[0];
  const uint64_t q = static_cast<uint64_t>(kPhiloxM0) * a0;
  PhiloxRow r;
  r.c0k = offset ^ key.k1[0];
  r.c1k = static_cast<uint32_t>(p1) ^ key.k0[1];
  r.c2k = static_cast<uint32_t>(q >> 32) ^ key.k1[1];
  r.d = static_cast<uint32_t>(q);
  return r;
}

// The four words of block (ctr, n, k, offset) given that row's constants.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t ctr,
                                              const PhiloxRow &w, const PhiloxKeys &key) {
  const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * ctr;     // round 1
  const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ w.c0k;
  const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * n2;      // round 2
  c[0] = static_cast<uint32_t>(p1 >> 32) ^ w.c1k;
  c[1] = static_cast<uint32_t>(p1);
  c[2] = static_cast<uint32_t>(p0) ^ w.c2k;
  c[3] = w.d;
#pragma unroll
  for (int r = 2; r < 10; ++r) {
    const uint64_t q0 = static_cast<uint64_t>(kPhiloxM0) * c[0];
    const uint64_t q1 = static_cast<uint64_t>(kPhiloxM1) * c[2];
    const uint32_t n0 = static_cast<uint32_t>(q1 >> 32) ^ c[1] ^ key.k0[r];
    const uint32_t m2 = static_cast<uint32_t>(q0 >> 32) ^ c[3] ^ key.k1[r];
    c[0] = n0;
    c[1] = static_cast<uint32_t>(q1);
    c[2] = m2;
    c[3] = static_cast<uint32_t>(q0);
  }
}

// 2^x by the hardware approximation (the skip test's bound carries margin
// for its error)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) by the hardware approximation (absolute error near 1e-7 for the
// block sums in [1, 16] it takes)
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// hi32(a * b) + c in one instruction on the FMA pipe
__device__ __forceinline__ uint32_t mad_hi_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Gumbel noise from one 32-bit word: u = (2 (x >> 9) + 1) 2^-24 (exact: the
// mantissa trick gives 1 + (x >> 9) 2^-23, and subtracting 1 - 2^-24 is exact
// by Sterbenz's lemma), g = -ln(-ln u).  The inner ln is the accurate logf,
// which keeps its relative accuracy for u next to 1 (the large g); its
// result lies in [6e-8, 16.7], where the hardware log2 (absolute error near
// 1e-6 in g) is accurate enough for the outer one.
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
  const float u = __uint_as_float(0x3F800000u | (x >> 9)) - 0x1.fffffep-1f;
  return -__logf(-logf(u));
}

// ONE_TILE: every CTA owns at most one tile per position (a small
// vocabulary); the position boundary is then all there is, and A is gathered
// by two sub-groups each loading half of every row (see the gather below)
template <int LDT, bool SAMPLE, int EPI, bool ONE_TILE, int REP>
__global__ void __launch_bounds__(chain_threads(EPI), 1)
    chain_kernel(const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmL,
                 const ChainParams p) {
  constexpr int LBOX_COLS = (LDT == DSPARK_BF16) ? 64 : 32;  // 128-byte rows
  constexpr int BPQ = BQ / LBOX_COLS;                        // boxes per quantum
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
  const int KB = (p.rank + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NUM_B_STAGES; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < NUM_L_STAGES; ++i) {
      mbar_init(&l_full[i], 1);
      mbar_init(&l_empty[i], EPI);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], EPI);
    }
    // the warps that gather A arrive: sub-group 0, and sub-group 1 too with
    // a single tile per position
    mbar_init(a_full, ONE_TILE ? 8 : 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0u;
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
      const uint64_t pol = policy_keep_tenths(p.v_keep_tenths);
      int last_it[NUM_B_STAGES];
      for (int s = 0; s < NUM_B_STAGES; ++s) last_it[s] = -1;
      int it = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        for (int i = 0; i < nt && ok; ++i) {
          const TileGeom g = tile_geom(k, i, qb, qe);
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const int s = it % NUM_B_STAGES;
            const uint32_t ph = (it / NUM_B_STAGES) & 1;
            if (!(ok = wait_bounded(&b_empty[s], ph ^ 1u, abort_flag, p.status)))
              break;
            mbar_arrive_expect_tx(&b_full[s], g.nq * B_BOX_BYTES);
            for (int j = 0; j < g.nq; ++j)
              tma_load_2d(smem + SMEM_B_OFF + s * B_STAGE_BYTES + j * B_BOX_BYTES,
                          &tmV, &b_full[s], kb * BK, (g.qa + j) * BQ, pol);
            last_it[s] = it;
          }
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
      int it = 0, ig = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        // A holds this position's gathered U rows
        if (!(ok = wait_bounded(a_full, k & 1, abort_flag, p.status))) break;
        tc_fence_after();
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
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const int s = it % NUM_B_STAGES;
            const uint32_t ph = (it / NUM_B_STAGES) & 1;
            if (!(ok = wait_bounded(&b_full[s], ph, abort_flag, p.status))) break;
            tc_fence_after();
            const int nk = min(BK, p.rank - kb * BK) / 16;
            for (int kk = 0; kk < nk; ++kk) {
              const uint64_t ad =
                  sw128_kmajor_desc(a_base + kb * A_KBLOCK_BYTES + kk * 32);
              const uint64_t bd =
                  sw128_kmajor_desc(b_base + s * B_STAGE_BYTES + kk * 32);
              umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&b_empty[s]);  // stage free once these MMAs retire
          }
          if (!ok) break;
          umma_commit(&acc_full[buf]);  // accumulator ready for the epilogue
        }
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
      int it = 0;
      bool ok = true;
      for (int k = 0; k < p.K && ok; ++k) {
        for (int i = 0; i < nt && ok; ++i) {
          const TileGeom g = tile_geom(k, i, qb, qe);
          const int c1 = p.l_k_is_dim1 ? k : m0;
          const int c2 = p.l_k_is_dim1 ? m0 : k;
          for (int j = 0; j < g.nq * BPQ; ++j, ++it) {
            const int s = it % NUM_L_STAGES;
            const uint32_t ph = (it / NUM_L_STAGES) & 1;
            if (!(ok = wait_bounded(&l_empty[s], ph ^ 1u, abort_flag, p.status)))
              break;
            mbar_arrive_expect_tx(&l_full[s], L_STAGE_BYTES);
            tma_load_3d(smem + SMEM_L_OFF + s * L_STAGE_BYTES, &tmL, &l_full[s],
                        g.qa * BQ + j * LBOX_COLS, c1, c2, pol);
            last_it[s] = it;
          }
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
    // ----------------------------- grid barrier, gather, epilogue per k
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // sub-group: with more than four epilogue warps, warps sharing a lane
    // quarter split each tile's 32-column chunks; sub-group 0 alone waits at
    // the grid barrier, decodes the winners and gathers U
    const int sg = (warp - 4) >> 2;
    constexpr int NSG = EPI / 4;
    const int row = q * 32 + lane;
    // REP > 1 (sampling a batch of at most 64 or 32 requests): the A rows
    // hold every request REP times and the copies split the vocabulary
    // chunks, so that the lane quarters that would hold padding rows share
    // the epilogue's arithmetic.  Copies of a request merge through its
    // winner slot like the CTAs do.
    constexpr int RROWS = BM / REP;     // requests per copy
    const int lrow = REP > 1 ? row % RROWS : row;  // this row's request in the tile
    const int cp = REP > 1 ? row / RROWS : 0;       // which copy of it
    const int m = m0 + lrow;
    const bool row_ok = m < p.N;
    // one CTA per tile (and one copy) writes the draft
    const bool writer = (grp == 0) && row_ok && sg == 0 && cp == 0;
    [[maybe_unused]] const PhiloxKeys pkeys = philox_keys(p.seed_lo, p.seed_hi);
    const uint32_t a_base = smem_u32(smem + SMEM_A_OFF);
    int ig = 0, lit = 0;
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
      } else if (sg == 0 || (ONE_TILE && sg == 1)) {
        // (sub-group 1 needs the winners only when it gathers: one tile per
        // position)
        if (!(ok = grid_wait(p, k - 1, m_tile, abort_flag, EPI))) break;
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
      // gather this position's U rows into A (the MMAs of position k-1 have
      // all retired: their last accumulator was consumed).  Two forms, the
      // same bytes:
      //  - with several tiles per position (the streaming case), one
      //    512-byte row per warp instruction (lane j copies 16-byte chunk j
      //    of the row) by sub-group 0: few, whole-row L2 requests, which
      //    stay fast while the rings stream;
      //  - with a single tile per position (ONE_TILE, a small vocabulary: the
      //    position boundary is all there is), every thread of sub-groups 0 and 1
      //    loads half of its own row, all loads in flight at once, and
      //    stores it itself: lower latency when nothing else is in flight.
      if constexpr (!ONE_TILE) {
        const int nchunk = sg == 0 ? KB * 8 : 0;
        for (int r = 0; r < 32 && sg == 0; ++r) {
          const int rp = __shfl_sync(0xFFFFFFFFu, prev, r);
          const int rrow = q * 32 + r;
          const bool rok = (m0 + (REP > 1 ? rrow % RROWS : rrow)) < p.N;
          if (lane < nchunk) {
            const int kb = lane >> 3, c = lane & 7;
            const uint32_t dst = a_base + kb * A_KBLOCK_BYTES + rrow * 128 +
                                 ((c ^ (rrow & 7)) << 4);
            if (rok && lane * 8 < p.rank)
              cp_async_16(dst, p.U + static_cast<size_t>(rp) * p.rank + lane * 8);
            else
              st_shared_zero16(dst);
          }
        }
        if (sg == 0) {
          cp_async_commit();
          cp_async_wait_all();
        }
      } else if (sg < 2) {
        const int kh = sg * 128;  // this thread's half of the row
        uint4 w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          w[c] = make_uint4(0u, 0u, 0u, 0u);
          if (row_ok && kh + c * 8 < p.rank)
            w[c] = ld_global_nc_v4(p.U + static_cast<size_t>(prev) * p.rank + kh + c * 8);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = kh + c * 8;
          const int kb = e >> 6, cc = (e & 63) >> 3;
          st_shared_v4(a_base + kb * A_KBLOCK_BYTES + row * 128 + ((cc ^ (row & 7)) << 4),
                       w[c]);
        }
      }
      if (sg == 0 || (ONE_TILE && sg == 1)) {
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full);
      }

      uint32_t best_key = 0u;  // below every real key
      int best_idx = 0x7FFFFFFF;
      float best_val = -INFINITY;  // the value behind best_key (sampling)
      // sampling: the row's best published so far by any thread of any CTA,
      // a shared threshold for the skip test
      uint32_t shared_key = 0u;
      unsigned long long *row_slot =
          row_ok ? &p.slots[static_cast<size_t>(k) * p.N + m] : nullptr;
      [[maybe_unused]] const PhiloxRow prow =
          philox_row(static_cast<uint32_t>(m), static_cast<uint32_t>(k), p.offset, pkeys);
      for (int i = 0; i < nt && ok; ++i, ++ig) {
        const TileGeom g = tile_geom(k, i, qb, qe);
        const int buf = ig & 1;
        const uint32_t aph = (ig >> 1) & 1;
        ok = __all_sync(0xFFFFFFFFu,
                        wait_bounded(&acc_full[buf], aph, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const int v_tile0 = g.qa * BQ;
        for (int j = 0; j < g.nq * BPQ; ++j, ++lit) {
          const int s = lit % NUM_L_STAGES;
          const uint32_t lph = (lit / NUM_L_STAGES) & 1;
          ok = __all_sync(0xFFFFFFFFu,
                          wait_bounded(&l_full[s], lph, abort_flag, p.status));
          if (!ok) break;
          const uint32_t box =
              smem_u32(smem + SMEM_L_OFF + s * L_STAGE_BYTES) + lrow * 128;
#pragma unroll
          for (int c = 0; c < CHUNKS_PER_BOX; ++c) {
            // sampling: chunks go to the sub-groups (and copies) by their
            // running index, so that every warp gets the same share whatever
            // a tile's width; the argmax chain splits each tile's chunks
            // (NSG = 2 divides a tile's chunk count)
            if constexpr (SAMPLE) {
              if ((NSG > 1 || REP > 1) &&
                  static_cast<unsigned>(lit * CHUNKS_PER_BOX + c) % (NSG * REP) !=
                      static_cast<unsigned>(sg * REP + cp))
                continue;
            } else {
              if (NSG > 1 && (j * CHUNKS_PER_BOX + c) % NSG != sg) continue;
            }
            const int col0 = j * LBOX_COLS + c * 32;
            if constexpr (SAMPLE) {
              // Two-level Gumbel-max draw over blocks of 16 vocabulary
              // entries (a piece is one block, j = v / 16): the block by the
              // Gumbel-max rule on key_j = L_j + g_j, L_j = log sum exp(adj /
              // tau) over the block, then the entry inside the winning block
              // by inverting its cumulative weights with a second uniform.
              // Block j takes words 2 (j % 2) and 2 (j % 2) + 1 of the Philox
              // block with counter (j / 2, n, k, offset): one Philox block
              // per 32-column chunk.  A block can beat the running best only
              // if g_j > best - margin - L_j, i.e. 1 - u < 1 - exp(-A) <= A
              // with A = exp(L_j - best + margin), computed for every block
              // from its weights relative to the best (16 ex2, no
              // logarithm).  It is skipped only when u <= 1 - A provably
              // holds (u exact from the word's mantissa, the bound on it
              // rounded down), the (1 + 2^-10) factor and the margin covering
              // every rounding and approximation error in A.  Blocks that
              // pass get their exact key, and their entry when the key beats
              // the running best.
              static_assert(SAMPLE_BLOCK == 16, "one 16-column tensor-memory load per block");
              const float s1 = p.inv_tau * 1.4426950408889634f;
              const int vc = v_tile0 + col0;  // a multiple of 32
              // the row's shared best, read once per chunk: the Philox rounds
              // cover its latency
              const unsigned long long shared_now =
                  row_slot ? *reinterpret_cast<volatile unsigned long long *>(row_slot) : 0ull;
              uint32_t wd[4];
              philox4x32_10(wd, static_cast<uint32_t>(vc >> 5), prow, pkeys);
#pragma unroll 1
              for (int h = 0; h < 2; ++h) {
                const int cb = col0 + h * SAMPLE_BLOCK;
                uint32_t acc[SAMPLE_BLOCK];
                tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + cb),
                                   acc);
                tmem_ld_wait(acc);
                float v[SAMPLE_BLOCK];
                if constexpr (LDT == DSPARK_BF16) {
#pragma unroll
                  for (int g8 = 0; g8 < 2; ++g8) {
                    const int chunk = c * 4 + h * 2 + g8;
                    const uint4 w = ld_shared_v4(box + ((chunk ^ (lrow & 7)) << 4));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                      v[8 * g8 + 2 * t] =
                          __uint_as_float(acc[8 * g8 + 2 * t]) + __uint_as_float(ww[t] << 16);
                      v[8 * g8 + 2 * t + 1] = __uint_as_float(acc[8 * g8 + 2 * t + 1]) +
                                              __uint_as_float(ww[t] & 0xFFFF0000u);
                    }
                  }
                } else {
#pragma unroll
                  for (int t = 0; t < 4; ++t) {
                    const int chunk = 4 * h + t;
                    const uint4 w = ld_shared_v4(box + ((chunk ^ (lrow & 7)) << 4));
                    v[4 * t + 0] = __uint_as_float(acc[4 * t + 0]) + __uint_as_float(w.x);
                    v[4 * t + 1] = __uint_as_float(acc[4 * t + 1]) + __uint_as_float(w.y);
                    v[4 * t + 2] = __uint_as_float(acc[4 * t + 2]) + __uint_as_float(w.z);
                    v[4 * t + 3] = __uint_as_float(acc[4 * t + 3]) + __uint_as_float(w.w);
                  }
                }
                const int vb = v_tile0 + cb;
                if (vb + SAMPLE_BLOCK > p.vocab) {
#pragma unroll
                  for (int e = 0; e < SAMPLE_BLOCK; ++e)
                    if (vb + e >= p.vocab) v[e] = -INFINITY;
                }
                const uint32_t xg = h ? wd[2] : wd[0];  // the block's Gumbel word
                const uint32_t xc = h ? wd[3] : wd[1];  // the word of its entry
                // The skip test's threshold: this thread's best or the row's
                // best published by any thread, whichever is larger.  Every
                // published key is some block's exact key, so a block skipped
                // against it (with the margin below) can neither win nor tie.
                shared_key = max(shared_key, static_cast<uint32_t>(shared_now >> 32));
                const uint32_t tkey = max(best_key, shared_key);
                const float tval = tkey == best_key ? best_val : f32_from_key(tkey);
                const bool none = tkey == 0u || tval != tval;  // nothing to beat yet
                const float margin = 1e-4f * (1.0f + fabsf(tval));
                // The block's weight relative to the threshold, rel = sum of
                // exp(adj / tau - best), so that exp(L_j - best) = rel: every
                // block's exact key is one Gumbel away and the test below is
                // tight, with no max shift and no logarithm.  An entry 126
                // octaves below the threshold flushes to zero (its block
                // could not win by any Gumbel value); one that would overflow
                // makes the block a candidate, whose exact key is computed
                // with the max shift.
                const float c2 = none ? 0.0f : tval * 1.4426950408889634f;
                float rel = 0.0f;
#pragma unroll
                for (int e = 0; e < SAMPLE_BLOCK; ++e) rel += ex2_approx(fmaf(v[e], s1, -c2));
                // candidate unless 1 - u >= A = exp(L_j - best + margin) =
                // rel e^margin (times 2^(2^-10) for the approximations): u =
                // u1 - (1 - 2^-24) with u1 = 1 + (xg >> 9) 2^-23 (one mad.hi),
                // and u1 <= RD((2 - 2^-23) - A) implies u < 1 - A (NaN A:
                // always a candidate)
                const float A =
                    none ? INFINITY
                         : rel * ex2_approx(fmaf(margin, 1.4426950408889634f, 0x1p-10f));
                const float u1 = __uint_as_float(mad_hi_u32(xg, 1u << 23, 0x3F800000u));
                const bool cand = !(u1 <= __fsub_rd(0x1.fffffep0f, A));
                if (__any_sync(0xFFFFFFFFu, cand) && cand) {
                  // the block's exact key, max-shifted: NaN if it holds a NaN
                  // (the first NaN is then its entry), +inf if it holds +inf
                  // (the first one is its entry), -inf if nothing is finite
                  float mx = v[0];
#pragma unroll
                  for (int e = 1; e < SAMPLE_BLOCK; ++e) mx = fmax_nan(mx, v[e]);
                  float key, sum = 0.0f;
                  float ex[SAMPLE_BLOCK];
                  int e_star = 0;
                  const bool finite = mx == mx && fabsf(mx) != INFINITY;
                  if (!finite) {
                    key = mx;
#pragma unroll
                    for (int e = SAMPLE_BLOCK - 1; e >= 0; --e)
                      e_star = (v[e] != v[e] || v[e] == mx) ? e : e_star;
                    if (mx == -INFINITY) e_star = 0;
                  } else {
#pragma unroll
                    for (int e = 0; e < SAMPLE_BLOCK; ++e) {
                      ex[e] = ex2_approx((v[e] - mx) * s1);
                      sum += ex[e];
                    }
                    key = fmaf(mx, p.inv_tau, lg2_approx(sum) * 0.6931471805599453f) +
                          gumbel_from_word(xg);
                  }
                  const uint32_t kk = f32_key(key);
                  if (kk >= best_key) {
                    if (finite) {
                      // the first entry whose cumulative weight exceeds u * sum
                      const float uc = __uint_as_float(0x3F800000u | (xc >> 9)) - 0x1.fffffep-1f;
                      const float target = uc * sum;
                      float cum = 0.0f;
                      int hit = -1, last = 0;
#pragma unroll
                      for (int e = 0; e < SAMPLE_BLOCK; ++e) {
                        cum += ex[e];
                        hit = (hit < 0 && cum > target) ? e : hit;
                        last = ex[e] > 0.0f ? e : last;
                      }
                      e_star = hit >= 0 ? hit : last;
                    }
                    const int idx = vb + e_star;
                    if (kk > best_key || idx < best_idx) {
                      best_key = kk;
                      best_idx = idx;
                      best_val = key;
                      // published at once so other threads skip against it
                      // (not a thread's first block of the position: every
                      // thread has one at the same moment, and those atomics
                      // on one slot per row cost more than they save; the
                      // end of the position publishes it anyway)
                      if (row_slot && !none)
                        atomicMax(row_slot,
                                  (static_cast<unsigned long long>(best_key) << 32) |
                                      static_cast<unsigned long long>(
                                          0xFFFFFFFFu - static_cast<uint32_t>(best_idx)));
                    }
                  }
                }
              }
            } else {
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
                  const uint4 w = ld_shared_v4(box + ((chunk ^ (lrow & 7)) << 4));
                  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int h = 0; h < 4; ++h) {
                    v[u * 8 + 2 * h] = __uint_as_float(acc[u * 8 + 2 * h]) +
                                       __uint_as_float(ww[h] << 16);
                    v[u * 8 + 2 * h + 1] = __uint_as_float(acc[u * 8 + 2 * h + 1]) +
                                           __uint_as_float(ww[h] & 0xFFFF0000u);
                  }
                }
              } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const uint4 w = ld_shared_v4(box + ((u ^ (lrow & 7)) << 4));
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
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&l_empty[s]);
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      if (!ok) break;
      // publish this CTA's row winners and arrive at position k's barrier
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
    if (ok && sg == 0) {
      // winners of the last position
      ok = grid_wait(p, p.K - 1, m_tile, abort_flag, EPI);
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

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ==========================================================================
// host side
// ==========================================================================
EncodeTiledFn encode_tiled_fn() {
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
static bool g_attr_done[128];

template <int LDT, bool SAMPLE, int EPI, int REP>
static cudaError_t set_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(chain_kernel<LDT, SAMPLE, EPI, false, REP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       CHAIN_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(chain_kernel<LDT, SAMPLE, EPI, true, REP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              CHAIN_SMEM_BYTES);
}

static cudaError_t ensure_kernel_attrs(int dev) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (g_attr_done[dev]) return cudaSuccess;
  cudaError_t e;
  if ((e = set_smem_attr<DSPARK_BF16, true, EPI_SAMPLE, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_BF16, true, EPI_SAMPLE_REP, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_BF16, true, EPI_SAMPLE_REP, 4>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_F32, true, EPI_SAMPLE, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_F32, true, EPI_SAMPLE_REP, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_F32, true, EPI_SAMPLE_REP, 4>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_BF16, false, EPI_ARGMAX, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<DSPARK_F32, false, EPI_ARGMAX, 1>()) != cudaSuccess) return e;
  g_attr_done[dev] = true;
  return cudaSuccess;
}

size_t chain_workspace_bytes(int32_t N, int32_t K) {
  const size_t n_mtiles = (static_cast<size_t>(N) + BM - 1) / BM;
  const size_t end = chain_counters_offset(N, K) + n_mtiles * K * 4;
  return ((end + 255) / 256) * 256;
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

  const int n_quanta = (a.vocab + BQ - 1) / BQ;
  // Leave at least one SM idle so that independent work (the scheduler on
  // another stream) runs alongside the chain instead of after it; the chain
  // is HBM-bound, so the SMs it gives up cost next to nothing.
  int groups = sms / n_mtiles;
  if (n_mtiles * groups > sms - 1 && groups > 1) groups = (sms - 1) / n_mtiles;
  const int n_vgroups = std::max(1, std::min(groups, n_quanta));
  const int grid = n_mtiles * n_vgroups;

  // V: dim0 = rank (contiguous), dim1 = vocab; 64 x 64 boxes, 128-B swizzle
  CUtensorMap tmV, tmL;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.rank),
                          static_cast<cuuint64_t>(a.vocab)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.rank) * 2};
    cuuint32_t box[2] = {BK, BQ};
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
  // everything after the status word is per-call state: clear it
  const size_t clear_bytes = chain_counters_offset(a.N, a.K) +
                             static_cast<size_t>(n_mtiles) * a.K * 4 -
                             kChainAbortOffset;
  if (cudaMemsetAsync(ws + kChainAbortOffset, 0, clear_bytes, stream) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;

  ChainParams p;
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
  p.n_mtiles = n_mtiles;
  p.n_vgroups = n_vgroups;
  p.n_quanta = n_quanta;
  p.l_k_is_dim1 = l_k_is_dim1;
  p.seed_lo = a.seed_lo;
  p.seed_hi = a.seed_hi;
  p.offset = a.offset;
  p.inv_tau = a.inv_tau;
  {
    const double v_bytes = static_cast<double>(a.vocab) * a.rank * 2;
    const int tenths = static_cast<int>(10.0 * kL2KeepBytes / v_bytes);
    p.v_keep_tenths = std::max(0, std::min(10, tenths));
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  // sampling a batch of at most 32 (64) requests: every request four
  // (two) times in the tile's rows
  const int rep = a.sample ? (a.N <= 32 ? 4 : a.N <= 64 ? 2 : 1) : 1;
  cfg.blockDim = dim3(chain_threads(!a.sample ? EPI_ARGMAX
                                    : rep == 1 ? EPI_SAMPLE : EPI_SAMPLE_REP));
  cfg.dynamicSmemBytes = CHAIN_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // at most one tile per position in every CTA: the widest group is at most
  // QPT quanta
  const bool one_tile = (n_quanta + n_vgroups - 1) / n_vgroups <= QPT;
  cudaError_t e;
#define DSPARK_LAUNCH(LDT, S, E, R)                                                   \
  e = one_tile ? cudaLaunchKernelEx(&cfg, chain_kernel<LDT, S, E, true, R>, tmV, tmL, p) \
               : cudaLaunchKernelEx(&cfg, chain_kernel<LDT, S, E, false, R>, tmV, tmL, p)
#define DSPARK_LAUNCH_REP(LDT)                 \
  if (rep == 4)                                \
    DSPARK_LAUNCH(LDT, true, EPI_SAMPLE_REP, 4); \
  else if (rep == 2)                           \
    DSPARK_LAUNCH(LDT, true, EPI_SAMPLE_REP, 2); \
  else                                         \
    DSPARK_LAUNCH(LDT, true, EPI_SAMPLE, 1)
  if (a.sample) {
    if (a.logits_dtype == DSPARK_BF16) {
      DSPARK_LAUNCH_REP(DSPARK_BF16);
    } else {
      DSPARK_LAUNCH_REP(DSPARK_F32);
    }
  } else {
    if (a.logits_dtype == DSPARK_BF16)
      DSPARK_LAUNCH(DSPARK_BF16, false, EPI_ARGMAX, 1);
    else
      DSPARK_LAUNCH(DSPARK_F32, false, EPI_ARGMAX, 1);
  }
#undef DSPARK_LAUNCH_REP
#undef DSPARK_LAUNCH
  if (e == cudaErrorCooperativeLaunchTooLarge) return DSPARK_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace dspark
