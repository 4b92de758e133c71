// Pieces shared by the persistent chain kernels (chain.cu, lmhead.cu): the
// vocabulary tiling, the bounded per-position grid barrier and the decoding
// of a row's packed winner key.
#pragma once

#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int BM = 128;  // requests per tile (MMA M)
constexpr int BN = 256;  // vocabulary entries per tile (MMA N, at most)
constexpr int BQ = 64;   // vocabulary quantum: tiles are 1..4 quanta wide
constexpr int QPT = BN / BQ;  // quanta per full tile
constexpr int BK = 64;   // reduction entries per K-block (128 bytes of bf16)

// Tile i of position k over the quanta [qb, qe) a CTA owns: even positions
// sweep upwards from qb, odd ones downwards from qe (the V tiles read last
// for position k are read first for k+1, while still in L2).  Every tile is
// QPT quanta wide except the last one processed.
struct TileGeom {
  int qa;  // first quantum
  int nq;  // quanta in the tile (1..QPT)
};

__device__ __forceinline__ TileGeom tile_geom(int k, int i, int qb, int qe) {
  TileGeom g;
  if ((k & 1) == 0) {
    g.qa = qb + QPT * i;
    g.nq = min(QPT, qe - g.qa);
  } else {
    const int top = qe - QPT * i;
    g.qa = max(qb, top - QPT);
    g.nq = top - g.qa;
  }
  return g;
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

// An epilogue warp waits until every epilogue warp of the CTAs sharing its
// 128-request tile has published position k (one arrival per epilogue warp
// and CTA; the tiles are independent chains).  Lane 0 polls with a time
// limit; the warp leaves together.  No barrier spans warps, so a warp that gives up can never leave
// another one blocked.
template <class P>
__device__ __forceinline__ bool grid_wait(const P &p, int k,
                                          int m_tile,
                                          volatile uint32_t *cta_abort,
                                          uint32_t arrivals_per_cta) {
  uint32_t r = 1;
  if ((threadIdx.x & 31) == 0) {
    const uint32_t target = arrivals_per_cta * static_cast<uint32_t>(p.n_vgroups) +
                            (*p.hang_test != 0u ? 1u : 0u);
    const uint32_t *cnt = &p.counters[k * p.n_mtiles + m_tile];
    if (ld_acquire_gpu(cnt) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_gpu(cnt) < target) {
        if (*cta_abort || *reinterpret_cast<volatile uint32_t *>(p.g_abort)) {
          r = 0;
          break;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          raise_status(p.status, DSPARK_DEV_TIMEOUT);
          r = 0;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  r = __shfl_sync(0xFFFFFFFFu, r, 0);
  return r != 0u;
}

__device__ __forceinline__ int decode_index(unsigned long long key, int vocab) {
  int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
  if (key == 0ull || idx < 0 || idx >= vocab) idx = 0;
  return idx;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library); nullptr if unavailable
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

}  // namespace dspark
