// Shared device helpers: status bits, bounded mbarrier waits, orderable keys
// for argmax reductions and the tcgen05 descriptors used by the chain GEMM.
#pragma once

#include <cstdint>

#include "../../include/dspark.h"
#include "ptx.cuh"

namespace dspark {

// Every spin on an mbarrier gives up after this long, sets
// DSPARK_DEV_TIMEOUT and lets the kernel return instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bit) {
  atomicOr(status, bit);
}

// Waits for the phase of `bar` with parity `parity`.  Returns false when the
// CTA has aborted (another role timed out) or this wait timed out.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity,
                                             volatile uint32_t *abort_flag,
                                             uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    // sleeps up to 20 us per test (woken by the phase's completion), so
    // the abort flag and the time limit are still checked that often
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1u;
      raise_status(status, DSPARK_DEV_TIMEOUT);
      return false;
    }
  }
}

// Order-preserving map of fp32 to uint32: a > b  <=>  key(a) > key(b) for
// non-NaN values, -0 and +0 share a key, NaN maps above everything.
__device__ __forceinline__ uint32_t f32_key(float v) {
  if (v != v) return 0xFFFFFFFFu;
  uint32_t b = __float_as_uint(v);
  if ((b << 1) == 0u) b = 0u;  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float f32_from_key(uint32_t k) {
  if (k == 0xFFFFFFFFu) return __uint_as_float(0x7FFFFFFFu);
  return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu)
                           : __uint_as_float(~k);
}

// the same for fp64
__device__ __forceinline__ uint64_t f64_key(double v) {
  if (v != v) return 0xFFFFFFFFFFFFFFFFull;
  uint64_t b = static_cast<uint64_t>(__double_as_longlong(v));
  if ((b << 1) == 0ull) b = 0ull;
  return (b & 0x8000000000000000ull) ? ~b : (b | 0x8000000000000000ull);
}

// ------------------------------------------------------------------------
// tcgen05 operand descriptors
//
// Shared-memory matrix descriptor (64 bit), K-major operand stored in the
// 128-byte swizzled canonical layout: rows of 64 bf16 (128 B), 8-row atoms of
// 1024 B stacked along M/N, 16-byte chunk c of row r stored at c ^ (r % 8).
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (unused for this layout)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 B between atoms)
//   bits 46-48  fixed 0b001
//   bits 61-63  swizzle mode, 2 = 128-byte swizzle
// ------------------------------------------------------------------------
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(uint32_t M,
                                                           uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

}  // namespace dspark
