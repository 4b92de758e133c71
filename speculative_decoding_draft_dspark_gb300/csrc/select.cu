// Confidence-scheduled verification on sm_103a: one persistent CTA.
//
// "Adaptive Verification in vLLM", section "Scheduling the budget":
//   survival  s[n,k] = prod_{j<=k} c[n,j]                 (running product)
//   order     every sampling request's slots by survival  (global top-B)
//   budget    B = argmax_b (N_sampling + P_b) / cost[T+b], P_b the sum of
//             the b best survivals ("an np.argmax over a cumulative sum")
//   allocate  each request keeps the contiguous prefix of its selected slots
//   compact   flattened verify list with per-request offsets
// and section "The cost model": the cost table is forced monotone.  The
// whole selection runs on the GPU and never reads back to the host.
//
// Numerics: survivals are fp64 products taken left to right (each one IEEE
// multiply), sort keys are their bit patterns, and P_b is the exact sum of
// the first b survivals rounded once, computed as a fixed-point prefix scan
// (integer addition is associative, so the parallel scan gives the same
// bits as any order): 128 bits wide when every nonzero survival lies within
// 2^61 of the largest (all terms exact), 256 bits otherwise.  f(b) is then
// one fp64 add and one fp64 divide.  B is therefore decided on exactly the
// values the definition names.
//
// The order: up to 4096 slots, 64-bit composites (the survival's fp64 bits
// truncated to 50, then the slot id) sorted per warp in registers and merged
// (merge path), with a check that sends ties of the truncated key to the
// exact path; larger batches, and that case, merge the fp64 keys by slot.
//
// The kernel runs the stages requested by a mask, so the fused call and the
// four separate calls share one implementation.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr unsigned FULL = 0xFFFFFFFFu;

// ------------------------------------------------------------------------
// 256-bit fixed-point accumulator for exact sums of non-negative doubles
// ------------------------------------------------------------------------
// Every term s is written as an integer X = s * 2^-u with the unit
// u = e_max - 1075 - kFixG, e_max being the biased exponent of the largest
// term: the largest term occupies bits [kFixG, kFixG + 53) and a sum of up
// to 2^14 terms stays below bit 256.  Bits of terms smaller than 2^-kFixG
// times the largest fall below the unit; they are folded into a sticky bit,
// which keeps the final rounding exact (they cannot reach the rounding
// position, kFixG - 53 bits above the unit).
constexpr int kFixG = 188;

struct Acc256 {
  unsigned long long w0, w1, w2, w3;
  uint32_t sticky;
};

__device__ __forceinline__ Acc256 acc_zero() { return Acc256{0, 0, 0, 0, 0}; }

__device__ __forceinline__ void acc_add(Acc256 &a, const Acc256 &b) {
  asm("add.cc.u64 %0, %0, %4;\n\t"
      "addc.cc.u64 %1, %1, %5;\n\t"
      "addc.cc.u64 %2, %2, %6;\n\t"
      "addc.u64 %3, %3, %7;"
      : "+l"(a.w0), "+l"(a.w1), "+l"(a.w2), "+l"(a.w3)
      : "l"(b.w0), "l"(b.w1), "l"(b.w2), "l"(b.w3));
  a.sticky |= b.sticky;
}

__device__ __forceinline__ unsigned long long acc_word(const Acc256 &a, int i) {
  return i == 0 ? a.w0 : i == 1 ? a.w1 : i == 2 ? a.w2 : i == 3 ? a.w3 : 0ull;
}

// m * 2^shift restricted to word i (bits [64 i, 64 i + 64)), m < 2^53
__device__ __forceinline__ unsigned long long shifted_word(unsigned long long m,
                                                           int shift, int i) {
  const int d = shift - 64 * i;
  if (d >= 0 && d < 64) return m << d;
  if (d < 0 && d > -64) return m >> (-d);
  return 0ull;
}

__device__ __forceinline__ Acc256 to_fixed(double s, int e_max) {
  Acc256 r = acc_zero();
  const unsigned long long bits =
      static_cast<unsigned long long>(__double_as_longlong(s));
  int ex = static_cast<int>((bits >> 52) & 0x7FF);
  unsigned long long m = bits & 0xFFFFFFFFFFFFFull;
  if (ex == 0)
    ex = 1;
  else
    m |= 1ull << 52;
  if (m == 0ull) return r;
  const int shift = ex - e_max + kFixG;
  if (shift >= 0) {
    r.w0 = shifted_word(m, shift, 0);
    r.w1 = shifted_word(m, shift, 1);
    r.w2 = shifted_word(m, shift, 2);
    r.w3 = shifted_word(m, shift, 3);
  } else if (shift > -53) {
    const int sh = -shift;
    r.w0 = m >> sh;
    r.sticky = (m & ((1ull << sh) - 1ull)) != 0ull;
  } else {
    r.sticky = 1u;
  }
  return r;
}

__device__ __forceinline__ uint32_t acc_bit(const Acc256 &a, int pos) {
  return static_cast<uint32_t>((acc_word(a, pos >> 6) >> (pos & 63)) & 1ull);
}

// any of the bits [0, pos) set
__device__ __forceinline__ bool acc_any_below(const Acc256 &a, int pos) {
  if (pos <= 0) return false;
  const int wi = pos >> 6, bi = pos & 63;
  bool any = false;
  if (wi > 0) any |= a.w0 != 0ull;
  if (wi > 1) any |= a.w1 != 0ull;
  if (wi > 2) any |= a.w2 != 0ull;
  if (wi > 3) any |= a.w3 != 0ull;
  if (bi != 0 && wi < 4) any |= (acc_word(a, wi) & ((1ull << bi) - 1ull)) != 0ull;
  return any;
}

// bits [pos, pos + 53) of a, pos >= 0
__device__ __forceinline__ unsigned long long acc_extract53(const Acc256 &a,
                                                             int pos) {
  const int wi = pos >> 6, bi = pos & 63;
  unsigned long long v = acc_word(a, wi) >> bi;
  if (bi != 0) v |= acc_word(a, wi + 1) << (64 - bi);
  return v & ((1ull << 53) - 1ull);
}

// a * 2^u rounded to the nearest double, ties to even
__device__ __forceinline__ double from_fixed(const Acc256 &a, int e_max) {
  int h = -1;
  if (a.w3)
    h = 192 + 63 - __clzll(static_cast<long long>(a.w3));
  else if (a.w2)
    h = 128 + 63 - __clzll(static_cast<long long>(a.w2));
  else if (a.w1)
    h = 64 + 63 - __clzll(static_cast<long long>(a.w1));
  else if (a.w0)
    h = 63 - __clzll(static_cast<long long>(a.w0));
  if (h < 0) return 0.0;
  const int u = e_max - 1075 - kFixG;
  int rb = h - 52;                 // lowest bit a 53-bit significand keeps
  const int rb_sub = -1074 - u;    // lowest bit a subnormal keeps
  if (rb < rb_sub) rb = rb_sub;
  if (rb < 0) rb = 0;              // whole value fits: exact
  unsigned long long mant = acc_extract53(a, rb);
  const bool round = rb >= 1 && acc_bit(a, rb - 1);
  const bool sticky = a.sticky != 0u || acc_any_below(a, rb - 1);
  if (round && (sticky || (mant & 1ull))) mant += 1ull;
  int e2 = rb + u;                 // value = mant * 2^e2
  if (mant == (1ull << 53)) {
    mant >>= 1;
    e2 += 1;
  }
  unsigned long long bits;
  if (mant >= (1ull << 52))
    bits = (static_cast<unsigned long long>(e2 + 52 + 1023) << 52) |
           (mant & ((1ull << 52) - 1ull));
  else
    bits = mant;  // subnormal, e2 == -1074
  return __longlong_as_double(static_cast<long long>(bits));
}

// ------------------------------------------------------------------------
// 128-bit form of the same fixed point, for when every nonzero term lies
// within 2^-kFixG128 of the largest: the largest term occupies bits
// [kFixG128, kFixG128 + 53), every term is an exact integer (no sticky
// bit), and a sum of up to 2^14 terms stays below bit 128.  The sums are
// then exact and one rounding gives the same double as the 256-bit form.
// ------------------------------------------------------------------------
constexpr int kFixG128 = 61;

struct Acc128 {
  unsigned long long lo, hi;
};

__device__ __forceinline__ void acc128_add(Acc128 &a, const Acc128 &b) {
  asm("add.cc.u64 %0, %0, %2;\n\t"
      "addc.u64 %1, %1, %3;"
      : "+l"(a.lo), "+l"(a.hi)
      : "l"(b.lo), "l"(b.hi));
}

// s * 2^-u, u = e_max - 1075 - kFixG128; requires the biased exponent of s
// (1 for subnormals) >= e_max - kFixG128
__device__ __forceinline__ Acc128 to_fixed128(double s, int e_max) {
  const unsigned long long bits =
      static_cast<unsigned long long>(__double_as_longlong(s));
  int ex = static_cast<int>((bits >> 52) & 0x7FF);
  unsigned long long m = bits & 0xFFFFFFFFFFFFFull;
  if (ex == 0)
    ex = 1;
  else
    m |= 1ull << 52;
  const int shift = ex - e_max + kFixG128;  // 0 .. kFixG128
  Acc128 r;
  r.lo = m << shift;
  r.hi = shift == 0 ? 0ull : m >> (64 - shift);
  return r;
}

// (hi:lo) * 2^u rounded to the nearest double, ties to even: the bit
// pattern of the non-negative, finite result (no caller comes near the
// overflow threshold)
__device__ __forceinline__ unsigned long long round_u128_to_f64(unsigned long long lo,
                                                               unsigned long long hi,
                                                               int u) {
  int h;
  if (hi)
    h = 64 + 63 - __clzll(static_cast<long long>(hi));
  else if (lo)
    h = 63 - __clzll(static_cast<long long>(lo));
  else
    return 0ull;
  int rb = h - 52;                 // lowest bit a 53-bit significand keeps
  const int rb_sub = -1074 - u;    // lowest bit a subnormal keeps
  if (rb < rb_sub) rb = rb_sub;
  unsigned long long mant;
  if (rb <= 0) {
    mant = lo << (-rb);            // the whole value fits (< 2^53): exact
  } else {
    if (rb > h + 1) return 0ull;   // below half the smallest subnormal
    mant = rb >= 64 ? hi >> (rb - 64) : (lo >> rb) | (hi << (64 - rb));
    mant &= (1ull << 53) - 1ull;
    const int pos = rb - 1;        // the round bit
    bool round, sticky;
    if (pos >= 64) {
      round = (hi >> (pos - 64)) & 1ull;
      sticky = lo != 0ull || (hi & ((1ull << (pos - 64)) - 1ull)) != 0ull;
    } else {
      round = (lo >> pos) & 1ull;
      sticky = pos > 0 && (lo & ((1ull << pos) - 1ull)) != 0ull;
    }
    if (round && (sticky || (mant & 1ull))) mant += 1ull;
  }
  int e2 = rb + u;                 // value = mant * 2^e2
  if (mant == (1ull << 53)) {
    mant >>= 1;
    e2 += 1;
  }
  return mant >= (1ull << 52)
             ? (static_cast<unsigned long long>(e2 + 52 + 1023) << 52) |
                   (mant & ((1ull << 52) - 1ull))
             : mant;  // subnormal, e2 == -1074
}

// a * 2^u rounded to the nearest double, ties to even
__device__ __forceinline__ double from_fixed128(const Acc128 &a, int e_max) {
  return __longlong_as_double(static_cast<long long>(
      round_u128_to_f64(a.lo, a.hi, e_max - 1075 - kFixG128)));
}

// ------------------------------------------------------------------------
// Conversions between fp32 and fp64 in integer arithmetic, exact (IEEE,
// ties to even): the fp64 pipe of this part issues about one warp
// instruction per 64 cycles of an SM sub-partition, conversions included,
// so the survival loop keeps only its multiply there (a 15-position batch
// of 1024 requests: 16.5 us with the conversions on the fp64 pipe, 9.5 us
// without).  An integer form of the multiply measured slower than the pipe.
// ------------------------------------------------------------------------
// batches from this many slots take the integer conversions
constexpr int kIntCvtMinSlots = 4096;

// c as a double, for c a non-negative finite float
__device__ __forceinline__ double f32_to_f64(float c) {
  const uint32_t b = __float_as_uint(c);
  const uint32_t e = b >> 23;  // sign 0
  uint32_t m = b & 0x7FFFFFu;
  unsigned long long bits;
  if (e != 0) {
    bits = (static_cast<unsigned long long>(e + 896u) << 52) |
           (static_cast<unsigned long long>(m) << 29);
  } else if (m != 0) {           // subnormal: normalise the significand
    const int sh = __clz(m) - 8;  // brings the top bit to bit 23
    m <<= sh;
    bits = (static_cast<unsigned long long>(897 - sh) << 52) |
           (static_cast<unsigned long long>(m & 0x7FFFFFu) << 29);
  } else {
    bits = 0ull;
  }
  return __longlong_as_double(static_cast<long long>(bits));
}

// d rounded to the nearest float, for d a non-negative double below 2^127
__device__ __forceinline__ float f64_to_f32_rn(double d) {
  const unsigned long long b =
      static_cast<unsigned long long>(__double_as_longlong(d));
  const int e = static_cast<int>(b >> 52);  // sign 0
  if (e == 0) return 0.0f;  // fp64 subnormals lie far below half an fp32 one
  const unsigned long long m = (b & ((1ull << 52) - 1ull)) | (1ull << 52);
  const int e32 = e - 1023 + 127;  // biased fp32 exponent of a normal result
  const int sh = e32 >= 1 ? 29 : 29 + 1 - e32;  // bits dropped from m
  if (sh > 54) return 0.0f;
  unsigned long long q = m >> sh;
  const bool round = (m >> (sh - 1)) & 1ull;
  const bool sticky = (m & ((1ull << (sh - 1)) - 1ull)) != 0ull;
  if (round && (sticky || (q & 1ull))) q += 1ull;
  // normal: q in [2^23, 2^24], a carry lands in the exponent (up to 2^127
  // at most); subnormal: q below 2^23, or 2^23 for the smallest normal
  const uint32_t bits = e32 >= 1
                            ? (static_cast<uint32_t>(e32 - 1) << 23) + static_cast<uint32_t>(q)
                            : static_cast<uint32_t>(q);
  return __uint_as_float(bits);
}

// ------------------------------------------------------------------------
// block-level scans and reductions (blockDim = SEL_THREADS)
// ------------------------------------------------------------------------
__device__ __forceinline__ int shfl_up(int v, int o) { return __shfl_up_sync(FULL, v, o); }
__device__ __forceinline__ float shfl_up(float v, int o) { return __shfl_up_sync(FULL, v, o); }
__device__ __forceinline__ float shfl_down(float v, int o) { return __shfl_down_sync(FULL, v, o); }
__device__ __forceinline__ Acc256 shfl_up(const Acc256 &v, int o) {
  Acc256 r;
  r.w0 = __shfl_up_sync(FULL, v.w0, o);
  r.w1 = __shfl_up_sync(FULL, v.w1, o);
  r.w2 = __shfl_up_sync(FULL, v.w2, o);
  r.w3 = __shfl_up_sync(FULL, v.w3, o);
  r.sticky = __shfl_up_sync(FULL, v.sticky, o);
  return r;
}

__device__ __forceinline__ Acc128 shfl_up(const Acc128 &v, int o) {
  Acc128 r;
  r.lo = __shfl_up_sync(FULL, v.lo, o);
  r.hi = __shfl_up_sync(FULL, v.hi, o);
  return r;
}

struct OpAddInt {
  __device__ int operator()(int a, int b) const { return a + b; }
};
struct OpMinInt {
  __device__ int operator()(int a, int b) const { return a < b ? a : b; }
};
struct OpMaxNan {
  __device__ float operator()(float a, float b) const { return fmax_nan(a, b); }
};
struct OpMinNan {
  __device__ float operator()(float a, float b) const {
    float d;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
  }
};
// two running maxima scanned together
struct MaxPair {
  float pre, run;
};
__device__ __forceinline__ MaxPair shfl_up(const MaxPair &v, int o) {
  return MaxPair{__shfl_up_sync(FULL, v.pre, o), __shfl_up_sync(FULL, v.run, o)};
}
struct OpMaxPair {
  __device__ MaxPair operator()(const MaxPair &a, const MaxPair &b) const {
    return MaxPair{fmax_nan(a.pre, b.pre), fmax_nan(a.run, b.run)};
  }
};

struct OpAcc {
  __device__ Acc256 operator()(Acc256 a, const Acc256 &b) const {
    acc_add(a, b);
    return a;
  }
};

struct OpAcc128 {
  __device__ Acc128 operator()(Acc128 a, const Acc128 &b) const {
    acc128_add(a, b);
    return a;
  }
};

// exclusive scan in thread order; `sh` holds SEL_WARPS + 1 values
template <typename T, typename Op>
__device__ T block_excl_scan(T v, Op op, T ident, T *sh, T *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = shfl_up(x, o);
    if (lane >= o) x = op(y, x);
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    T t = sh[lane];
    T s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = shfl_up(s, o);
      if (lane >= o) s = op(y, s);
    }
    T prev = shfl_up(s, 1);
    sh[lane] = lane == 0 ? ident : prev;
    if (lane == 31) sh[SEL_WARPS] = s;
  }
  __syncthreads();
  T in_warp = shfl_up(x, 1);
  if (lane == 0) in_warp = ident;
  T r = op(sh[w], in_warp);
  if (total) *total = sh[SEL_WARPS];
  __syncthreads();
  return r;
}

// exclusive scan in reverse thread order: op over the values of threads
// tid+1 .. blockDim-1
template <typename Op>
__device__ float block_excl_scan_rev(float v, Op op, float ident, float *sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float y = shfl_down(x, o);
    if (lane + o < 32) x = op(x, y);
  }
  if (lane == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    float s = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y = shfl_down(s, o);
      if (lane + o < 32) s = op(s, y);
    }
    float next = shfl_down(s, 1);
    sh[lane] = lane == 31 ? ident : next;
  }
  __syncthreads();
  float in_warp = shfl_down(x, 1);
  if (lane == 31) in_warp = ident;
  const float r = op(in_warp, sh[w]);
  __syncthreads();
  return r;
}

template <typename T, typename Op>
__device__ T block_reduce(T v, Op op, T ident, T *sh) {
  T tot;
  block_excl_scan(v, op, ident, sh, &tot);
  return tot;
}

// argmax over (orderable key, index): larger key, then smaller index
__device__ void block_argmax(unsigned long long &key, int &idx,
                             unsigned long long *shk, int *shi) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long k2 = __shfl_down_sync(FULL, key, o);
    const int i2 = __shfl_down_sync(FULL, idx, o);
    if (k2 > key || (k2 == key && i2 < idx)) {
      key = k2;
      idx = i2;
    }
  }
  if (lane == 0) {
    shk[w] = key;
    shi[w] = idx;
  }
  __syncthreads();
  if (w == 0) {
    key = shk[lane];
    idx = shi[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long k2 = __shfl_down_sync(FULL, key, o);
      const int i2 = __shfl_down_sync(FULL, idx, o);
      if (k2 > key || (k2 == key && i2 < idx)) {
        key = k2;
        idx = i2;
      }
    }
    if (lane == 0) {
      shk[SEL_WARPS] = key;
      shi[SEL_WARPS] = idx;
    }
  }
  __syncthreads();
  key = shk[SEL_WARPS];
  idx = shi[SEL_WARPS];
  __syncthreads();
}

// first index with value (smaller index wins), carrying a double payload
__device__ void block_argmin_idx(int &idx, double &val, int *shi, double *shv) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int i2 = __shfl_down_sync(FULL, idx, o);
    const double v2 = __shfl_down_sync(FULL, val, o);
    if (i2 < idx) {
      idx = i2;
      val = v2;
    }
  }
  if (lane == 0) {
    shi[w] = idx;
    shv[w] = val;
  }
  __syncthreads();
  if (w == 0) {
    idx = shi[lane];
    val = shv[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int i2 = __shfl_down_sync(FULL, idx, o);
      const double v2 = __shfl_down_sync(FULL, val, o);
      if (i2 < idx) {
        idx = i2;
        val = v2;
      }
    }
    if (lane == 0) {
      shi[SEL_WARPS] = idx;
      shv[SEL_WARPS] = val;
    }
  }
  __syncthreads();
  idx = shi[SEL_WARPS];
  val = shv[SEL_WARPS];
  __syncthreads();
}

__device__ __forceinline__ double key_value(unsigned long long key) {
  return __longlong_as_double(static_cast<long long>(key - 1ull));
}

__device__ __forceinline__ double f64_from_key(unsigned long long k) {
  if (k == 0xFFFFFFFFFFFFFFFFull)
    return __longlong_as_double(0x7FF8000000000000ll);
  const unsigned long long b =
      (k & 0x8000000000000000ull) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
  return __longlong_as_double(static_cast<long long>(b));
}

// ------------------------------------------------------------------------
// global priority order (larger key first, then smaller slot) of NK slots,
// on the fp64 keys: the requests' runs of K arrive sorted (a survival never
// increases along a request), and level l merges neighbouring runs of
// K * 2^l (merge path): every thread writes ceil(NK / blockDim), at least
// four, consecutive outputs, finding how many of them come from the left
// run by a binary search (the co-rank) and then merging sequentially.  Only
// 16-bit slot ids move (between sidx and stmp); keys stay indexed by slot.
// n log2(n / K) merge steps in log2(NK / K) levels.  On return sidx[0 ..
// NK) is the order and keys[0 .. NK) the keys in that order.  Batches of
// more than 4096 slots take this path; smaller ones only when the fast
// order below finds two survivals it cannot tell apart.
// ------------------------------------------------------------------------
__device__ __forceinline__ bool prio_first(unsigned long long ka, uint32_t sa,
                                           unsigned long long kb, uint32_t sb) {
  return ka > kb || (ka == kb && sa < sb);
}

constexpr int kMaxPerThread = (kMaxSlots + SEL_THREADS - 1) / SEL_THREADS;
// outputs per thread and merge level, at least: fewer, longer runs mean
// fewer co-rank searches, which bound a level (random key reads)
constexpr int kMergeMinOut = 4;

__device__ void block_merge_runs(unsigned long long *keys, uint16_t *sidx,
                                 uint16_t *stmp, const int NK, const int K) {
  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int C = (NK + NT - 1) / NT;  // final reorder: outputs per thread
  const int p0 = min(NK, tid * C), p1 = min(NK, p0 + C);
  const int Cm = max(C, kMergeMinOut);  // merge levels: outputs per thread
  const int m0 = min(NK, tid * Cm), m1 = min(NK, m0 + Cm);
  uint16_t *src = sidx, *dst = stmp;
  __syncthreads();  // the keys are in place
  for (int i = tid; i < NK; i += NT) sidx[i] = static_cast<uint16_t>(i);
  __syncthreads();
  for (int L = K; L < NK; L <<= 1) {
    int p = m0;
    while (p < m1) {
      // the pair of runs [base, base + L) and [base + L, base + 2L) holding p
      const int base = p - p % (2 * L);
      const int a_len = min(L, NK - base);
      const int b0 = base + a_len;
      const int b_len = min(L, NK - b0);
      const uint16_t *A = src + base;
      const uint16_t *B = src + b0;
      const int q = p - base;
      // co-rank: the number of A's elements among the pair's first q outputs
      int lo = max(0, q - b_len), hi = min(q, a_len);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const uint32_t x = A[mid], y = B[q - mid - 1];
        if (prio_first(keys[x], x, keys[y], y))
          lo = mid + 1;
        else
          hi = mid;
      }
      int ia = lo, ib = q - lo;
      // heads of both runs; an exhausted run's head is never taken (its
      // index is clamped so the read stays inside the run)
      uint32_t xa = A[min(ia, a_len - 1)];
      uint32_t xb = b_len > 0 ? B[min(ib, b_len - 1)] : 0u;
      unsigned long long ka = keys[xa], kb = keys[xb];
      const int stop = min(m1, b0 + b_len);
      for (; p < stop; ++p) {
        const bool take_a = ia < a_len && (ib >= b_len || prio_first(ka, xa, kb, xb));
        dst[p] = static_cast<uint16_t>(take_a ? xa : xb);
        ia += take_a ? 1 : 0;
        ib += take_a ? 0 : 1;
        // refill the head that moved, without a branch
        const uint16_t *next = take_a ? A + min(ia, a_len - 1) : B + min(ib, max(b_len - 1, 0));
        const uint32_t x = *next;
        const unsigned long long kx = keys[x];
        xa = take_a ? x : xa;
        ka = take_a ? kx : ka;
        xb = take_a ? xb : x;
        kb = take_a ? kb : kx;
      }
    }
    __syncthreads();
    uint16_t *t = src;
    src = dst;
    dst = t;
  }
  // keys into sorted order: every thread reads its outputs' keys before any
  // thread writes
  unsigned long long kv[kMaxPerThread];
#pragma unroll
  for (int c = 0; c < kMaxPerThread; ++c)
    if (p0 + c < p1) kv[c] = keys[src[p0 + c]];
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kMaxPerThread; ++c) {
    if (p0 + c < p1) {
      keys[p0 + c] = kv[c];
      if (src != sidx) sidx[p0 + c] = src[p0 + c];
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------------
// Fast order for up to kFastMaxNK slots, on one 64-bit composite per slot:
// the top 50 bits of the survival's fp64 pattern (sign 0, exponent, 38
// mantissa bits), subtracted from their largest value, then the 14-bit
// slot; non-sampling slots get a key part above every survival.  Ascending
// composites are survival descending, slot ascending, and every comparison
// is one 64-bit compare of one shared-memory word.  Each warp first sorts
// segments of 128 composites in registers (a bitonic network over
// shuffles), then merge levels (merge path, as above) combine the runs.
// Truncating the bit pattern is monotone, so the result is the fp64 order
// wherever neighbours differ in those 50 bits; two neighbours equal there
// but different in fp64 (within 2^-38 of each other) are detected
// afterwards and send the whole order to the fp64 merge above.
// ------------------------------------------------------------------------
constexpr int kFastMaxNK = 4096;
constexpr int kCompSlotBits = 14;  // slot ids below 16384
constexpr int kCompDrop = 14;      // fp64 bits dropped from the key part
// key part of survival 0 (bits 0) is kCompTop; of 1.0, kCompTop - (1.0's
// bits >> kCompDrop); the key part of non-sampling slots is kCompTop + 1
constexpr unsigned long long kCompTop = 0x3FF0000000000000ull >> kCompDrop;
constexpr unsigned long long kCompNonSampling = (kCompTop + 1ull) << kCompSlotBits;
static_assert(kFastMaxNK <= (1 << kCompSlotBits), "slot ids fit the composite");
static_assert(((kCompTop + 1ull) << kCompSlotBits) < ~0ull - (1ull << kCompSlotBits),
              "composites stay below the padding value");
constexpr int kCompSegPerLane = 4;
constexpr int kCompSegLen = 32 * kCompSegPerLane;

// ascending bitonic sort of the warp's 32 * E composites (lane l holds
// elements l * E .. l * E + E - 1); fully unrolled (a rolled form with
// runtime stage and distance loops measured slower)
template <int E>
__device__ __forceinline__ void warp_bitonic_composite(unsigned long long (&v)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 2; s <= 32 * E; s <<= 1) {
#pragma unroll
    for (int d = s >> 1; d >= E; d >>= 1) {  // partner in another lane
      const int m = d / E;
      const bool lower = (lane & m) == 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned long long o = __shfl_xor_sync(FULL, v[e], m);
        const bool up = ((lane * E + e) & s) == 0;
        v[e] = (lower == up) ? (o < v[e] ? o : v[e]) : (o > v[e] ? o : v[e]);
      }
    }
#pragma unroll
    for (int dd = E / 2; dd >= 1; dd >>= 1) {  // partner in this lane
      if (dd >= s) continue;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e & dd) continue;
        const int ee = e | dd;
        const bool up = ((lane * E + e) & s) == 0;
        const unsigned long long x = v[e], y = v[ee];
        const bool sw = up ? (x > y) : (x < y);
        v[e] = sw ? y : x;
        v[ee] = sw ? x : y;
      }
    }
  }
}

// Orders keys[0 .. NK) (fp64 survival bits + 1 by slot, 0 for non-sampling)
// with the composites; ca, cb hold NK composites each.  Returns false, with
// keys and sidx untouched, if two eligible neighbours tie in fp32 but differ
// in fp64.
__device__ bool fast_order(unsigned long long *keys, uint16_t *sidx,
                           unsigned long long *ca, unsigned long long *cb,
                           const int NK, const int S) {
  constexpr int E = kCompSegPerLane;
  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = NT >> 5;
  // composites, sorted per 128-slot segment
  for (int base = warp * kCompSegLen; base < NK; base += nwarps * kCompSegLen) {
    unsigned long long v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = base + lane * E + e;
      unsigned long long c = ~0ull;  // past NK: sorts last, not written
      if (i < NK) {
        const unsigned long long k = keys[i];
        c = k == 0ull ? kCompNonSampling
                      : ((kCompTop - ((k - 1ull) >> kCompDrop)) << kCompSlotBits);
        c |= static_cast<unsigned long long>(i);
      }
      v[e] = c;
    }
    warp_bitonic_composite<E>(v);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = base + lane * E + e;
      if (i < NK) ca[i] = v[e];
    }
  }
  __syncthreads();
  // merge levels: every thread writes Cm consecutive outputs of a pair of
  // runs after finding its co-rank by binary search
  const int Cm = max((NK + NT - 1) / NT, kMergeMinOut);
  const int m0 = min(NK, tid * Cm), m1 = min(NK, m0 + Cm);
  unsigned long long *src = ca, *dst = cb;
  for (int L = kCompSegLen; L < NK; L <<= 1) {
    int p = m0;
    while (p < m1) {
      const int base = p - p % (2 * L);
      const int a_len = min(L, NK - base);
      const int b0 = base + a_len;
      const int b_len = min(L, NK - b0);
      const unsigned long long *A = src + base;
      const unsigned long long *B = src + b0;
      const int q = p - base;
      int lo = max(0, q - b_len), hi = min(q, a_len);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (A[mid] < B[q - mid - 1])
          lo = mid + 1;
        else
          hi = mid;
      }
      int ia = lo, ib = q - lo;
      unsigned long long ka = ia < a_len ? A[ia] : ~0ull;
      unsigned long long kb = ib < b_len ? B[ib] : ~0ull;
      const int stop = min(m1, b0 + b_len);
      for (; p < stop; ++p) {
        const bool take_a = ka < kb;  // composites are distinct; ~0 = exhausted
        dst[p] = take_a ? ka : kb;
        if (take_a) {
          ++ia;
          ka = ia < a_len ? A[ia] : ~0ull;
        } else {
          ++ib;
          kb = ib < b_len ? B[ib] : ~0ull;
        }
      }
    }
    __syncthreads();
    unsigned long long *t = src;
    src = dst;
    dst = t;
  }
  // eligible neighbours with equal key parts must be equal in fp64
  constexpr unsigned long long kSlotMask = (1ull << kCompSlotBits) - 1ull;
  int bad = 0;
  for (int j = tid; j + 1 < S; j += NT) {
    const unsigned long long x = src[j], y = src[j + 1];
    if ((x >> kCompSlotBits) == (y >> kCompSlotBits) &&
        keys[x & kSlotMask] != keys[y & kSlotMask])
      bad = 1;
  }
  if (__syncthreads_or(bad)) return false;
  // slots and keys into sorted order (all reads before any write)
  constexpr int kMaxOut = (kFastMaxNK + SEL_THREADS - 1) / SEL_THREADS;
  unsigned long long kv[kMaxOut];
  uint32_t sv[kMaxOut];
#pragma unroll
  for (int c = 0; c < kMaxOut; ++c) {
    const int j = tid + c * NT;
    if (j < NK) {
      sv[c] = static_cast<uint32_t>(src[j] & kSlotMask);
      kv[c] = keys[sv[c]];
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kMaxOut; ++c) {
    const int j = tid + c * NT;
    if (j < NK) {
      keys[j] = kv[c];
      sidx[j] = static_cast<uint16_t>(sv[c]);
    }
  }
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------------
// the scheduler kernel
// ------------------------------------------------------------------------
constexpr int kMaxChunk = (kMaxSlots + 1 + SEL_THREADS - 1) / SEL_THREADS + 1;

// Survival products of `conf` (fp64, left to right, clamped) and sort keys
// (bits(s) + 1, 0 for non-sampling requests), by slot; returns this
// thread's count of sampling requests.  kIntCvt: the fp32 <-> fp64
// conversions in integer arithmetic, which pays once the fp64 pipe is the
// bound (thousands of slots); small batches wait on the longer dependent
// chain instead, and keep the pipe's conversions.
template <bool kIntCvt>
__device__ __forceinline__ int survival_products(const SelectArgs &a, const float *conf,
                                                 const bool outputs,
                                                 unsigned long long *keys, uint32_t &st) {
  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int N = a.N, K = a.K;
  int my_ns = 0;
  constexpr int KG = 8;  // confidences loaded together (one memory round trip)
  for (int n = tid; n < N; n += NT) {
    const bool samp = a.mask == nullptr || a.mask[n] != 0;
    my_ns += samp ? 1 : 0;
    const float *cn = conf + static_cast<size_t>(n) * K;
    double prod = 1.0;
    for (int k0 = 0; k0 < K; k0 += KG) {
      float cg[KG];
#pragma unroll
      for (int u = 0; u < KG; ++u) cg[u] = k0 + u < K ? cn[k0 + u] : 0.0f;
#pragma unroll
      for (int u = 0; u < KG; ++u) {
        const int k = k0 + u;
        if (k >= K) break;
        float c = cg[u];
        if (!(c >= 0.0f && c <= 1.0f)) {
          st |= DSPARK_DEV_CONF_OOR;
          c = (c > 1.0f) ? 1.0f : 0.0f;  // NaN and negatives -> 0
        }
        if (c == 0.0f) c = 0.0f;  // -0 -> +0: sort keys are bit patterns
        prod = __dmul_rn(prod, kIntCvt ? f32_to_f64(c) : static_cast<double>(c));
        if (outputs && a.survival)
          a.survival[static_cast<size_t>(n) * K + k] =
              samp ? (kIntCvt ? f64_to_f32_rn(prod) : __double2float_rn(prod)) : 0.0f;
        keys[n * K + k] =
            samp ? static_cast<unsigned long long>(__double_as_longlong(prod)) + 1ull
                 : 0ull;
      }
    }
  }
  return my_ns;
}

// Survival products of `conf` (fp64, left to right, clamped), sort keys
// (bits(s) + 1, 0 for non-sampling requests) and the merged order.  With
// `outputs`, writes survival, sorted_slots, n_eligible and n_sampling.
__device__ void survival_order(const SelectArgs &a, const float *conf,
                               const bool outputs, unsigned long long *keys,
                               uint16_t *sidx, uint16_t *stmp,
                               unsigned long long *sortbuf, int *sh_int, int &n_s,
                               uint32_t &st, const int T_pf) {
  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int N = a.N, K = a.K, NK = N * K;
  const int my_ns = NK >= kIntCvtMinSlots
                        ? survival_products<true>(a, conf, outputs, keys, st)
                        : survival_products<false>(a, conf, outputs, keys, st);
  n_s = block_reduce(my_ns, OpAddInt(), 0, sh_int);
  const int S = n_s * K;
  // the cost entries the budget reads into L1 (128-byte lines) while the
  // order is built: cost[T .. T + S], and with forcing also the entries
  // before T (running max) or after T + S (suffix minimum)
  if (T_pf >= 0 && T_pf < a.L) {
    const int lo = (a.flags & DSPARK_COST_FORCE_MONOTONE) ? 0 : T_pf;
    const int hi = (a.flags & DSPARK_COST_FORCE_SUFFIX_MIN) ? a.L : min(a.L, T_pf + S + 1);
    for (int line = (lo >> 5) + tid; line * 32 < hi; line += NT)  // 32 floats a line
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a.cost + line * 32));
  }

  bool done = false;
  if (NK <= kFastMaxNK) {
    __syncthreads();  // keys by slot are in place
    done = fast_order(keys, sidx, sortbuf, sortbuf + NK, NK, S);
  }
  if (!done) block_merge_runs(keys, sidx, stmp, NK, K);
  if (outputs) {
    if (a.sorted_slots)
      for (int j = tid; j < S; j += NT) a.sorted_slots[j] = sidx[j];
    if (tid == 0) {
      if (a.n_eligible) *a.n_eligible = S;
      if (a.n_sampling) *a.n_sampling = n_s;
    }
  }
}

__global__ void __launch_bounds__(SEL_THREADS, 1)
    select_kernel(const SelectArgs a, const uint32_t stages, const int cap) {
  extern __shared__ __align__(16) uint8_t dsm[];
  // cap = N * K slots (0 without the survival stage)
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(dsm);  // [cap+1]
  uint16_t *sidx = reinterpret_cast<uint16_t *>(keys + cap + 1);          // [cap]
  uint16_t *stmp = sidx + cap;                                            // [cap]
  // two composite arrays for the fast order: [2 * cap]
  unsigned long long *sortbuf = reinterpret_cast<unsigned long long *>(
      dsm + ((static_cast<size_t>(cap + 1) * 8 + static_cast<size_t>(cap) * 4 + 7) & ~static_cast<size_t>(7)));
  double *Pd = reinterpret_cast<double *>(keys);  // after the scan: P_{j+1}
  int *len_sm = reinterpret_cast<int *>(dsm);     // after the budget

  __shared__ int sh_int[SEL_WARPS + 1];
  __shared__ float sh_f[SEL_WARPS + 1];
  __shared__ MaxPair sh_mp[SEL_WARPS + 1];
  __shared__ Acc256 sh_acc[SEL_WARPS + 1];
  __shared__ unsigned long long sh_k[SEL_WARPS + 1];
  __shared__ double sh_d[SEL_WARPS + 1];
  __shared__ int sh_B;

  const int tid = threadIdx.x;
  const int NT = blockDim.x;
  const int N = a.N, K = a.K, NK = N * K;
  const bool fused_order = (stages & kStageSurvival) != 0;
  int S = 0, n_s = 0;
  uint32_t st = 0;

  // The budget reads cost[T .. T + b_max]: T is loaded now and the slice
  // pulled into L1 before the order phase (see survival_order)
  const int T_pf = (stages & kStageBudget) && (stages & kStageSurvival) ? *a.T_dev : -1;

  // ---------------------------------------------------- survival + order
  // Stale sizing: the budget comes from a.conf_size, then survival and order
  // are rebuilt from a.conf for the allocation.
  const bool stale = a.conf_size != nullptr && (stages & kStageSurvival) &&
                     (stages & kStageBudget) && (stages & kStageAllocate);
  if (stages & kStageSurvival) {
    survival_order(a, stale ? a.conf_size : a.conf, !stale, keys, sidx, stmp, sortbuf,
                   sh_int, n_s, st, T_pf);
    S = n_s * K;

    // exact prefix sums of the sorted survivals
    int e_max = 1;
    if (S > 0) {
      const int ex = static_cast<int>(((keys[0] - 1ull) >> 52) & 0x7FF);
      e_max = ex == 0 ? 1 : ex;
    }
    const int C = (S + NT - 1) / NT;
    const int j0 = min(S, tid * C), j1 = min(S, j0 + C);
    // the smallest nonzero survival: the sorted keys end with the zeros
    // (key 1), so it sits just before the first of them
    if (tid == 0) sh_int[SEL_WARPS] = e_max;
    __syncthreads();
    for (int j = j0; j < j1; ++j) {
      if (keys[j] != 1ull && (j + 1 == S || keys[j + 1] == 1ull)) {
        const int ex = static_cast<int>(((keys[j] - 1ull) >> 52) & 0x7FF);
        sh_int[SEL_WARPS] = ex == 0 ? 1 : ex;
      }
    }
    __syncthreads();
    const bool narrow = sh_int[SEL_WARPS] >= e_max - kFixG128;
    __syncthreads();
    if (narrow) {
      Acc128 tot = {0ull, 0ull};
      for (int j = j0; j < j1; ++j) acc128_add(tot, to_fixed128(key_value(keys[j]), e_max));
      Acc128 run = block_excl_scan(tot, OpAcc128(), Acc128{0ull, 0ull},
                                   reinterpret_cast<Acc128 *>(sh_acc),
                                   static_cast<Acc128 *>(nullptr));
      for (int j = j0; j < j1; ++j) {
        acc128_add(run, to_fixed128(key_value(keys[j]), e_max));
        const double P = from_fixed128(run, e_max);
        Pd[j] = P;  // this thread's own element: no other thread reads it
        if (a.prefix_sum) a.prefix_sum[j + 1] = P;
      }
    } else {
      Acc256 tot = acc_zero();
      for (int j = j0; j < j1; ++j) acc_add(tot, to_fixed(key_value(keys[j]), e_max));
      Acc256 run = block_excl_scan(tot, OpAcc(), acc_zero(), sh_acc,
                                   static_cast<Acc256 *>(nullptr));
      for (int j = j0; j < j1; ++j) {
        acc_add(run, to_fixed(key_value(keys[j]), e_max));
        const double P = from_fixed(run, e_max);
        Pd[j] = P;  // this thread's own element: no other thread reads it
        if (a.prefix_sum) a.prefix_sum[j + 1] = P;
      }
    }
    if (tid == 0 && a.prefix_sum) a.prefix_sum[0] = 0.0;
    __syncthreads();
  } else if (stages & kStageBudget) {
    S = *a.n_eligible_in;
    n_s = *a.n_sampling_in;
    if (S < 0) S = 0;
    if (S > NK) S = NK;
  }

  // ---------------------------------------------------------------- budget
  if (stages & kStageBudget) {
    const int T = *a.T_dev;
    const int L = a.L;
    int B = 0;
    double objective = 0.0;
    if (T < 0 || T >= L) {
      st |= DSPARK_DEV_TABLE_SHORT;
    } else {
      const int b_max = min(S, L - 1 - T);
      const int nb = b_max + 1;
      const int C2 = (nb + NT - 1) / NT;
      const int b0 = min(nb, tid * C2), b1 = min(nb, b0 + C2);  // [b0, b1)
      const bool has_next = b1 < nb && b1 > b0;                // f(b1) too
      const float *cost = a.cost + T;
      const int mode = (a.flags & DSPARK_COST_FORCE_MONOTONE)   ? 1
                       : (a.flags & DSPARK_COST_FORCE_SUFFIX_MIN) ? 2
                                                                 : 0;
      float cf[kMaxChunk + 1];  // forced cost at b0 .. b1 (inclusive)
      const int cnt = (b1 - b0) + (has_next ? 1 : 0);
      if (mode == 1) {
        // one scan for both: the maximum of cost[0 .. T) (its total) and
        // the running maximum of the chunks before this thread's
        MaxPair v{-INFINITY, -INFINITY};
        for (int i = tid; i < T; i += NT) v.pre = fmax_nan(v.pre, a.cost[i]);
        for (int b = b0; b < b1; ++b) v.run = fmax_nan(v.run, cost[b]);
        MaxPair tot;
        const MaxPair ex = block_excl_scan(v, OpMaxPair(), MaxPair{-INFINITY, -INFINITY},
                                           sh_mp, &tot);
        float run = fmax_nan(ex.run, tot.pre);
        for (int i = 0; i < cnt; ++i) {
          run = fmax_nan(run, cost[b0 + i]);
          cf[i] = run;
        }
      } else if (mode == 2) {
        float post = INFINITY;
        for (int i = T + nb + tid; i < L; i += NT) post = OpMinNan()(post, a.cost[i]);
        post = block_reduce(post, OpMinNan(), INFINITY, sh_f);
        float loc = INFINITY;
        for (int b = b0; b < b1; ++b) loc = OpMinNan()(loc, cost[b]);
        float run = block_excl_scan_rev(loc, OpMinNan(), INFINITY, sh_f);
        run = OpMinNan()(run, post);  // min over cost[T+b1 ..]
        if (has_next) cf[cnt - 1] = run;  // forced value at b1
        for (int i = b1 - b0 - 1; i >= 0; --i) {
          run = OpMinNan()(run, cost[b0 + i]);
          cf[i] = run;
        }
      } else {
        for (int i = 0; i < cnt; ++i) cf[i] = cost[b0 + i];
      }
      const double dc = static_cast<double>(a.draft_cost);
      const double ns = static_cast<double>(n_s);
      // P_b of the chunk's points
      double Pl[kMaxChunk + 1];
      for (int i = 0; i < cnt; ++i) {
        const int b = b0 + i;
        Pl[i] = b == 0 ? 0.0 : (fused_order ? Pd[b - 1] : a.prefix_in[b]);
      }
      const bool greedy = (a.flags & DSPARK_BUDGET_GREEDY_STOP) != 0;
      // f(b) = fl(fl(N_s + P_b) / fl(cost'[T+b] + draft_cost)) in fp64.  The
      // fp64 divide is slow on this part, so the argmax first evaluates f in
      // fp32 (relative error < 3e-7) and divides in fp64 only where the fp32
      // value is within 1e-4 of the fp32 maximum: the fp64 maximiser, and
      // every b tied with it, is always among those.  Denominators that are
      // not normal positive fp32 numbers, or an fp32 overflow, send every b
      // through fp64 instead.
      float fa[kMaxChunk + 1];
      bool fast = !greedy;
      float amax = -INFINITY;
      for (int i = 0; i < cnt; ++i) {
        const float den32 = cf[i] + a.draft_cost;
        if (!(den32 > 0.0f)) st |= DSPARK_DEV_COST_NONPOS;
        const float num32 = f64_to_f32_rn(Pl[i]) + static_cast<float>(n_s);
        fa[i] = __fdiv_rn(num32, den32);
        fast = fast && den32 >= 1.17549435e-38f && isfinite(fa[i]);
        if (i < b1 - b0) amax = fmaxf(amax, fa[i]);
      }
      // one reduction for both: a thread that cannot take the fp32 filter
      // contributes NaN, which the maximum propagates to every thread
      amax = block_reduce(fast ? amax : NAN, OpMaxNan(), -INFINITY, sh_f);
      fast = !(amax != amax);
      const float thr = amax - amax * 1e-4f;
      unsigned long long best_k = 0ull;
      int best_b = INT_MAX;
      int gstop = INT_MAX;
      double gval = 0.0;
      double f_prev = 0.0;
      for (int i = 0; i < cnt; ++i) {
        const int b = b0 + i;
        if (fast && !(fa[i] >= thr)) continue;
        const double den = __dadd_rn(static_cast<double>(cf[i]), dc);
        const double f = __ddiv_rn(__dadd_rn(ns, Pl[i]), den);
        if (b < b1) {
          const unsigned long long k = f64_key(f);
          if (k > best_k || (k == best_k && b < best_b)) {
            best_k = k;
            best_b = b;
          }
        }
        if (greedy) {
          if (i > 0 && gstop == INT_MAX && !(f > f_prev)) {
            gstop = b - 1;
            gval = f_prev;
          }
          f_prev = f;
        }
      }
      if (greedy) {
        // the objective at b_max for "never stopped"
        if (b1 == nb && b1 > b0 && gstop == INT_MAX) {
          gstop = INT_MAX - 1;  // marker: reached the end
          gval = f_prev;
        }
        block_argmin_idx(gstop, gval, sh_int, sh_d);
        B = (gstop >= INT_MAX - 1) ? b_max : gstop;
        objective = gval;
      } else {
        block_argmax(best_k, best_b, sh_k, sh_int);
        B = best_b;
        objective = f64_from_key(best_k);
      }
    }
    if (tid == 0) {
      sh_B = B;
      if (a.B) *a.B = B;
      if (a.objective) *a.objective = objective;
    }
    __syncthreads();
  } else if (stages & kStageAllocate) {
    if (tid == 0) {
      int B = *a.B_in;
      sh_B = B < 0 ? 0 : (B > NK ? NK : B);
    }
    __syncthreads();
  }

  if (stale) {
    // the budget pass is done with keys (its prefix sums were written over
    // them): order the current confidences for the allocation
    __syncthreads();
    int n_s2 = 0;
    survival_order(a, a.conf, true, keys, sidx, stmp, sortbuf, sh_int, n_s2, st, -1);
    if (tid == 0) sh_B = min(sh_B, n_s2 * K);
    __syncthreads();
  }

  // -------------------------------------------------------------- allocate
  if (stages & kStageAllocate) {
    const int B = sh_B;
    for (int n = tid; n < N; n += NT) len_sm[n] = 0;
    __syncthreads();
    for (int j = tid; j < B; j += NT) {
      const int id = fused_order ? static_cast<int>(sidx[j]) : a.sorted_in[j];
      if (id >= 0 && id < NK) atomicAdd(&len_sm[id / K], 1);
    }
    __syncthreads();
    if (a.draft_len)
      for (int n = tid; n < N; n += NT) a.draft_len[n] = len_sm[n];
  }

  // --------------------------------------------------------------- compact
  if (stages & kStageCompact) {
    const bool from_sm = (stages & kStageAllocate) != 0;
    const int C3 = (N + NT - 1) / NT;
    const int n0 = min(N, tid * C3), n1 = min(N, n0 + C3);
    int loc = 0;
    for (int n = n0; n < n1; ++n) {
      int ln = from_sm ? len_sm[n] : a.len_in[n];
      ln = ln < 0 ? 0 : (ln > K ? K : ln);
      loc += ln;
    }
    int total = 0;
    int off = block_excl_scan(loc, OpAddInt(), 0, sh_int, &total);
    for (int n = n0; n < n1; ++n) {
      int ln = from_sm ? len_sm[n] : a.len_in[n];
      ln = ln < 0 ? 0 : (ln > K ? K : ln);
      if (a.cu_len) a.cu_len[n] = off;
      for (int k = 0; k < ln; ++k) {
        const int idx = n * K + k;
        if (a.verify_idx) a.verify_idx[off + k] = idx;
        if (a.verify_tok && a.draft) a.verify_tok[off + k] = a.draft[idx];
      }
      off += ln;
    }
    if (tid == 0 && a.cu_len) a.cu_len[N] = total;
  }

  if (st) raise_status(a.status, st);
}

// forced cost table, one CTA: running max from the left or min from the right
__global__ void __launch_bounds__(SEL_THREADS, 1)
    force_monotone_kernel(const float *in, float *out, const int L,
                          const uint32_t mode) {
  __shared__ float sh_f[SEL_WARPS + 1];
  const int tid = threadIdx.x, NT = blockDim.x;
  const int C = (L + NT - 1) / NT;
  const int i0 = min(L, tid * C), i1 = min(L, i0 + C);
  if (mode == DSPARK_COST_FORCE_MONOTONE) {
    float loc = -INFINITY;
    for (int i = i0; i < i1; ++i) loc = fmax_nan(loc, in[i]);
    float run = block_excl_scan(loc, OpMaxNan(), -INFINITY, sh_f,
                                static_cast<float *>(nullptr));
    for (int i = i0; i < i1; ++i) {
      run = fmax_nan(run, in[i]);
      out[i] = run;
    }
  } else {
    float loc = INFINITY;
    for (int i = i0; i < i1; ++i) loc = OpMinNan()(loc, in[i]);
    float run = block_excl_scan_rev(loc, OpMinNan(), INFINITY, sh_f);
    for (int i = i1 - 1; i >= i0; --i) {
      run = OpMinNan()(run, in[i]);
      out[i] = run;
    }
  }
}

// verify_tok[j] = draft[verify_idx[j]] for j < *B (after the chain has
// finished, when the scheduler ran alongside it without the draft)
__global__ void __launch_bounds__(256)
    gather_verify_kernel(const int32_t *verify_idx, const int32_t *B_dev,
                         const int32_t *draft, const int NK,
                         int32_t *verify_tok) {
  int B = *B_dev;
  B = B < 0 ? 0 : (B > NK ? NK : B);
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < B;
       j += gridDim.x * blockDim.x) {
    const int idx = verify_idx[j];
    verify_tok[j] = (idx >= 0 && idx < NK) ? draft[idx] : 0;
  }
}

// ==========================================================================
// host side
// ==========================================================================
static std::mutex g_sel_mu;
static bool g_sel_attr[128];

dspark_status select_launch(const SelectArgs &a, uint32_t stages,
                            cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return DSPARK_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_sel_mu);
    if (!g_sel_attr[dev]) {
      if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      g_sel_attr[dev] = true;
    }
  }
  const int NK = a.N * a.K;
  int cap = 0;
  size_t dyn = 0;
  if (stages & kStageSurvival) {
    cap = NK;  // keys by slot, then in order; two 16-bit slot arrays
    dyn = static_cast<size_t>(cap + 1) * 8 + static_cast<size_t>(cap) * 4;
    if (NK <= kFastMaxNK)  // two composite arrays
      dyn = ((dyn + 7) & ~static_cast<size_t>(7)) + static_cast<size_t>(NK) * 16;
  }
  if (stages & kStageAllocate) {
    const size_t need = static_cast<size_t>(a.N) * 4;
    if (need > dyn) dyn = need;
  }
  dyn = (dyn + 15) & ~static_cast<size_t>(15);
  select_kernel<<<1, SEL_THREADS, dyn, stream>>>(a, stages, cap);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status gather_verify_launch(const int32_t *verify_idx,
                                   const int32_t *B_dev, const int32_t *draft,
                                   int32_t NK, int32_t *verify_tok,
                                   cudaStream_t stream) {
  const int blocks = (NK + 255) / 256 < 8 ? (NK + 255) / 256 : 8;
  gather_verify_kernel<<<blocks, 256, 0, stream>>>(verify_idx, B_dev, draft, NK,
                                                   verify_tok);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status force_monotone_launch(const float *in, float *out, int32_t L,
                                    uint32_t mode, cudaStream_t stream) {
  force_monotone_kernel<<<1, SEL_THREADS, 0, stream>>>(in, out, L, mode);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
