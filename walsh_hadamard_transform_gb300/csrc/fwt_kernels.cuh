// Pass kernels of the batched Walsh-Hadamard transform (sm_103a).
//
// One launch = one pass over every vector of the batch: a full HBM read and write
// of the data.  A pass transforms a contiguous group of index bits of each 2^n
// vector with the on-chip tile engine:
//
//   row tiles:    bits [0, K) of each vector; a tile is 2^TB contiguous elements
//                 (one vector, one row of the Kronecker split, or several short
//                 vectors).  This is the whole transform when n fits a tile, and
//                 the I (x) H_b factor of the Kronecker split otherwise.
//   column tiles: bits [L, L + K) of each vector; a tile is 2^K rows spaced 2^L
//                 elements apart, times one 16- to 128-byte segment of contiguous
//                 columns.  This is the H_a (x) I factor of the Kronecker split
//                 ("[QDP] [feature] Pr4 kronecker fwt", section "Why submit PR4",
//                 deliverables: Y = (H_{n1} (x) I)(I (x) H_{n2}) X; iThome "Day
//                 18" FWT post, section "Kronecker block GEMM idea": Z = X H_b,
//                 Y = H_a Z).  The strided tile is read and written in place, so
//                 the transpose between the two factors happens in the loads and
//                 stores and never as a separate pass or a temporary buffer.
//
// fp64 runs its butterflies exactly in 64-bit fixed point on the integer units
// (GB300's fp64 add rate is about 1/64 of its fp32 rate, while 64-bit integer
// adds run near the fp32 rate): the tile's largest binary exponent sets a common
// scale, every element is converted to an int64 with min(61 - K, 51) fraction bits (integer
// bit arithmetic), the K stages run exactly, and each result is rounded once back
// to fp64 (the hardware int64 -> fp64 conversion, round to nearest even, then an
// exponent-field add; an all-integer exact rounding where results could be
// subnormal or overflow).  A tile holding an Inf or NaN takes a plain fp64 path.
//
// Tiles are staged three ways: 16-byte vector loads and stores (DirectMover),
// untiled bulk copies of whole contiguous tiles (BulkMover, fp64 row tiles), and
// TMA 2-D tensor copies of strided column tiles (TmaMover); the staged kernels run
// three CTAs an SM at 80 registers a thread.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

#include "tile_engine.cuh"
#include "tma.cuh"

namespace fwt {

struct PassParams {
  const void* in[2];
  void* out[2];
  long long comp_elems;  // elements per array (batch * 2^n)
  int stride_log;        // column tiles: log2 of the row stride L; row tiles: 0
  int do_scale;          // apply the normalisation in this pass
  float scale_f32;       // 2^{-n/2} rounded to fp32
  double scale_f64;      // 2^{-n/2} in fp64
  int scale_exp;         // fixed point: floor(-n/2) as a binary exponent
  int scale_half;        // fixed point: n odd, also divide by sqrt(2)
  unsigned long long rsqrt2_q64;  // floor(2^64 / sqrt(2))
  int ld_policy;         // L2 eviction priority of the loads: 0 normal, 1 first, 2 last
  int st_policy;         // ... and of the stores
  int bits_lo, bits_k;   // run-time bit-range tiles: transformed tile bits [lo, lo + k)
  uint32_t bits_mask;    // ... or, when non-zero, this set of tile bits
  int prefetch_ahead;    // staged tiles: also prefetch into L2 the tile this many ahead (0: off)
  const float* theta;    // phase pass: angles, theta[b * theta_stride + i]
  long long theta_stride;
  int n;                 // phase pass: log2 of the vector length
  int bulk;              // row tiles: stage whole tiles with bulk copies where eligible
};

// ---- arithmetic policies ----------------------------------------------------------
struct ArithF32 {
  static constexpr bool kRadix4 = false;
  __device__ static float add(float a, float b) { return a + b; }
  __device__ static float sub(float a, float b) { return a - b; }
};
struct ArithF64 {
  static constexpr bool kRadix4 = false;
  __device__ static double add(double a, double b) { return a + b; }
  __device__ static double sub(double a, double b) { return a - b; }
};
// Integer policies: wrap-around arithmetic in unsigned types, with the three-operand
// forms used by the two-stage butterflies.  The int32 passes are bound by HBM, not by
// issue, and measured no faster at radix 4 (one short column pass slower), so only
// the 64-bit fixed-point arithmetic takes it.
template <typename U, typename W, bool RADIX4>
struct ArithInt {
  static constexpr bool kRadix4 = RADIX4;
  __device__ static U add(U a, U b) { return (U)((W)a + (W)b); }
  __device__ static U sub(U a, U b) { return (U)((W)a - (W)b); }
  __device__ static U add3(U a, U b, U c) { return (U)((W)a + (W)b + (W)c); }
  __device__ static U add_sub(U a, U b, U c) { return (U)((W)a + (W)b - (W)c); }
  __device__ static U sub2(U a, U b, U c) { return (U)((W)a - (W)b - (W)c); }
  __device__ static U sub_add(U a, U b, U c) { return (U)((W)a - (W)b + (W)c); }
};
using ArithU32 = ArithInt<uint32_t, uint32_t, false>;  // two's complement wrap, bit-exact
// fixed point: magnitudes stay below 2^62 by construction; no wrap occurs
using ArithI64 = ArithInt<long long, unsigned long long, true>;

// ---- global memory access -------------------------------------------------------
// Every load and store carries an L2 eviction-priority policy chosen per pass: loads
// are normal priority (reading with evict-first made the in-place column passes,
// which write back the lines they read, 1-7% slower), an intermediate that the next
// pass reads back from L2 is kept (evict last, chunked schedules), and the final
// result streams out (evict first).
__device__ __forceinline__ unsigned long long l2_policy(int kind) {
  unsigned long long pol;
  if (kind == 1) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else if (kind == 2) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
template <typename U>
__device__ __forceinline__ typename Vec16<U>::type ldg16(const void* p, unsigned long long pol) {
  using V = typename Vec16<U>::type;
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return *reinterpret_cast<V*>(&v);
}
template <typename U>
__device__ __forceinline__ void stg16(void* p, const typename Vec16<U>::type& val,
                                      unsigned long long pol) {
  const uint4 v = *reinterpret_cast<const uint4*>(&val);
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// Tile-local index -> element offset within the array.
template <class S, bool COLS, bool RAGGED = (!COLS && S::TB > S::TK)>
struct TileMap {
  long long base;
  int L;
  long long valid;  // row tiles: elements of this tile inside the array
  __device__ __forceinline__ long long off(uint32_t u) const {
    if constexpr (!COLS) {
      return base + (long long)u;
    } else {
      constexpr int CWL = S::TS;  // column bits sit below the transformed rows
      return base + ((long long)(u >> CWL) << L) + (long long)(u & ((1u << CWL) - 1u));
    }
  }
  __device__ __forceinline__ bool in_range(uint32_t u) const {
    if constexpr (RAGGED) return (long long)u < valid;  // ragged last tile
    else return true;
  }
  __device__ static TileMap make(const PassParams& p, long long tile) {
    TileMap m;
    m.L = p.stride_log;
    if constexpr (!COLS) {
      m.base = tile << S::TB;
      m.valid = p.comp_elems - m.base;
    } else {
      const int chunks_lg = p.stride_log - S::TS;
      const long long cc = tile & ((1ll << chunks_lg) - 1);
      const long long hb = tile >> chunks_lg;
      m.base = (hb << (p.stride_log + S::TK)) + (cc << S::TS);
      m.valid = 0;
    }
    return m;
  }
};

template <class S, class Map, typename T, typename U>
__device__ __forceinline__ void load_tile(const T* in, const Map& m, U (&x)[S::NE], int policy) {
  using V = typename Vec16<U>::type;
  const uint32_t t = threadIdx.x;
  const unsigned long long pol = l2_policy(policy);
#pragma unroll
  for (int j = 0; j < S::NV; ++j) {
    const uint32_t u = S::idx1(t, j * S::VEC);
    V v;
    if (m.in_range(u)) v = ldg16<U>(in + m.off(u), pol);
    else v = V{};
    const U* pv = reinterpret_cast<const U*>(&v);
#pragma unroll
    for (int i = 0; i < S::VEC; ++i) x[j * S::VEC + i] = pv[i];
  }
}

template <class S, class Map, typename T, typename U>
__device__ __forceinline__ void store_tile(T* out, const Map& m, const U (&x)[S::NE], int policy) {
  using V = typename Vec16<U>::type;
  const uint32_t t = threadIdx.x;
  const unsigned long long pol = l2_policy(policy);
#pragma unroll
  for (int j = 0; j < S::NV; ++j) {
    const uint32_t u = S::idx3(t, j * S::VEC);
    V v;
    U* pv = reinterpret_cast<U*>(&v);
#pragma unroll
    for (int i = 0; i < S::VEC; ++i) pv[i] = x[j * S::VEC + i];
    if (m.in_range(u)) stg16<U>(out + m.off(u), v, pol);
  }
}

// ---- tile movers: HBM <-> registers ----------------------------------------------
// Direct: 16-byte vector loads into layout L1, stores from layout L3.
template <class S, bool COLS, bool RAGGED = (!COLS && S::TB > S::TK)>
struct DirectMover {
  using Map = TileMap<S, COLS, RAGGED>;
  Map m;
  const void* in;
  void* out;
  __device__ DirectMover(const PassParams& p, unsigned char*) {
    const bool im = blockIdx.y != 0;
    in = im ? p.in[1] : p.in[0];
    out = im ? p.out[1] : p.out[0];
    m = Map::make(p, (long long)blockIdx.x);
  }
  template <typename U>
  __device__ __forceinline__ bool load(U (&x)[S::NE], int policy) {
    load_tile<S>(static_cast<const U*>(in), m, x, policy);
    return true;
  }
  template <typename U>
  __device__ __forceinline__ void store(const U (&x)[S::NE], int policy) {
    store_tile<S>(static_cast<U*>(out), m, x, policy);
  }
};

// Parameters of a TMA column pass: one tensor map per part (rows of 2^L
// elements, box of CW columns x up to 256 rows), then the common parameters.
struct TmaPassParams {
  CUtensorMap map[2];
  PassParams p;
};

// Waits (bounded) for a staged tile on its mbarrier, as a CTA-wide decision.  On
// give-up every thread learns it, and the copies still in flight get one more
// bounded wait so the CTA does not leave while they may still write its shared
// memory.
__device__ __forceinline__ bool wait_tile(uint64_t* bar) {
  const bool ok = mbar_wait_bounded(bar, 0);
  if (!__syncthreads_or(!ok)) return true;
  if (threadIdx.x == 0) mbar_wait_bounded(bar, 0);
  __syncthreads();
  return false;
}

// TMA: the column tile arrives in shared memory in natural order; threads pick up
// layout L1 there, and write layout L3 back there for a TMA store.
template <class S, int ESZ>
struct TmaMover {
  // L2 prefetch of a later tile: segments of 128+ bytes, and fp64 64-byte segments (at
  // half the distance; measured 5% faster: fp64 n = 22 column pass 1.61 -> 1.53 ms).  fp32
  // 64-byte and all 32-byte segments measured slower with it at any distance.
  static constexpr bool kPrefetch = (ESZ << S::TS) >= 128 || (ESZ == 8 && (ESZ << S::TS) == 64);
  static constexpr int kPrefetchDiv = (ESZ << S::TS) >= 128 ? 1 : 2;
  static constexpr int BOXR = S::TK >= 8 ? 256 : (1 << S::TK);  // rows per copy
  static constexpr int NBOX = (1 << S::TK) / BOXR;
  static constexpr uint32_t BOX_ELEMS = (uint32_t)BOXR << S::TS;
  const CUtensorMap* map;
  int col0, row0;
  int pf_col = -1, pf_row = 0;  // tile to prefetch into L2 (none: pf_col < 0)
  unsigned char* smem;
  uint64_t* bar;
  __device__ TmaMover(const TmaPassParams& tp, unsigned char* smem_raw, uint64_t* barrier) {
    const bool im = blockIdx.y != 0;
    map = im ? &tp.map[1] : &tp.map[0];
    const int chunks_lg = tp.p.stride_log - S::TS;
    const long long tile = blockIdx.x;
    col0 = (int)((tile & ((1ll << chunks_lg) - 1)) << S::TS);
    row0 = (int)((tile >> chunks_lg) << S::TK);
    // Wide segments (128 bytes and more) prefetch into L2 the tile prefetch_ahead
    // tiles on (two an SM: it starts while this one runs; measured 5% faster), fp64
    // 64-byte segments the tile half as far on.
    const int ahead = tp.p.prefetch_ahead / kPrefetchDiv;
    const long long next = tile + ahead;
    if (kPrefetch && ahead > 0 && next < (long long)gridDim.x) {
      pf_col = (int)((next & ((1ll << chunks_lg) - 1)) << S::TS);
      pf_row = (int)((next >> chunks_lg) << S::TK);
    }
    smem = smem_raw;
    bar = barrier;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
  }
  template <typename U>
  __device__ __forceinline__ bool load(U (&x)[S::NE], int policy) {
    if (threadIdx.x == 0) {
      const unsigned long long pol = l2_policy(policy);
      mbar_arrive_expect_tx(bar, (uint32_t)(sizeof(U) << S::TB));
#pragma unroll
      for (int i = 0; i < NBOX; ++i)
        tma_load_2d(smem + (size_t)i * BOX_ELEMS * sizeof(U), map, col0, row0 + i * BOXR, bar, pol);
      if (pf_col >= 0) {
#pragma unroll
        for (int i = 0; i < NBOX; ++i) tma_prefetch_2d(map, pf_col, pf_row + i * BOXR);
      }
    }
    if (!wait_tile(bar)) return false;  // the whole tile is skipped
    const U* sm = reinterpret_cast<const U*>(smem);
#pragma unroll
    for (int j = 0; j < S::NV; ++j) get_vec<U, S::VEC>(sm + S::idx1(threadIdx.x, j * S::VEC), x, j);
    __syncthreads();  // the tile engine reuses the buffer
    return true;
  }
  template <typename U>
  __device__ __forceinline__ void store(const U (&x)[S::NE], int policy) {
    U* sm = reinterpret_cast<U*>(smem);
    __syncthreads();  // the engine's last reads of the buffer are done
#pragma unroll
    for (int j = 0; j < S::NV; ++j) put_vec<U, S::VEC>(sm + S::idx3(threadIdx.x, j * S::VEC), x, j);
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned long long pol = l2_policy(policy);
#pragma unroll
      for (int i = 0; i < NBOX; ++i)
        tma_store_2d(map, col0, row0 + i * BOXR, smem + (size_t)i * BOX_ELEMS * sizeof(U), pol);
      tma_store_commit_and_wait();
    }
  }
};

// Bulk: a contiguous row tile (2^TB elements, never ragged) arrives in shared
// memory in natural order through untiled bulk copies (16 KiB each) that complete
// on one mbarrier; threads pick up layout L1 there and write layout L3 back for
// bulk stores.  The loads bypass L1 and the registers, like the TMA column tiles.
template <class S>
struct BulkMover {
  const char* src;
  char* dst;
  int prefetch;  // tiles ahead to prefetch into L2 (0: none)
  unsigned char* smem;
  uint64_t* bar;
  __device__ BulkMover(const PassParams& p, unsigned char* smem_raw, uint64_t* barrier) {
    const bool im = blockIdx.y != 0;
    // prefetch into L2 the tile prefetch_ahead tiles on (two an SM, so it starts
    // while this one runs; measured 3-5% faster)
    prefetch = p.prefetch_ahead > 0 && (long long)blockIdx.x + p.prefetch_ahead < (long long)gridDim.x
                   ? p.prefetch_ahead
                   : 0;
    src = static_cast<const char*>(im ? p.in[1] : p.in[0]);
    dst = static_cast<char*>(im ? p.out[1] : p.out[0]);
    smem = smem_raw;
    bar = barrier;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
  }
  template <typename U>
  __device__ __forceinline__ bool load(U (&x)[S::NE], int policy) {
    constexpr uint32_t BYTES = (uint32_t)sizeof(U) << S::TB;
    constexpr uint32_t CH = BYTES < 16384u ? BYTES : 16384u;
    if (threadIdx.x == 0) {
      const unsigned long long pol = l2_policy(policy);
      const char* g = src + (size_t)blockIdx.x * BYTES;
      mbar_arrive_expect_tx(bar, BYTES);
#pragma unroll
      for (uint32_t o = 0; o < BYTES; o += CH) bulk_load(smem + o, g + o, CH, bar, pol);
      if (prefetch) {
        const char* nxt = g + (size_t)prefetch * BYTES;
#pragma unroll
        for (uint32_t o = 0; o < BYTES; o += CH) bulk_prefetch(nxt + o, CH);
      }
    }
    if (!wait_tile(bar)) return false;  // the whole tile is skipped
    const U* sm = reinterpret_cast<const U*>(smem);
#pragma unroll
    for (int j = 0; j < S::NV; ++j) get_vec<U, S::VEC>(sm + S::idx1(threadIdx.x, j * S::VEC), x, j);
    __syncthreads();  // the tile engine reuses the buffer
    return true;
  }
  template <typename U>
  __device__ __forceinline__ void store(const U (&x)[S::NE], int policy) {
    constexpr uint32_t BYTES = (uint32_t)sizeof(U) << S::TB;
    constexpr uint32_t CH = BYTES < 16384u ? BYTES : 16384u;
    U* sm = reinterpret_cast<U*>(smem);
    __syncthreads();  // the engine's last reads of the buffer are done
#pragma unroll
    for (int j = 0; j < S::NV; ++j) put_vec<U, S::VEC>(sm + S::idx3(threadIdx.x, j * S::VEC), x, j);
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned long long pol = l2_policy(policy);
      char* g = dst + (size_t)blockIdx.x * BYTES;
#pragma unroll
      for (uint32_t o = 0; o < BYTES; o += CH) bulk_store(g + o, smem + o, CH, pol);
      tma_store_commit_and_wait();
    }
  }
};

// Which tile bits a pass transforms: fixed by the shape, or given at run time.
template <class S>
struct StaticBits {
  static constexpr uint32_t r1 = S::RM1, r2 = S::RM2, r3 = S::RM3;
  static constexpr int tk = S::TK;
  static constexpr bool kMayTruncate = S::TK <= 13;  // transformed bits known at compile time
  __device__ explicit StaticBits(const PassParams&) {}
};
template <class S>
struct RuntimeBits {
  uint32_t r1, r2, r3;
  int tk;
  static constexpr bool kMayTruncate = true;  // decided at run time from tk
  __device__ explicit RuntimeBits(const PassParams& p) {
    uint32_t rm[3];
    if (p.bits_mask) S::round_masks_set(p.bits_mask, rm);
    else S::round_masks(p.bits_lo, p.bits_k, rm);
    r1 = rm[0];
    r2 = rm[1];
    r3 = rm[2];
    tk = p.bits_mask ? __popc(p.bits_mask) : p.bits_k;
  }
};

// ---- fp32 / int32 / plain fp64 tile ---------------------------------------------
template <class S, class A, typename T, class Mover, class Bits>
__device__ __forceinline__ void plain_tile(const PassParams& p, unsigned char* smem_raw, Mover& mv,
                                           const Bits& bits) {
  T x[S::NE];
  if (!mv.load(x, p.ld_policy)) return;
  tile_rounds<S, A>(x, reinterpret_cast<T*>(smem_raw), bits.r1, bits.r2, bits.r3);
  if (p.do_scale) {
    if constexpr (sizeof(T) == 4 && !std::is_integral<T>::value) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = x[r] * p.scale_f32;
    } else if constexpr (sizeof(T) == 8) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = x[r] * p.scale_f64;
    }
  }
  mv.store(x, p.st_policy);
}

// ---- fp64 in exact 64-bit fixed point -------------------------------------------
// Tile-wide exponent scan: the largest high word without its sign bit carries the
// largest biased exponent, and is >= 0x7ff00000 exactly when an Inf or NaN is
// present.
__device__ __forceinline__ uint32_t abs_hi(long long bits) {
  return (uint32_t)((unsigned long long)bits >> 32) & 0x7fffffffu;
}

// 64-bit logical right shift with the PTX rule that amounts of 64 or more give 0.
__device__ __forceinline__ unsigned long long shr64(unsigned long long v, uint32_t s) {
  unsigned long long r;
  asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"(v), "r"(s));
  return r;
}

// q = v * 2^(F + 1023 - emax) as an integer, for |v| < 2^(emax - 1022): |q| <= 2^(F+1).
// Integer bit arithmetic only.  Modes:
//   TO_FIXED_ANY:   any F (shifts either way), rounded half away from zero.
//   TO_FIXED_ROUND: F <= 51, so every element shifts right by at least one bit;
//                   rounded half away from zero (the rounding folded into the shift).
//   TO_FIXED_TRUNC: F <= 51 and emax >= F + 12, so a zero or subnormal element would
//                   shift right by 64 bits or more whatever its leading bit: every
//                   element is taken as a normal number, and the magnitude is
//                   truncated (error below one unit instead of half a unit, and of
//                   either sign, so the errors of a tile carry no common bias).
enum ToFixedMode { TO_FIXED_ANY, TO_FIXED_ROUND, TO_FIXED_TRUNC };
template <int MODE>
__device__ __forceinline__ long long to_fixed(long long bits, int emax, int F) {
  const unsigned long long b = (unsigned long long)bits;
  const int e = (int)((uint32_t)(b >> 32) >> 20) & 0x7ff;
  unsigned long long mag;
  if constexpr (MODE == TO_FIXED_TRUNC) {
    const unsigned long long m = (b & 0x000fffffffffffffull) | (1ull << 52);
    mag = shr64(m, (uint32_t)(emax - e + 52 - F));  // >= 1
  } else {
    const unsigned long long m =
        (b & 0x000fffffffffffffull) | ((unsigned long long)(e != 0) << 52);
    // v = m * 2^(max(e,1) - 1075), so q = m * 2^(max(e,1) - emax + F - 52)
    const int sh = max(e, 1) - emax + F - 52;
    if constexpr (MODE == TO_FIXED_ROUND) {  // sh <= -1: shift by -sh - 1, add the half, halve
      mag = (shr64(m, (uint32_t)(-sh - 1)) + 1ull) >> 1;
    } else {  // either way, without a divergent branch: (sh >= 0: rs = 0, exact)
      const int rs = min(max(-sh, 0), 63);
      mag = ((((m << 1) >> rs) + 1ull) >> 1) << max(sh, 0);
    }
  }
  const unsigned long long neg = (unsigned long long)((long long)b >> 63);  // 0 or ~0
  return (long long)((mag ^ neg) - neg);
}

// Exact rounding of q * 2^e0 (optionally also / sqrt 2) to the nearest fp64, ties
// to even, including subnormal results and overflow to Inf.
__device__ __forceinline__ long long from_fixed_exact(long long q, int e0, int half,
                                                      unsigned long long rsqrt2) {
  const unsigned long long sign = (unsigned long long)q & 0x8000000000000000ull;
  unsigned long long a = q < 0 ? (unsigned long long)(-q) : (unsigned long long)q;
  if (half) a = __umul64hi(a, rsqrt2);  // a / sqrt(2), truncated (error < 1 unit)
  if (a == 0) return 0;
  const int top = 63 - __clzll((long long)a);
  int be = top + e0 + 1023;  // biased exponent of the result
  if (be >= 1) {
    unsigned long long mant;
    if (top <= 52) {
      mant = a << (52 - top);
    } else {
      const int rs = top - 52;
      mant = a >> rs;
      const unsigned long long rem = a & ((1ull << rs) - 1ull);
      const unsigned long long halfulp = 1ull << (rs - 1);
      mant += (rem > halfulp) || (rem == halfulp && (mant & 1ull));
      if (mant >> 53) { mant >>= 1; ++be; }
    }
    if (be >= 2047) return (long long)(sign | 0x7ff0000000000000ull);  // overflow -> Inf
    return (long long)(sign | ((unsigned long long)be << 52) | (mant & 0x000fffffffffffffull));
  }
  // subnormal result, in units of 2^-1074
  const int rs = -(e0 + 1074);
  if (rs <= 0) return (long long)(sign | (a << (-rs)));  // exact: fits in 52 bits when be < 1
  if (rs >= 64) {
    const bool up = rs == 64 && a > 0x8000000000000000ull;
    return (long long)(sign | (up ? 1ull : 0ull));
  }
  unsigned long long t = a >> rs;
  const unsigned long long rem = a & ((1ull << rs) - 1ull);
  const unsigned long long halfulp = 1ull << (rs - 1);
  t += (rem > halfulp) || (rem == halfulp && (t & 1ull));
  return (long long)(sign | t);
}

// The same rounding through the hardware int64 -> fp64 conversion (round to
// nearest even; it runs on the fp64 unit, beside the integer pipes), followed by an
// exact power-of-two rescale done as an add to the exponent field.  Valid when
// every nonzero result is a normal number: -1022 <= e0 <= 960 (|q| < 2^63).
// e0_field = e0 << 52.  HALF also divides by sqrt(2) first (a compile-time choice,
// so the unrolled per-element code carries no predicated-off multiply).
template <bool HALF>
__device__ __forceinline__ long long from_fixed_cvt(long long q, long long e0_field,
                                                    unsigned long long rsqrt2) {
  if constexpr (HALF) {
    const unsigned long long neg = (unsigned long long)(q >> 63);
    const unsigned long long a = __umul64hi(((unsigned long long)q ^ neg) - neg, rsqrt2);
    q = (long long)((a ^ neg) - neg);
  }
  const long long b = __double_as_longlong(__ll2double_rn(q));
  // the exponent field sits in the high word, which is zero exactly when q == 0
  const uint32_t hi = (uint32_t)((unsigned long long)b >> 32);
  const uint32_t hi_scaled = hi == 0u ? 0u : hi + (uint32_t)((unsigned long long)e0_field >> 32);
  return (long long)(((unsigned long long)hi_scaled << 32) | (uint32_t)b);
}

template <class S, class Mover, class Bits>
__device__ __forceinline__ void fixed_tile(const PassParams& p, unsigned char* smem_raw, Mover& mv,
                                           const Bits& bits) {
  __shared__ uint32_t red[32];
  long long x[S::NE];
  if (!mv.load(x, p.ld_policy)) return;
  // tile-wide largest exponent (and whether any Inf/NaN is present)
  uint32_t key = 0;
#pragma unroll
  for (int r = 0; r < S::NE; ++r) key = max(key, abs_hi(x[r]));
  key = __reduce_max_sync(0xffffffffu, key);
  if ((threadIdx.x & 31u) == 0) red[threadIdx.x >> 5] = key;
  __syncthreads();
  key = red[0];
#pragma unroll
  for (int w = 1; w < S::NT / 32; ++w) key = max(key, red[w]);
  if (key >= 0x7ff00000u) {  // rare: a tile with Inf/NaN takes plain IEEE fp64 adds
    double xd[S::NE];
#pragma unroll
    for (int r = 0; r < S::NE; ++r) xd[r] = __longlong_as_double(x[r]);
    tile_rounds<S, ArithF64>(xd, reinterpret_cast<double*>(smem_raw), bits.r1, bits.r2,
                             bits.r3);
    if (p.do_scale) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) xd[r] = xd[r] * p.scale_f64;
    }
    mv.store(xd, p.st_policy);
    return;
  }
  const int emax = max((int)(key >> 20), 1);  // zeros and subnormals scale as exponent 1
  // Fraction bits: headroom for the growth (|q| <= 2^(F+1) grows by 2^tk), at most 51 so
  // that every element shifts right and passes over few bits take the truncating
  // conversion too (their error bound sqrt(T) 2^-51 stays far below the specification;
  // measured 7-16% faster for factors of 4 to 9 bits than 61 - tk with the general form).
  const int F = min(61 - bits.tk, 51);
  // (uniform branches) Tiles of up to 2^13 transformed elements truncate: their error
  // bound sqrt(T) 2^-F stays far below the fp64 specification; tiles of 2^14 round.
  bool converted = false;
  if constexpr (Bits::kMayTruncate) {
    if (bits.tk <= 13 && F <= 51 && emax >= F + 12) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = to_fixed<TO_FIXED_TRUNC>(x[r], emax, F);
      converted = true;
    }
  }
  if (!converted) {
    if (F <= 51) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = to_fixed<TO_FIXED_ROUND>(x[r], emax, F);
    } else {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = to_fixed<TO_FIXED_ANY>(x[r], emax, F);
    }
  }
  tile_rounds<S, ArithI64>(x, reinterpret_cast<long long*>(smem_raw), bits.r1, bits.r2,
                           bits.r3);
  const int e0 = emax - 1023 - F + (p.do_scale ? p.scale_exp : 0);
  const int half = p.do_scale ? p.scale_half : 0;
  // every nonzero |q| lies in [1, 2^63): results are normal numbers iff
  // 1 <= e0 + 1023 and e0 + 1023 + 63 <= 2046 (uniform over the tile)
  if (e0 >= -1022 && e0 <= 960) {
    const long long e0_field = (long long)((unsigned long long)(long long)e0 << 52);
    if (half) {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = from_fixed_cvt<true>(x[r], e0_field, p.rsqrt2_q64);
    } else {
#pragma unroll
      for (int r = 0; r < S::NE; ++r) x[r] = from_fixed_cvt<false>(x[r], e0_field, p.rsqrt2_q64);
    }
  } else {  // rare: a rolled loop over a local copy keeps this code small
    long long xl[S::NE];
#pragma unroll
    for (int r = 0; r < S::NE; ++r) xl[r] = x[r];
#pragma unroll 1
    for (int r = 0; r < S::NE; ++r) xl[r] = from_fixed_exact(xl[r], e0, half, p.rsqrt2_q64);
#pragma unroll
    for (int r = 0; r < S::NE; ++r) x[r] = xl[r];
  }
  mv.store(x, p.st_policy);
}

// ---- kernels --------------------------------------------------------------------
// KIND: 0 = fp32, 1 = fp64 (fixed point), 2 = int32, 3 = fp64 plain IEEE
// At most 128 registers a thread, so that 512 threads (16 warps) fit an SM
// whatever the tile size.
template <class S, int KIND, class Mover, class Bits>
__device__ __forceinline__ void tile_body(const PassParams& p, unsigned char* smem_raw, Mover& mv,
                                          const Bits& bits) {
  if constexpr (KIND == 0) plain_tile<S, ArithF32, float>(p, smem_raw, mv, bits);
  else if constexpr (KIND == 1) fixed_tile<S>(p, smem_raw, mv, bits);
  else if constexpr (KIND == 2) plain_tile<S, ArithU32, uint32_t>(p, smem_raw, mv, bits);
  else plain_tile<S, ArithF64, double>(p, smem_raw, mv, bits);
}

template <class S, int KIND, bool COLS>
__global__ void __launch_bounds__(S::NT, (S::NT < 512 ? 512 / S::NT : 1)) fwt_tile_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  DirectMover<S, COLS> mv(p, smem_raw);
  tile_body<S, KIND>(p, smem_raw, mv, StaticBits<S>(p));
}

// Row pass with bulk-copied tiles (fp64 fixed point: 3 CTAs an SM, as the TMA column
// pass; whole tiles only).
template <class S, int KIND>
__global__ void __launch_bounds__(S::NT, KIND == 1 ? (S::NT < 768 ? 768 / S::NT : 1)
                                                   : (S::NT < 512 ? 512 / S::NT : 1))
    fwt_row_bulk_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  BulkMover<S> mv(p, smem_raw, &bar);
  tile_body<S, KIND>(p, smem_raw, mv, StaticBits<S>(p));
}

// The same over bulk-copied whole tiles (fp64 fixed point: three CTAs an SM).
template <class S, int KIND>
__global__ void __launch_bounds__(S::NT, KIND == 1 ? (S::NT < 768 ? 768 / S::NT : 1)
                                                   : (S::NT < 512 ? 512 / S::NT : 1))
    fwt_rowbits_bulk_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  BulkMover<S> mv(p, smem_raw, &bar);
  tile_body<S, KIND>(p, smem_raw, mv, RuntimeBits<S>(p));
}

// Contiguous tiles of 2^TB elements whose transformed bits [bits_lo, bits_lo +
// bits_k) are chosen at run time: a transform on a sub-range of the index bits
// that lies within the low TB bits (several vectors per tile when 2^n < 2^TB).
template <class S, int KIND>
__global__ void __launch_bounds__(S::NT, (S::NT < 512 ? 512 / S::NT : 1))
    fwt_rowbits_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  DirectMover<S, false, true> mv(p, smem_raw);
  tile_body<S, KIND>(p, smem_raw, mv, RuntimeBits<S>(p));
}

// Column pass with TMA-staged tiles.  The loads do not go through L1, so the kernel
// can trade registers (80 a thread, a few spilled to L1) for a third resident CTA
// per SM: 24 warps instead of 16 hide more of the TMA and integer latencies.  Taken
// where it measured faster: the fp64 fixed-point tiles (about 20% at 2^13-element
// tiles) and the 4-byte 64-byte-segment tiles of 256 threads (about 7%).
template <class S>
constexpr int col_tma_min_blocks(int kind) {
  return (kind == 1 || ((kind == 0 || kind == 2) && S::TS == 4 && S::NT == 256))
             ? (S::NT < 768 ? 768 / S::NT : 1)
             : (S::NT < 512 ? 512 / S::NT : 1);
}
template <class S, int KIND>
__global__ void __launch_bounds__(S::NT, col_tma_min_blocks<S>(KIND))
    fwt_col_tma_kernel(const __grid_constant__ TmaPassParams tp) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  TmaMover<S, (KIND == 1 || KIND == 3) ? 8 : 4> mv(tp, smem_raw, &bar);
  tile_body<S, KIND>(tp.p, smem_raw, mv, StaticBits<S>(tp.p));
}

// ---- one-pass transform of a vector spread over a thread-block cluster -----------------
// A vector of 2^n elements, n = TB + CL, is held by a cluster of 2^CL CTAs, CTA r
// owning the contiguous slice [r 2^TB, (r+1) 2^TB).  Each CTA transforms the low TB
// index bits of its slice with the tile engine.  CTA s then finishes the slice
// positions [s M, (s+1) M), M = 2^TB / 2^CL: it gathers the elements of all 2^CL
// slices at those positions through distributed shared memory, runs the CL
// butterfly stages in registers and writes the 2^CL outputs.  The gather is a pull
// (each CTA parks its slice in its own shared memory; after a cluster barrier CTA s
// reads the positions from every CTA, ld.shared::cluster; a last barrier keeps the
// slices alive until all reads are done) or, for large clusters, a push (after a
// barrier every CTA stores its elements straight into the finishing CTAs' shared
// memory, st.shared::cluster, slot r of s's buffer; after a second barrier CTA s
// reads its positions locally).  The whole transform costs one HBM read and one
// write of each element (the second Kronecker factor moves over the cluster's
// shared memory instead of HBM).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// 16-byte store into the shared memory of CTA `rank` of the cluster, at the same
// offset as `local` in this CTA.
__device__ __forceinline__ void st_dsmem16(void* local, uint32_t rank, const uint4& v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(remote), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Hands this CTA's transformed slice (layout L3) to the CTAs that finish it: the
// element at slice position i goes to CTA s = i / M, into slot `rank` of s's buffer
// (element rank M + i mod M).  A warp's 16-byte vectors are 512 contiguous bytes of
// one slice, so each store instruction goes to one CTA, conflict-free.
template <class S, int CL, typename U>
__device__ __forceinline__ void push_to_owners(const U (&x)[S::NE], U* sm, uint32_t rank) {
  constexpr int M = 1 << (S::TB - CL);
  using V = typename Vec16<U>::type;
#pragma unroll
  for (int j = 0; j < S::NV; ++j) {
    const uint32_t i = S::idx3(threadIdx.x, j * S::VEC);
    const uint32_t owner = i >> (S::TB - CL);  // uniform over the warp
    U* dst = sm + rank * M + (i & (M - 1));
    V v;
    U* pv = reinterpret_cast<U*>(&v);
#pragma unroll
    for (int e = 0; e < S::VEC; ++e) pv[e] = x[j * S::VEC + e];
    if (owner == rank) *reinterpret_cast<V*>(dst) = v;
    else st_dsmem16(dst, owner, *reinterpret_cast<const uint4*>(&v));
  }
}

// The 2^CL slices' elements at this CTA's 16-byte position j (offset within its
// share), from its own buffer after the push.
template <int C, int M, int VEC, typename U>
__device__ __forceinline__ void gather_share(const U* sm, uint32_t j, U (&y)[C * VEC]) {
  using V = typename Vec16<U>::type;
#pragma unroll
  for (int r = 0; r < C; ++r) {
    const V v = *reinterpret_cast<const V*>(sm + r * M + j);
    const U* pv = reinterpret_cast<const U*>(&v);
#pragma unroll
    for (int e = 0; e < VEC; ++e) y[r * VEC + e] = pv[e];
  }
}

// 16-byte load from the shared memory of CTA `rank` of the cluster, at the same
// offset as `local` in this CTA.
__device__ __forceinline__ uint4 ld_dsmem16(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// The 2^CL slices' elements at slice position i, read from every CTA's parked slice.
template <int C, int VEC, typename U>
__device__ __forceinline__ void gather_remote(const U* sm, uint32_t i, U (&y)[C * VEC]) {
#pragma unroll
  for (int r = 0; r < C; ++r) {
    const uint4 v = ld_dsmem16(sm + i, (uint32_t)r);
    const U* pv = reinterpret_cast<const U*>(&v);
#pragma unroll
    for (int e = 0; e < VEC; ++e) y[r * VEC + e] = pv[e];
  }
}

// Layout L3 back to the tile buffer in natural order (after the engine's last reads).
template <class S, typename U>
__device__ __forceinline__ void park_natural(const U (&x)[S::NE], U* sm) {
  __syncthreads();
#pragma unroll
  for (int j = 0; j < S::NV; ++j) put_vec<U, S::VEC>(sm + S::idx3(threadIdx.x, j * S::VEC), x, j);
}

// 32-bit load from the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t ld_dsmem32(const void* local, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// fp64 one-pass on a cluster of 2^CL CTAs, in exact fixed point: one binary
// exponent for the whole 2^(TB+CL)-element vector (the largest over the cluster),
// each slice transformed in int64 by the tile engine, the top CL bits across the
// cluster, one rounding to fp64 on the way out.  The vector has F = 61 - (TB + CL)
// fraction bits, so the per-pass bound sqrt(2^(TB+CL)) 2^-(F+1) stays below 1e-12
// only for TB + CL <= 14: the registry builds it for TB = 13, CL = 1.  Every CTA
// takes every cluster barrier whatever happens (a slice whose bulk copy gave up
// computes on zeros and stores nothing), so no CTA waits on one that left.
template <class S, int CL>
__device__ __forceinline__ void cluster_fixed_body(const PassParams& p, unsigned char* smem_raw,
                                                   uint64_t* bar) {
  constexpr int C = 1 << CL;
  constexpr int M = 1 << (S::TB - CL);            // slice positions each CTA finishes
  constexpr int GROUPS = M / S::VEC / S::NT;      // 16-byte positions a thread finishes
  static_assert(GROUPS >= 1, "each thread finishes at least one 16-byte position");
  static_assert(S::TB + CL <= 14, "the fixed-point error bound needs vectors of <= 2^14");
  __shared__ uint32_t red[32];
  __shared__ uint32_t slice_key;
  long long* sm = reinterpret_cast<long long*>(smem_raw);
  const uint32_t t = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const long long vbase = ((long long)blockIdx.x >> CL) << (S::TB + CL);
  long long* out = static_cast<long long*>(blockIdx.y != 0 ? p.out[1] : p.out[0]);

  BulkMover<S> mv(p, smem_raw, bar);
  long long x[S::NE];
  const bool loaded = mv.load(x, p.ld_policy);
  if (!loaded) {
#pragma unroll
    for (int r = 0; r < S::NE; ++r) x[r] = 0;
  }
  // largest exponent of the slice, then of the vector
  uint32_t key = 0;
#pragma unroll
  for (int r = 0; r < S::NE; ++r) key = max(key, abs_hi(x[r]));
  key = __reduce_max_sync(0xffffffffu, key);
  if ((t & 31u) == 0) red[t >> 5] = key;
  __syncthreads();
  if (t == 0) {
    uint32_t k = red[0];
#pragma unroll
    for (int w = 1; w < S::NT / 32; ++w) k = max(k, red[w]);
    slice_key = k;
  }
  cluster_sync_all();  // every slice's key is visible to the cluster
  key = 0;
#pragma unroll
  for (int r = 0; r < C; ++r) key = max(key, ld_dsmem32(&slice_key, (uint32_t)r));
  const unsigned long long pol = l2_policy(p.st_policy);

  if (key >= 0x7ff00000u) {  // rare (cluster-uniform): Inf/NaN take plain IEEE fp64 adds
    double xd[S::NE];
#pragma unroll
    for (int r = 0; r < S::NE; ++r) xd[r] = __longlong_as_double(x[r]);
    double* smd = reinterpret_cast<double*>(sm);
    tile_rounds<S, ArithF64>(xd, smd);
    park_natural<S>(xd, smd);
    cluster_sync_all();  // every slice is in its CTA's shared memory
#pragma unroll 2
    for (int q = 0; q < GROUPS; ++q) {
      const uint32_t i = rank * M + (t + q * S::NT) * S::VEC;
      double y[C * S::VEC];
      gather_remote<C, S::VEC>(smd, i, y);
      butterflies<ArithF64>(y, (uint32_t)(C - 1) << S::LV);
      if (p.do_scale) {
#pragma unroll
        for (int e = 0; e < C * S::VEC; ++e) y[e] = y[e] * p.scale_f64;
      }
      if (loaded) {
#pragma unroll
        for (int r = 0; r < C; ++r) {
          double2 v = make_double2(y[r * S::VEC], y[r * S::VEC + 1]);
          stg16<double>(out + vbase + ((long long)r << S::TB) + i, v, pol);
        }
      }
    }
    cluster_sync_all();  // no CTA leaves while others still read its shared memory
    return;
  }

  const int emax = max((int)(key >> 20), 1);
  constexpr int F = 61 - (S::TB + CL);
  static_assert(F <= 51, "vectors this long always shift right");
#pragma unroll
  for (int r = 0; r < S::NE; ++r) x[r] = to_fixed<TO_FIXED_ROUND>(x[r], emax, F);
  tile_rounds<S, ArithI64>(x, sm);
  park_natural<S>(x, sm);
  cluster_sync_all();  // every slice is in its CTA's shared memory
  const int e0 = emax - 1023 - F + (p.do_scale ? p.scale_exp : 0);
  const int half = p.do_scale ? p.scale_half : 0;
  const bool normal = e0 >= -1022 && e0 <= 960;  // results are normal numbers (uniform)
  const long long e0_field = (long long)((unsigned long long)(long long)e0 << 52);
#pragma unroll 2
  for (int q = 0; q < GROUPS; ++q) {
    const uint32_t i = rank * M + (t + q * S::NT) * S::VEC;
    long long y[C * S::VEC];
    gather_remote<C, S::VEC>(sm, i, y);
    butterflies<ArithI64>(y, (uint32_t)(C - 1) << S::LV);
    if (normal) {
#pragma unroll
      for (int e = 0; e < C * S::VEC; ++e)
        y[e] = half ? from_fixed_cvt<true>(y[e], e0_field, p.rsqrt2_q64)
                    : from_fixed_cvt<false>(y[e], e0_field, p.rsqrt2_q64);
    } else {
#pragma unroll 1
      for (int e = 0; e < C * S::VEC; ++e) y[e] = from_fixed_exact(y[e], e0, half, p.rsqrt2_q64);
    }
    if (loaded) {
#pragma unroll
      for (int r = 0; r < C; ++r) {
        longlong2 v = make_longlong2(y[r * S::VEC], y[r * S::VEC + 1]);
        stg16<long long>(out + vbase + ((long long)r << S::TB) + i, v, pol);
      }
    }
  }
  cluster_sync_all();  // no CTA leaves while others still read its shared memory
}

// fp32 / int32 body of the cluster kernel (see above).
template <class S, int KIND, int CL>
__device__ __forceinline__ void cluster_plain_body(const PassParams& p, unsigned char* smem_raw) {
  using T = typename std::conditional<KIND == 0, float, uint32_t>::type;
  using A = typename std::conditional<KIND == 0, ArithF32, ArithU32>::type;
  constexpr int C = 1 << CL;
  constexpr int M = 1 << (S::TB - CL);  // slice positions each CTA finishes
  constexpr int GROUPS = M / S::VEC / S::NT;  // 16-byte positions a thread finishes
  static_assert(GROUPS >= 1, "each thread finishes at least one 16-byte position");
  T* sm = reinterpret_cast<T*>(smem_raw);
  const uint32_t t = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const long long vec = (long long)blockIdx.x >> CL;
  const bool im = blockIdx.y != 0;
  const T* in = static_cast<const T*>(im ? p.in[1] : p.in[0]);
  T* out = static_cast<T*>(im ? p.out[1] : p.out[0]);
  const long long vbase = vec << (S::TB + CL);

  // low TB bits of the slice, in the tile engine
  TileMap<S, false, false> m;
  m.base = vbase + ((long long)rank << S::TB);
  m.L = 0;
  m.valid = 0;
  T x[S::NE];
  load_tile<S>(in, m, x, p.ld_policy);
  tile_rounds<S, A>(x, sm);
  // Clusters of up to 4 CTAs pull the other slices' elements from their CTAs'
  // shared memory; larger ones, where remote loads would keep many more requests in
  // flight for each thread, push their elements to the finishing CTAs instead
  // (measured: pull faster at 2 and 4 CTAs, push at 8 and 16).
  constexpr bool kPush = C >= 8;
  if constexpr (kPush) {
    cluster_sync_all();  // every CTA is done with its buffer; the peers write into it next
    push_to_owners<S, CL>(x, sm, rank);
  } else {
    park_natural<S>(x, sm);
  }
  cluster_sync_all();  // every share (push) or slice (pull) is in place

  // top CL bits of this CTA's share
  const unsigned long long pol = l2_policy(p.st_policy);
#pragma unroll
  for (int q = 0; q < GROUPS; ++q) {
    const uint32_t j = (t + q * S::NT) * S::VEC, i = rank * M + j;  // share offset, slice position
    T y[C * S::VEC];
    if constexpr (kPush) gather_share<C, M, S::VEC>(sm, j, y);
    else gather_remote<C, S::VEC>(sm, i, y);
    butterflies<A>(y, (uint32_t)(C - 1) << S::LV);
    if constexpr (KIND == 0) {
      if (p.do_scale) {
#pragma unroll
        for (int e = 0; e < C * S::VEC; ++e) y[e] = y[e] * p.scale_f32;
      }
    }
#pragma unroll
    for (int r = 0; r < C; ++r) {
      typename Vec16<T>::type v;
      T* pv = reinterpret_cast<T*>(&v);
#pragma unroll
      for (int e = 0; e < S::VEC; ++e) pv[e] = y[r * S::VEC + e];
      stg16<T>(out + vbase + ((long long)r << S::TB) + i, v, pol);
    }
  }
  if constexpr (!kPush) cluster_sync_all();  // no CTA leaves while others still read its shared memory
}

// 768 threads an SM at up to 80 registers: a third resident CTA per SM measured
// 2-10% faster than two at 128 registers for every cluster shape.
template <class S, int KIND, int CL>
__global__ void __launch_bounds__(S::NT, (S::NT < 768 ? 768 / S::NT : 1))
    fwt_cluster_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if constexpr (KIND == 1) {
    __shared__ __align__(8) uint64_t bar;
    cluster_fixed_body<S, CL>(p, smem_raw, &bar);
  } else {
    cluster_plain_body<S, KIND, CL>(p, smem_raw);
  }
}

// ---- fused diagonal phase + transform (first pass, fp32) ----------------------------
// The first pass of y = s * H (e^{i theta} . x): each CTA loads the real part,
// the imaginary part and the angles of one row tile, rotates every amplitude by
// its phase (sincosf), and transforms both rotated parts in turn through the same
// shared buffer.  Later passes (if any) are ordinary column passes.  Three CTAs an SM
// (80 registers, a few spilled): the loads of three arrays need the warps more than the
// registers (at two CTAs an SM, 108 registers, it measured 1.30 ms against 1.09 ms for
// n = 24, batch 16).
template <class S>
__global__ void __launch_bounds__(S::NT, (S::NT < 768 ? 768 / S::NT : 1))
    fwt_phase_row_kernel(const PassParams p) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  float* sm = reinterpret_cast<float*>(smem_raw);
  const auto m = TileMap<S, false, true>::make(p, (long long)blockIdx.x);
  const float* in_re = static_cast<const float*>(p.in[0]);
  const float* in_im = static_cast<const float*>(p.in[1]);
  const unsigned long long pol = l2_policy(p.ld_policy);
  const long long vmask = (1ll << p.n) - 1;
  float xr[S::NE], xi[S::NE];
#pragma unroll
  for (int j = 0; j < S::NV; ++j) {
    const uint32_t u = S::idx1(threadIdx.x, j * S::VEC);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, th = a;
    if (m.in_range(u)) {
      const long long g = m.off(u);
      a = ldg16<float>(in_re + g, pol);
      b = ldg16<float>(in_im + g, pol);
      th = ldg16<float>(p.theta + (g >> p.n) * p.theta_stride + (g & vmask), pol);
    }
    const float* pa = reinterpret_cast<const float*>(&a);
    const float* pb = reinterpret_cast<const float*>(&b);
    const float* pt = reinterpret_cast<const float*>(&th);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float sn, cs;
      sincosf(pt[i], &sn, &cs);
      xr[j * 4 + i] = pa[i] * cs - pb[i] * sn;
      xi[j * 4 + i] = pa[i] * sn + pb[i] * cs;
    }
  }
  tile_rounds<S, ArithF32>(xr, sm);
  if (p.do_scale) {
#pragma unroll
    for (int r = 0; r < S::NE; ++r) xr[r] *= p.scale_f32;
  }
  store_tile<S>(static_cast<float*>(p.out[0]), m, xr, p.st_policy);
  __syncthreads();  // the buffer's last reads (layout L3) are done
  tile_rounds<S, ArithF32>(xi, sm);
  if (p.do_scale) {
#pragma unroll
    for (int r = 0; r < S::NE; ++r) xi[r] *= p.scale_f32;
  }
  store_tile<S>(static_cast<float*>(p.out[1]), m, xi, p.st_policy);
}

// The same for vectors of 2^NL <= 4 elements: one thread per vector.
template <int NL>
__global__ void __launch_bounds__(256) fwt_phase_small_kernel(const PassParams p) {
  pdl_begin();
  const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (p.comp_elems >> NL)) return;
  const float* in_re = static_cast<const float*>(p.in[0]);
  const float* in_im = static_cast<const float*>(p.in[1]);
  float xr[1 << NL], xi[1 << NL];
#pragma unroll
  for (int i = 0; i < (1 << NL); ++i) {
    float sn, cs;
    sincosf(p.theta[row * p.theta_stride + i], &sn, &cs);
    const float a = in_re[(row << NL) + i], b = in_im[(row << NL) + i];
    xr[i] = a * cs - b * sn;
    xi[i] = a * sn + b * cs;
  }
  butterflies<ArithF32>(xr, (1u << NL) - 1u);
  butterflies<ArithF32>(xi, (1u << NL) - 1u);
  const float s = p.do_scale ? p.scale_f32 : 1.0f;
#pragma unroll
  for (int i = 0; i < (1 << NL); ++i) {
    static_cast<float*>(p.out[0])[(row << NL) + i] = xr[i] * s;
    static_cast<float*>(p.out[1])[(row << NL) + i] = xi[i] * s;
  }
}

// Vectors of 2^NL <= 4 elements: one thread per vector, plain arithmetic.
template <typename T, class A, int NL>
__global__ void __launch_bounds__(256) fwt_small_kernel(const PassParams p) {
  pdl_begin();
  const bool im = blockIdx.y != 0;
  const T* in = static_cast<const T*>(im ? p.in[1] : p.in[0]);
  T* out = static_cast<T*>(im ? p.out[1] : p.out[0]);
  const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (p.comp_elems >> NL)) return;
  T x[1 << NL];
#pragma unroll
  for (int i = 0; i < (1 << NL); ++i) x[i] = in[(row << NL) + i];
  butterflies<A>(x, (1u << NL) - 1u);
  if (p.do_scale) {
#pragma unroll
    for (int i = 0; i < (1 << NL); ++i) {
      if constexpr (sizeof(T) == 4 && !std::is_integral<T>::value) x[i] = x[i] * p.scale_f32;
      else if constexpr (sizeof(T) == 8) x[i] = x[i] * p.scale_f64;
    }
  }
#pragma unroll
  for (int i = 0; i < (1 << NL); ++i) out[(row << NL) + i] = x[i];
}

}  // namespace fwt
