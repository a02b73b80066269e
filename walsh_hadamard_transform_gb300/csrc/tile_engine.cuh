// On-chip tile engine for the batched Walsh-Hadamard transform (sm_103a).
//
// A CTA owns one tile of 2^TB elements of one real array (the real or the
// imaginary part of a batch of split complex vectors).  Within the tile the
// transform acts on TK consecutive tile-index bits starting at bit TS; the other
// tile-index bits are independent lanes of the same transform (several short
// vectors packed into one tile, or the contiguous columns of a strided tile of
// the Kronecker column pass).
//
// The butterfly network of the transform (iThome "Day 18" FWT post, section
// "Tensor Core wants matrix multiplication": stage 0 local pairs, stage 1 stride
// 2, stage 2 stride 4, ...) factors over index bits, and its stages commute, so
// the stages may run in any order as long as every transformed bit gets exactly
// one stage.  The tile moves through three register layouts:
//
//   L1  (load):  registers hold tile bits [0,LV) (one 16-byte vector) and the top
//                E-LV bits; lanes hold bits [LV, LV+5); warps the rest.  Global
//                loads are 16-byte vectors, 512 contiguous bytes per warp.
//   L2:          registers hold bits [LV, LV+E); threads hold [0,LV) and the top.
//   L3  (store): registers hold bits [0,LV) and [LV+5, E+5); lanes [LV, LV+5);
//                warps the top.  Global stores are 16-byte vectors again.
//
// Each layout runs the butterflies of the register bits that are transformed and
// not done yet; the two layout changes go through one XOR-swizzled shared-memory
// buffer of the whole tile (iThome "Day 18" FWT post, intro: registers, warp
// exchange and swizzled shared memory for the single-block path).  Each element
// therefore costs one HBM read and one HBM write per pass.
//
// The swizzle XORs the low three bits of a 16-byte chunk index with the XOR-fold
// of its higher 3-bit groups.  It keeps 16-byte vectors contiguous and makes the
// vector accesses of L1/L3 and the scalar accesses of L2 free of bank conflicts
// (checked on the host by fwt_selfcheck()).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fwt {

__host__ __device__ constexpr int ilog2c(long long v) { return v <= 1 ? 0 : 1 + ilog2c(v >> 1); }

// Swizzled 16-byte chunk index (GF(2)-linear, bijective on any power-of-two range).
__host__ __device__ constexpr uint32_t swz_chunk(uint32_t c) {
  return c ^ (((c >> 3) ^ (c >> 6) ^ (c >> 9) ^ (c >> 12) ^ (c >> 15)) & 7u);
}

// Compile-time description of one tile shape and its three layouts.
//   TB: log2 elements per tile.  TS, TK: transformed tile bits [TS, TS+TK).
//   LV: log2 elements per 16-byte vector.  PL: log2 threads per CTA.
template <int TB_, int TS_, int TK_, int LV_, int PL_>
struct Shape {
  static constexpr int TB = TB_, TS = TS_, TK = TK_, LV = LV_, PL = PL_;
  static constexpr int EL = TB - PL;  // log2 elements per thread
  static constexpr int NT = 1 << PL, NE = 1 << EL, VEC = 1 << LV, NV = NE / VEC;
  static_assert(PL >= 5, "at least one warp");
  static_assert(EL >= 5, "L2 must hold the five lane bits of L1");
  static_assert(LV <= PL && PL <= EL + 5 - LV, "L3 must hold the warp bits of L1");
  static_assert(TS + TK <= TB, "transform bits inside the tile");

  // element index (tile-local) of register r of thread t in each layout
  __host__ __device__ static constexpr uint32_t idx1(uint32_t t, uint32_t r) {
    return (r & (VEC - 1)) | (t << LV) | ((r >> LV) << (LV + PL));
  }
  __host__ __device__ static constexpr uint32_t idx2(uint32_t t, uint32_t r) {
    return (t & (VEC - 1)) | (r << LV) | ((t >> LV) << (LV + EL));
  }
  __host__ __device__ static constexpr uint32_t idx3(uint32_t t, uint32_t r) {
    return (r & (VEC - 1)) | ((t & 31u) << LV) | ((r >> LV) << (LV + 5)) | ((t >> 5) << (EL + 5));
  }
  // register bit h -> tile-index bit, per layout
  __host__ __device__ static constexpr int rbit(int layout, int h) {
    return layout == 1 ? (h < LV ? h : h + PL) : layout == 2 ? h + LV : (h < LV ? h : h + 5);
  }
  // tile-index bits held in registers by a layout
  __host__ __device__ static constexpr uint32_t reg_elem_bits(int layout) {
    uint32_t m = 0;
    for (int h = 0; h < EL; ++h) m |= 1u << rbit(layout, h);
    return m;
  }
  static constexpr uint32_t TSET = ((TK >= 32 ? 0u : (1u << TK)) - 1u) << TS;
  static constexpr uint32_t DONE1 = reg_elem_bits(1) & TSET;
  static constexpr uint32_t DONE2 = reg_elem_bits(2) & TSET & ~DONE1;
  static constexpr uint32_t DONE3 = reg_elem_bits(3) & TSET & ~(DONE1 | DONE2);
  static_assert((DONE1 | DONE2 | DONE3) == TSET, "every transformed bit gets one stage");
  // the same sets as register-bit masks
  __host__ __device__ static constexpr uint32_t reg_mask(int layout, uint32_t elem_set) {
    uint32_t m = 0;
    for (int h = 0; h < EL; ++h)
      if ((elem_set >> rbit(layout, h)) & 1u) m |= 1u << h;
    return m;
  }
  static constexpr uint32_t RM1 = reg_mask(1, DONE1);
  static constexpr uint32_t RM2 = reg_mask(2, DONE2);
  static constexpr uint32_t RM3 = reg_mask(3, DONE3);
  // The same three register masks for transformed tile bits [ts, ts+tk) given at
  // run time (a transform on a sub-range of the index bits).
  __host__ __device__ static constexpr void round_masks(int ts, int tk, uint32_t (&rm)[3]) {
    round_masks_set((tk <= 0 ? 0u : ((tk >= 32 ? 0u : (1u << tk)) - 1u)) << ts, rm);
  }
  // ... and for any set of tile bits (a bit mask below 2^TB): the three layouts'
  // register bits cover every tile bit, so any set is partitioned among the rounds.
  __host__ __device__ static constexpr void round_masks_set(uint32_t tset, uint32_t (&rm)[3]) {
    const uint32_t d1 = reg_elem_bits(1) & tset;
    const uint32_t d2 = reg_elem_bits(2) & tset & ~d1;
    const uint32_t d3 = reg_elem_bits(3) & tset & ~(d1 | d2);
    rm[0] = reg_mask(1, d1);
    rm[1] = reg_mask(2, d2);
    rm[2] = reg_mask(3, d3);
  }
  // swizzled shared-memory element offset of a tile index
  __host__ __device__ static constexpr uint32_t phys(uint32_t idx) {
    return (swz_chunk(idx >> LV) << LV) | (idx & (VEC - 1));
  }

  // The same offsets, split into a per-thread table of 8 values and a
  // compile-time constant per register, so each shared-memory access needs no
  // address arithmetic.  The swizzle is linear over XOR and the thread and
  // register parts of a chunk index occupy disjoint bits, so
  //   phys = table[h(register)] + const(register),
  // where the table entry absorbs the thread's part of the 3-bit XOR.
  __host__ __device__ static constexpr uint32_t fold7(uint32_t v) {
    return (v ^ (v >> 3) ^ (v >> 6) ^ (v >> 9) ^ (v >> 12)) & 7u;
  }
  // layout 1, vector j: chunk = t | j << PL
  __host__ __device__ static void table1(uint32_t t, uint32_t (&tab)[8]) {
    const uint32_t lo = (t & 7u) ^ fold7(t >> 3);
    for (uint32_t h = 0; h < 8; ++h) tab[h] = ((t & ~7u) + (lo ^ h)) << LV;
  }
  __host__ __device__ static constexpr uint32_t h1(int j) { return fold7((uint32_t)j << (PL - 3)); }
  __host__ __device__ static constexpr uint32_t c1(int j) { return ((uint32_t)j << PL) << LV; }
  // layout 2, register r: chunk = r | (t >> LV) << EL, plus the element within the vector
  __host__ __device__ static void table2(uint32_t t, uint32_t (&tab)[8]) {
    const uint32_t tt = (t >> LV) << EL;
    const uint32_t g = fold7(tt >> 3);
    for (uint32_t h = 0; h < 8; ++h) tab[h] = ((tt + (h ^ g)) << LV) + (t & (VEC - 1));
  }
  __host__ __device__ static constexpr uint32_t h2(int r) {
    return ((uint32_t)r & 7u) ^ fold7((uint32_t)r >> 3);
  }
  __host__ __device__ static constexpr uint32_t c2(int r) { return ((uint32_t)r & ~7u) << LV; }
  // layout 3, vector j: chunk = (t & 31) | j << 5 | (t >> 5) << (EL + 5 - LV)
  __host__ __device__ static void table3(uint32_t t, uint32_t (&tab)[8]) {
    const uint32_t lp = t & 31u, wp = (t >> 5) << (EL + 5 - LV);
    const uint32_t g = fold7(lp >> 3) ^ fold7(wp >> 3);
    for (uint32_t h = 0; h < 8; ++h) tab[h] = (wp + (lp & ~7u) + ((lp & 7u) ^ g ^ h)) << LV;
  }
  __host__ __device__ static constexpr uint32_t h3(int j) { return fold7((uint32_t)j << 2); }
  __host__ __device__ static constexpr uint32_t c3(int j) { return ((uint32_t)j << 5) << LV; }
};

// In-register butterflies over the register bits in `mask`: pairs (r, r | 2^h) with
// bit h of r clear become (a + b, a - b).  A compile-time mask folds the tests
// away; a run-time mask is uniform over the CTA, so its tests never diverge.
//
// Integer arithmetic (A::kRadix4) takes two stages at once where the mask allows:
// a quadruple (a, b, c, d) = x[r], x[r+2^h], x[r+2^(h+1)], x[r+3*2^h] becomes
// (a+b+c+d, a-b+c-d, a+b-c-d, a-b-c+d), six three-operand sums instead of eight
// two-operand ones.  Integer sums are exact (or wrap identically), so grouping the
// stages changes no bit of the result.
template <class A, typename U>
__device__ __forceinline__ void radix2(U& a, U& b) {
  const U s = A::add(a, b), d = A::sub(a, b);
  a = s;
  b = d;
}
template <class A, typename U>
__device__ __forceinline__ void radix4(U& a, U& b, U& c, U& d) {
  const U s = A::add(a, b), t = A::sub(a, b);
  const U y0 = A::add3(s, c, d);     // + + + +
  const U y1 = A::add_sub(t, c, d);  // + - + -
  const U y2 = A::sub2(s, c, d);     // + + - -
  const U y3 = A::sub_add(t, c, d);  // + - - +
  a = y0;
  b = y1;
  c = y2;
  d = y3;
}
template <class A, int NE, typename U>
__device__ __forceinline__ void butterflies(U (&x)[NE], uint32_t mask) {
  constexpr int LOG = ilog2c(NE);
#pragma unroll
  for (int h = 0; h < LOG; ++h) {
    const bool here = (mask >> h) & 1u;
    if constexpr (A::kRadix4) {
      if (h + 1 < LOG && here && ((mask >> (h + 1)) & 1u)) {
#pragma unroll
        for (int r = 0; r < NE; ++r)
          if (!((r >> h) & 3))
            radix4<A>(x[r], x[r | (1 << h)], x[r | (2 << h)], x[r | (3 << h)]);
        mask &= ~(2u << h);  // stage h + 1 is done
        continue;
      }
    }
    if (here) {
#pragma unroll
      for (int r = 0; r < NE; ++r)
        if (!((r >> h) & 1)) radix2<A>(x[r], x[r | (1 << h)]);
    }
  }
}

template <typename U> struct Vec16;
template <> struct Vec16<float> { using type = float4; };
template <> struct Vec16<uint32_t> { using type = uint4; };
template <> struct Vec16<double> { using type = double2; };
template <> struct Vec16<long long> { using type = longlong2; };

// Store / load one 16-byte vector of registers x[j*VEC .. j*VEC+VEC-1].
template <typename U, int VEC, int NE>
__device__ __forceinline__ void put_vec(U* p, const U (&x)[NE], int j) {
  using V = typename Vec16<U>::type;
  V v;
  U* pv = reinterpret_cast<U*>(&v);
#pragma unroll
  for (int i = 0; i < VEC; ++i) pv[i] = x[j * VEC + i];
  *reinterpret_cast<V*>(p) = v;
}
template <typename U, int VEC, int NE>
__device__ __forceinline__ void get_vec(const U* p, U (&x)[NE], int j) {
  using V = typename Vec16<U>::type;
  const V v = *reinterpret_cast<const V*>(p);
  const U* pv = reinterpret_cast<const U*>(&v);
#pragma unroll
  for (int i = 0; i < VEC; ++i) x[j * VEC + i] = pv[i];
}

// Rounds 1-3 of the tile transform.  On entry x holds the tile in layout L1; on
// exit it holds the transformed tile in layout L3.  `sm` is the tile-sized
// shared buffer; nothing may be pending on it on entry, and its last reads (the
// L3 loads) are not yet fenced by a barrier on exit.
template <class S, class A, typename U>
__device__ __forceinline__ void tile_rounds(U (&x)[S::NE], U* sm, uint32_t rm1 = S::RM1,
                                            uint32_t rm2 = S::RM2, uint32_t rm3 = S::RM3) {
  const uint32_t t = threadIdx.x;
  uint32_t tab[8];
  butterflies<A>(x, rm1);
  // L1 -> shared (16-byte vectors)
  S::table1(t, tab);
#pragma unroll
  for (int j = 0; j < S::NV; ++j) put_vec<U, S::VEC>(sm + tab[S::h1(j)] + S::c1(j), x, j);
  __syncthreads();
  // shared -> L2 (scalars)
  S::table2(t, tab);
#pragma unroll
  for (int r = 0; r < S::NE; ++r) x[r] = sm[tab[S::h2(r)] + S::c2(r)];
  butterflies<A>(x, rm2);
  __syncthreads();
  // L2 -> shared (scalars)
#pragma unroll
  for (int r = 0; r < S::NE; ++r) sm[tab[S::h2(r)] + S::c2(r)] = x[r];
  __syncthreads();
  // shared -> L3 (16-byte vectors)
  S::table3(t, tab);
#pragma unroll
  for (int j = 0; j < S::NV; ++j) get_vec<U, S::VEC>(sm + tab[S::h3(j)] + S::c3(j), x, j);
  butterflies<A>(x, rm3);
}

}  // namespace fwt
