// The compiled kernel set of one element type, registered by the per-type
// translation units (rows_*.cu, cols_*.cu compile in parallel).
#pragma once

#include <utility>
#include <vector>

#include "../../include/fwt.h"
#include "registry.cuh"

namespace fwt {

// Row passes: vectors of 2^NL <= 4 (one thread each), row tiles for K = 3 .. KMAX,
// and run-time bit-range tiles of 2^10 .. 2^KMAX elements.
template <int DT, int KIND, int LV, typename T, class A, int KMAX>
struct RowSet {
  template <int... Ks>
  static void rows(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
    (v.push_back(row_entry<DT, KIND, LV, Ks + 3>()), ...);
  }
  template <int... Ts>
  static void rowbits(std::vector<KernelEntry>& v, std::integer_sequence<int, Ts...>) {
    (v.push_back(rowbits_entry<DT, KIND, LV, Ts + 10>()), ...);
  }
  static void add(std::vector<KernelEntry>& v) {
    v.push_back(small_entry<DT, T, A, 0>());
    v.push_back(small_entry<DT, T, A, 1>());
    v.push_back(small_entry<DT, T, A, 2>());
    rows(v, std::make_integer_sequence<int, KMAX - 2>{});
    rowbits(v, std::make_integer_sequence<int, KMAX - 9>{});
  }
};

// One-pass cluster transforms for 4-byte types: slices of 2^13, 2^14 or 2^15
// elements on clusters of 2 .. 16 CTAs (n = 14 .. 18).
template <int DT, int KIND>
struct ClusterSet {
  static void add(std::vector<KernelEntry>& v) {
    v.push_back(cluster_entry<DT, KIND, 14, 1>());
    v.push_back(cluster_entry<DT, KIND, 14, 2>());
    v.push_back(cluster_entry<DT, KIND, 14, 3>());
    v.push_back(cluster_entry<DT, KIND, 14, 4>());
    v.push_back(cluster_entry<DT, KIND, 13, 1>());
    v.push_back(cluster_entry<DT, KIND, 13, 2>());
    v.push_back(cluster_entry<DT, KIND, 13, 3>());
    v.push_back(cluster_entry<DT, KIND, 15, 3>());
  }
};

// fp32 fused phase + transform first passes, K = 0 .. 13 (tiles of 32 elements a
// thread: both rotated parts stay in registers).
struct PhaseSet {
  template <int... Ks>
  static void add_k(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
    (v.push_back(phase_entry<Ks>()), ...);
  }
  static void add(std::vector<KernelEntry>& v) { add_k(v, std::make_integer_sequence<int, 14>{}); }
};

// Column passes: for each segment width CB of 16..128 bytes, column factors K
// with tiles of 2^10 .. 2^TBMAX elements, each with TMA staging and (from 32
// bytes up) with vector loads; and the factors too short for those (K = 1 .. 4
// for 4-byte, 1 .. 5 for 8-byte elements: wide segments of 2^(10-K) elements,
// vector loads).
template <int DT, int KIND, int LV, int TBMAX>
struct ColSet {
  template <int CB, bool TMA, int K0, int... Ks>
  static void cols(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
    (v.push_back(col_entry<DT, KIND, LV, Ks + K0, CB, TMA>()), ...);
  }
  template <int CB>
  static void width(std::vector<KernelEntry>& v) {
    constexpr int CWL = ilog2c(CB) - ilog2c(16 >> LV);
    // 16-byte segments are half a DRAM sector: only the TMA-staged variant
    if constexpr (CB > 16) cols<CB, false, 10 - CWL>(v, std::make_integer_sequence<int, TBMAX - 9>{});
    cols<CB, true, 10 - CWL>(v, std::make_integer_sequence<int, TBMAX - 9>{});
  }
  template <int... Ks>
  static void short_cols(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
    // K = Ks + 1 rows of 2^(10 - K) elements: CB = 2^(10 - K) * element bytes
    (v.push_back(col_entry<DT, KIND, LV, Ks + 1, (1 << (9 - Ks)) * (16 >> LV), false>()), ...);
  }
  static void add(std::vector<KernelEntry>& v) {
    width<16>(v);
    width<32>(v);
    width<64>(v);
    width<128>(v);
    // below the shortest 128-byte factor (10 - log2 of its columns)
    short_cols(v, std::make_integer_sequence<int, 9 - (ilog2c(128) - ilog2c(16 >> LV))>{});
  }
};

}  // namespace fwt
