// Table of compiled pass kernels, their launchers and host-side shape checks.
#pragma once

#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fwt_kernels.cuh"

namespace fwt {

enum PassKind {
  KIND_SMALL = 0,
  KIND_ROW = 1,
  KIND_COL = 2,
  KIND_ROWBITS = 3,
  KIND_PHASE = 4,
  KIND_CLUSTER = 5  // one pass over a vector spread across a thread-block cluster
};

struct KernelEntry {
  int dtype;  // FWT_C32 / FWT_C64 / FWT_I32
  int kind;   // PassKind
  int K;      // transformed index bits of the pass
  int TB;     // log2 elements per tile (0 for the small kernel)
  int TS;     // first transformed tile bit (column tiles: log2 columns per tile)
  int col_bytes;  // column tiles: bytes of contiguous columns per row (16 .. 128)
  int tma;        // column tiles staged through shared memory by TMA copies
  int threads;
  size_t smem;  // dynamic shared memory per CTA
  cudaError_t (*launch)(const PassParams&, long long tiles, int ncomp, cudaStream_t);
  cudaError_t (*setup)();  // per-device attributes; call with the device current
  int (*selfcheck)();      // host-only index-map and bank-conflict check
  const void* fn;
  int (*capacity)() = nullptr;  // cluster kernels: resident clusters (device current)
};

// Elements per thread for a tile of 2^TB elements: enough registers that the
// three layouts exist (see tile_engine.cuh), at least 32.
__host__ __device__ constexpr int choose_el(int TB, int LV) {
  return (TB - 5 + LV + 1) / 2 > 5 ? (TB - 5 + LV + 1) / 2 : 5;
}

// Whether pass kernels are launched with programmatic stream serialisation (see
// pdl_begin in tma.cuh); set with fwt_set_pdl.
int pdl_mode();

// Launches a pass kernel: `cluster` > 1 groups its CTAs into thread-block clusters,
// and with PDL on a grid of up to kPdlMaxCtas CTAs may start while the previous kernel
// on the stream drains.  That shortens back-to-back launch-bound transforms (n = 10 ..
// 14, batch 64: 5-13% a step); on grids of many waves it measured neutral (fp64,
// n = 24) or slower (fp32 n = 24: 13%), so those launch plainly.
constexpr unsigned long long kPdlMaxCtas = 2048;
template <typename... KArgs, typename... Args>
cudaError_t launch_pass(void (*kernel)(KArgs...), dim3 grid, unsigned threads, size_t smem,
                        cudaStream_t st, unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_mode() && (unsigned long long)grid.x * grid.y * grid.z <= kPdlMaxCtas) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- host-side checks of a tile shape ----------------------------------------------
template <class S>
uint32_t host_idx(int layout, uint32_t t, uint32_t r) {
  return layout == 1 ? S::idx1(t, r) : layout == 2 ? S::idx2(t, r) : S::idx3(t, r);
}

// Shared-memory wavefronts of one warp-wide access: `bytes` per lane (4, 8 or 16).
inline int smem_wavefronts(const uint32_t* byte_addr, int bytes) {
  // lanes per phase: 32 for 4-byte, 16 for 8-byte, 8 for 16-byte accesses
  const int per = bytes == 4 ? 32 : bytes == 8 ? 16 : 8;
  int total = 0;
  for (int ph = 0; ph < 32 / per; ++ph) {
    int worst = 0;
    for (int bank = 0; bank < 32; ++bank) {
      std::vector<uint32_t> words;
      for (int l = ph * per; l < (ph + 1) * per; ++l) {
        for (int w = 0; w < bytes / 4; ++w) {
          const uint32_t word = byte_addr[l] / 4 + w;
          if ((int)(word % 32) != bank) continue;
          bool dup = false;
          for (uint32_t v : words) dup |= v == word;
          if (!dup) words.push_back(word);
        }
      }
      if ((int)words.size() > worst) worst = (int)words.size();
    }
    total += worst;
  }
  return total;
}

// DIRECT: the tile is loaded and stored with 16-byte vector accesses (rather than
// TMA copies), so its global accesses must fill whole sectors too.
template <class S, bool COLS, bool DIRECT = true>
int check_shape(const char* name) {
  int fails = 0;
  const uint32_t n = 1u << S::TB;
  std::vector<uint8_t> seen(n);
  // 1. each layout is a bijection (thread, register) -> tile index
  for (int layout = 1; layout <= 3; ++layout) {
    std::fill(seen.begin(), seen.end(), 0);
    for (uint32_t t = 0; t < (uint32_t)S::NT; ++t)
      for (uint32_t r = 0; r < (uint32_t)S::NE; ++r) {
        const uint32_t u = host_idx<S>(layout, t, r);
        if (u >= n || seen[u]++) {
          if (fails < 4) fprintf(stderr, "fwt_selfcheck %s: layout %d not a bijection\n", name, layout);
          ++fails;
          t = S::NT; break;
        }
      }
  }
  // 2. register bit h of each layout flips tile bit rbit(layout, h)
  for (int layout = 1; layout <= 3; ++layout)
    for (int h = 0; h < S::EL; ++h)
      for (uint32_t t = 0; t < (uint32_t)S::NT; t += 7)
        for (uint32_t r = 0; r < (uint32_t)S::NE; ++r)
          if (!((r >> h) & 1u) &&
              host_idx<S>(layout, t, r | (1u << h)) != (host_idx<S>(layout, t, r) | (1u << S::rbit(layout, h)))) {
            if (fails < 8) fprintf(stderr, "fwt_selfcheck %s: register bit map wrong\n", name);
            ++fails;
          }
  // 3. the three rounds transform each bit of [TS, TS+TK) exactly once
  if ((S::DONE1 & S::DONE2) || (S::DONE1 & S::DONE3) || (S::DONE2 & S::DONE3) ||
      (S::DONE1 | S::DONE2 | S::DONE3) != S::TSET) {
    fprintf(stderr, "fwt_selfcheck %s: rounds do not partition the transformed bits\n", name);
    ++fails;
  }
  // 4a. the kernels' table-based shared-memory offsets equal the swizzle map
  for (uint32_t t = 0; t < (uint32_t)S::NT; ++t) {
    uint32_t tab[8];
    bool ok = true;
    S::table1(t, tab);
    for (int j = 0; j < S::NV; ++j) ok &= tab[S::h1(j)] + S::c1(j) == S::phys(S::idx1(t, j * S::VEC));
    S::table2(t, tab);
    for (int r = 0; r < S::NE; ++r) ok &= tab[S::h2(r)] + S::c2(r) == S::phys(S::idx2(t, r));
    S::table3(t, tab);
    for (int j = 0; j < S::NV; ++j) ok &= tab[S::h3(j)] + S::c3(j) == S::phys(S::idx3(t, j * S::VEC));
    if (!ok) {
      if (fails < 12) fprintf(stderr, "fwt_selfcheck %s: shared-memory address table wrong\n", name);
      ++fails;
      break;
    }
  }
  // 4b. shared-memory accesses are conflict-free (one wavefront per phase)
  const int esz = 16 / S::VEC;
  uint32_t addr[32];
  for (uint32_t w = 0; w < (uint32_t)S::NT / 32; ++w) {
    for (int j = 0; j < S::NV; ++j) {  // L1 writes and L3 reads: 16-byte vectors
      for (int layout = 1; layout <= 3; layout += 2) {
        for (int l = 0; l < 32; ++l)
          addr[l] = S::phys(host_idx<S>(layout, w * 32 + l, j * S::VEC)) * esz;
        if (smem_wavefronts(addr, 16) != 4) {
          if (fails < 12) fprintf(stderr, "fwt_selfcheck %s: bank conflict layout %d\n", name, layout);
          ++fails;
        }
      }
    }
    for (int r = 0; r < S::NE; ++r) {  // L2 reads and writes: scalars
      for (int l = 0; l < 32; ++l) addr[l] = S::phys(S::idx2(w * 32 + l, r)) * esz;
      if (smem_wavefronts(addr, esz) != (esz == 4 ? 1 : 2)) {
        if (fails < 12) fprintf(stderr, "fwt_selfcheck %s: bank conflict layout 2\n", name);
        ++fails;
      }
    }
  }
  // 4c. TMA-staged column tiles: layout L1 reads and layout L3 writes of the
  //     natural-order tile are conflict-free too
  if (COLS) {
    for (uint32_t w = 0; w < (uint32_t)S::NT / 32; ++w)
      for (int j = 0; j < S::NV; ++j)
        for (int layout = 1; layout <= 3; layout += 2) {
          for (int l = 0; l < 32; ++l) addr[l] = host_idx<S>(layout, w * 32 + l, j * S::VEC) * esz;
          if (smem_wavefronts(addr, 16) != 4) {
            if (fails < 12) fprintf(stderr, "fwt_selfcheck %s: natural-order conflict layout %d\n", name, layout);
            ++fails;
          }
        }
  }
  // 5. global accesses: every warp-wide 16-byte load (L1) and store (L3) fills
  //    whole 32-byte sectors (row tiles: 512 contiguous bytes)
  const int L = COLS ? S::TS + 3 : 0;  // any row stride >= the column width
  for (int layout = 1; DIRECT && layout <= 3; layout += 2)
    for (uint32_t w = 0; w < (uint32_t)S::NT / 32; ++w)
      for (int j = 0; j < S::NV; ++j) {
        std::vector<long long> sectors;
        for (int l = 0; l < 32; ++l) {
          const uint32_t u = host_idx<S>(layout, w * 32 + l, j * S::VEC);
          long long off = COLS ? ((long long)(u >> S::TS) << L) + (u & ((1u << S::TS) - 1u)) : u;
          const long long sec = off * esz / 32;
          bool dup = false;
          for (long long v : sectors) dup |= v == sec;
          if (!dup) sectors.push_back(sec);
        }
        if ((int)sectors.size() != 16) {
          if (fails < 16) fprintf(stderr, "fwt_selfcheck %s: uncoalesced global access\n", name);
          ++fails;
        }
      }
  return fails;
}

// ---- per-shape launch / setup ----------------------------------------------------------
// fp64 fixed-point row passes over whole tiles of up to 2^13 elements (three CTAs an
// SM) take the bulk-copy kernel when the pass asks for it (p.bulk); everything else
// the direct-load kernel.  (2^14-element tiles, one 512-thread CTA an SM, measured
// 12% slower with bulk copies than with vector loads.)
template <class S, int KIND, bool COLS>
constexpr bool has_bulk_row() { return KIND == 1 && !COLS && S::TB <= 13; }

template <class S, int KIND, bool COLS>
cudaError_t launch_tile(const PassParams& p, long long tiles, int ncomp, cudaStream_t st) {
  const size_t smem = (size_t)(1u << S::TB) * (KIND == 1 || KIND == 3 ? 8 : 4);
  const dim3 grid((unsigned)tiles, (unsigned)ncomp);
  if constexpr (has_bulk_row<S, KIND, COLS>()) {
    if (p.bulk && (p.comp_elems & ((1ll << S::TB) - 1)) == 0) {
      return launch_pass(fwt_row_bulk_kernel<S, KIND>, grid, S::NT, smem, st, 1, p);
    }
  }
  return launch_pass(fwt_tile_kernel<S, KIND, COLS>, grid, S::NT, smem, st, 1, p);
}
template <class S, int KIND, bool COLS>
cudaError_t setup_tile() {
  const size_t smem = (size_t)(1u << S::TB) * (KIND == 1 || KIND == 3 ? 8 : 4);
  if constexpr (has_bulk_row<S, KIND, COLS>()) {
    const cudaError_t err = cudaFuncSetAttribute(
        fwt_row_bulk_kernel<S, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  return cudaFuncSetAttribute(fwt_tile_kernel<S, KIND, COLS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename T, class A, int NL>
cudaError_t launch_small(const PassParams& p, long long tiles, int ncomp, cudaStream_t st) {
  return launch_pass(fwt_small_kernel<T, A, NL>, dim3((unsigned)tiles, (unsigned)ncomp), 256, 0, st,
                     1, p);
}
inline int selfcheck_none() { return 0; }

// The driver's tensor-map encoder, resolved once at run time (nullptr if absent).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// A 2-D tiled tensor map (no interleave, no swizzle, no fill), from a small
// per-thread cache of recently encoded maps: a transform called again on the same
// buffers reuses them instead of encoding again.  false if the encoder is missing
// or refuses the arguments.
bool tensor_map_2d(CUtensorMap* out, CUtensorMapDataType dt, void* base, const cuuint64_t dims[2],
                   cuuint64_t row_stride_bytes, const cuuint32_t box[2], int l2_promotion);
// L2 sector promotion of TMA column tiles, in bytes (0, 64, 128 or 256).
int tma_l2_promotion();

template <class S, int KIND>
cudaError_t launch_col_tma(const PassParams& p, long long tiles, int ncomp, cudaStream_t st) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  constexpr int esz = (KIND == 1 || KIND == 3) ? 8 : 4;
  const CUtensorMapDataType dt = esz == 8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT64
                                 : KIND == 2 ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t rows = (cuuint64_t)(p.comp_elems >> p.stride_log);
  if (rows > 0xffffffffull) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {1ull << p.stride_log, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)esz << p.stride_log};
  const cuuint32_t box[2] = {1u << S::TS, (cuuint32_t)TmaMover<S, (KIND == 1 || KIND == 3) ? 8 : 4>::BOXR};
  TmaPassParams tp;
  tp.p = p;
  const int promo = tma_l2_promotion();
  for (int c = 0; c < ncomp; ++c) {
    if (p.in[c] != p.out[c]) return cudaErrorInvalidValue;  // column passes run in place
    if (!tensor_map_2d(&tp.map[c], dt, p.out[c], dims, strides[0], box, promo))
      return cudaErrorInvalidValue;
  }
  if (ncomp == 1) tp.map[1] = tp.map[0];
  const size_t smem = (size_t)esz << S::TB;
  return launch_pass(fwt_col_tma_kernel<S, KIND>, dim3((unsigned)tiles, (unsigned)ncomp), S::NT, smem,
                     st, 1, tp);
}
template <class S, int KIND>
cudaError_t setup_col_tma() {
  const size_t smem = (size_t)((KIND == 1 || KIND == 3) ? 8 : 4) << S::TB;
  return cudaFuncSetAttribute(fwt_col_tma_kernel<S, KIND>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

inline cudaError_t setup_none() { return cudaSuccess; }

// Row pass over bits [0, K): tiles of 2^max(K, 10) contiguous elements.
template <int DT, int KIND, int LV, int K>
KernelEntry row_entry() {
  constexpr int TB = K > 10 ? K : 10;
  constexpr int EL = choose_el(TB, LV);
  using S = Shape<TB, 0, K, LV, TB - EL>;
  KernelEntry e;
  e.dtype = DT; e.kind = KIND_ROW; e.K = K; e.TB = TB; e.TS = 0; e.col_bytes = 0; e.tma = 0;
  e.threads = S::NT;
  e.smem = (size_t)(1u << TB) * (16 >> LV);
  e.launch = &launch_tile<S, KIND, false>;
  e.setup = &setup_tile<S, KIND, false>;
  e.selfcheck = [] { return check_shape<S, false>("row"); };
  e.fn = (const void*)&fwt_tile_kernel<S, KIND, false>;
  return e;
}

// Column pass over bits [L, L + K): tiles of 2^K rows x CB bytes of columns
// (CB = 32, 64 or 128: two, four or eight 16-byte vectors).
template <int DT, int KIND, int LV, int K, int CB, bool TMA>
KernelEntry col_entry() {
  constexpr int CWL = ilog2c(CB) - ilog2c(16 >> LV);  // log2 columns of CB bytes
  constexpr int TB = K + CWL;
  constexpr int EL = choose_el(TB, LV);
  using S = Shape<TB, CWL, K, LV, TB - EL>;
  KernelEntry e;
  e.dtype = DT; e.kind = KIND_COL; e.K = K; e.TB = TB; e.TS = CWL; e.col_bytes = CB;
  e.tma = TMA ? 1 : 0;
  e.threads = S::NT;
  e.smem = (size_t)(1u << TB) * (16 >> LV);
  if constexpr (TMA) {
    e.launch = &launch_col_tma<S, KIND>;
    e.setup = &setup_col_tma<S, KIND>;
    e.selfcheck = [] { return check_shape<S, true, false>("col tma"); };
    e.fn = (const void*)&fwt_col_tma_kernel<S, KIND>;
  } else {
    e.launch = &launch_tile<S, KIND, true>;
    e.setup = &setup_tile<S, KIND, true>;
    e.selfcheck = [] { return check_shape<S, true>("col"); };
    e.fn = (const void*)&fwt_tile_kernel<S, KIND, true>;
  }
  return e;
}

template <class S, int KIND>
cudaError_t launch_rowbits(const PassParams& p, long long tiles, int ncomp, cudaStream_t st) {
  const size_t smem = (size_t)(1u << S::TB) * (KIND == 1 || KIND == 3 ? 8 : 4);
  const dim3 grid((unsigned)tiles, (unsigned)ncomp);
  if constexpr (has_bulk_row<S, KIND, false>()) {
    if (p.bulk && (p.comp_elems & ((1ll << S::TB) - 1)) == 0) {
      return launch_pass(fwt_rowbits_bulk_kernel<S, KIND>, grid, S::NT, smem, st, 1, p);
    }
  }
  return launch_pass(fwt_rowbits_kernel<S, KIND>, grid, S::NT, smem, st, 1, p);
}
template <class S, int KIND>
cudaError_t setup_rowbits() {
  const size_t smem = (size_t)(1u << S::TB) * (KIND == 1 || KIND == 3 ? 8 : 4);
  if constexpr (has_bulk_row<S, KIND, false>()) {
    const cudaError_t err = cudaFuncSetAttribute(
        fwt_rowbits_bulk_kernel<S, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  return cudaFuncSetAttribute(fwt_rowbits_kernel<S, KIND>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Contiguous tiles of 2^TB elements transforming a run-time range of their bits.
template <int DT, int KIND, int LV, int TB>
KernelEntry rowbits_entry() {
  constexpr int EL = choose_el(TB, LV);
  using S = Shape<TB, 0, TB, LV, TB - EL>;
  KernelEntry e;
  e.dtype = DT; e.kind = KIND_ROWBITS; e.K = TB; e.TB = TB; e.TS = 0; e.col_bytes = 0; e.tma = 0;
  e.threads = S::NT;
  e.smem = (size_t)(1u << TB) * (16 >> LV);
  e.launch = &launch_rowbits<S, KIND>;
  e.setup = &setup_rowbits<S, KIND>;
  e.selfcheck = [] {
    int f = 0;
    for (int ts = 0; ts < TB; ++ts)  // every run-time range: the rounds partition it
      for (int tk = 0; ts + tk <= TB; ++tk) {
        uint32_t rm[3];
        S::round_masks(ts, tk, rm);
        uint32_t seen = 0;
        bool ok = true;
        for (int L = 1; L <= 3; ++L)
          for (int h = 0; h < S::EL; ++h)
            if ((rm[L - 1] >> h) & 1u) {
              const uint32_t b = 1u << S::rbit(L, h);
              ok &= !(seen & b);
              seen |= b;
            }
        const uint32_t want = (tk == 0 ? 0u : ((1u << tk) - 1u)) << ts;
        if (!ok || seen != want) {
          if (f < 4) fprintf(stderr, "fwt_selfcheck rowbits TB=%d: range [%d, %d) not covered once\n", TB, ts, ts + tk);
          ++f;
        }
      }
    return f;
  };
  e.fn = (const void*)&fwt_rowbits_kernel<S, KIND>;
  return e;
}

template <class S>
cudaError_t launch_phase_row(const PassParams& p, long long tiles, int, cudaStream_t st) {
  const size_t smem = (size_t)4 << S::TB;
  return launch_pass(fwt_phase_row_kernel<S>, dim3((unsigned)tiles), S::NT, smem, st, 1, p);
}
template <class S>
cudaError_t setup_phase_row() {
  return cudaFuncSetAttribute(fwt_phase_row_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)((size_t)4 << S::TB));
}
template <int NL>
cudaError_t launch_phase_small(const PassParams& p, long long tiles, int, cudaStream_t st) {
  return launch_pass(fwt_phase_small_kernel<NL>, dim3((unsigned)tiles), 256, 0, st, 1, p);
}

// fp32 phase-then-transform first pass over bits [0, K) (K <= 2: a thread per vector).
template <int K>
KernelEntry phase_entry() {
  KernelEntry e;
  e.dtype = FWT_C32; e.kind = KIND_PHASE; e.K = K; e.TS = 0; e.col_bytes = 0; e.tma = 0;
  if constexpr (K <= 2) {
    e.TB = 0; e.threads = 256; e.smem = 0;
    e.launch = &launch_phase_small<K>;
    e.setup = &setup_none;
    e.selfcheck = &selfcheck_none;
    e.fn = (const void*)&fwt_phase_small_kernel<K>;
  } else {
    constexpr int TB = K > 10 ? K : 10;
    constexpr int EL = choose_el(TB, 2);
    using S = Shape<TB, 0, K, 2, TB - EL>;
    e.TB = TB; e.threads = S::NT; e.smem = (size_t)4 << TB;
    e.launch = &launch_phase_row<S>;
    e.setup = &setup_phase_row<S>;
    e.selfcheck = [] { return check_shape<S, false>("phase row"); };
    e.fn = (const void*)&fwt_phase_row_kernel<S>;
  }
  return e;
}

template <class S, int KIND, int CL>
cudaError_t launch_cluster(const PassParams& p, long long tiles, int ncomp, cudaStream_t st) {
  return launch_pass(fwt_cluster_kernel<S, KIND, CL>, dim3((unsigned)tiles, (unsigned)ncomp),
                     S::NT, (size_t)(KIND == 1 ? 8 : 4) << S::TB, st, 1u << CL, p);
}
template <class S, int KIND, int CL>
cudaError_t setup_cluster() {
  cudaError_t err = cudaFuncSetAttribute(fwt_cluster_kernel<S, KIND, CL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((size_t)(KIND == 1 ? 8 : 4) << S::TB));
  if (err == cudaSuccess && CL > 3)
    err = cudaFuncSetAttribute(fwt_cluster_kernel<S, KIND, CL>,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return err;
}
// Clusters of 2^CL CTAs that can be resident at once (0: the shape cannot run).
template <class S, int KIND, int CL>
int cluster_capacity() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1u << CL, 1, 1);
  cfg.blockDim = dim3(S::NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)(KIND == 1 ? 8 : 4) << S::TB;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1u << CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fwt_cluster_kernel<S, KIND, CL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// One-pass transform of 2^(TB + CL)-element vectors on clusters of 2^CL CTAs
// (fp32 / int32, and fp64 fixed point for TB + CL = 14).  K = TB + CL is the
// vector's n.
template <int DT, int KIND, int TB, int CL>
KernelEntry cluster_entry() {
  constexpr int LV = KIND == 1 ? 1 : 2;
  constexpr int EL = choose_el(TB, LV);
  using S = Shape<TB, 0, TB, LV, TB - EL>;
  KernelEntry e;
  e.dtype = DT; e.kind = KIND_CLUSTER; e.K = TB + CL; e.TB = TB; e.TS = CL; e.col_bytes = 0;
  e.tma = 0; e.threads = S::NT; e.smem = (size_t)(KIND == 1 ? 8 : 4) << TB;
  e.launch = &launch_cluster<S, KIND, CL>;
  e.setup = &setup_cluster<S, KIND, CL>;
  e.selfcheck = [] { return check_shape<S, false>("cluster slice"); };
  e.fn = (const void*)&fwt_cluster_kernel<S, KIND, CL>;
  e.capacity = &cluster_capacity<S, KIND, CL>;
  return e;
}

template <int DT, typename T, class A, int NL>
KernelEntry small_entry() {
  KernelEntry e;
  e.dtype = DT; e.kind = KIND_SMALL; e.K = NL; e.TB = 0; e.TS = 0; e.col_bytes = 0; e.tma = 0;
  e.threads = 256; e.smem = 0;
  e.launch = &launch_small<T, A, NL>;
  e.setup = &setup_none;
  e.selfcheck = &selfcheck_none;
  e.fn = (const void*)&fwt_small_kernel<T, A, NL>;
  return e;
}

// fp64 diagonal phase, element by element (rows_c64.cu); sms sizes the grid.
cudaError_t launch_phase_apply_c64(const double* re_in, const double* im_in, const double* theta,
                                   long long theta_stride, double* re_out, double* im_out, int n,
                                   long long batch, int sms, cudaStream_t st);
// Fills the fp64 phase kernel's table on the current device (once per device).
cudaError_t setup_phase_table_c64();
cudaError_t read_device_error_c32(unsigned int* out);
// Records a failed CUDA call for fwt_last_cuda_error() (calling thread).
void set_last_cuda_error(int err);
cudaError_t launch_bounded_wait_probe(cudaStream_t st);
cudaError_t read_device_error_c64(unsigned int* out);
cudaError_t read_device_error_i32(unsigned int* out);
void register_rows_c32(std::vector<KernelEntry>& v);
void register_rows_c64(std::vector<KernelEntry>& v);
void register_rows_i32(std::vector<KernelEntry>& v);
void register_cols_c32(std::vector<KernelEntry>& v);
void register_cols_c64(std::vector<KernelEntry>& v);
void register_cols_i32(std::vector<KernelEntry>& v);

}  // namespace fwt
