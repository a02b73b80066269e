// C ABI of the batched Walsh-Hadamard transform: argument checks, the pass
// planner (Kronecker split of H_n into on-chip factors) and the launches.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fwt.h"
#include "registry.cuh"

namespace fwt {
namespace {

thread_local int g_last_cuda_error = 0;

// per-thread pass tracing into caller-owned events
thread_local void** g_trace_events = nullptr;
thread_local int g_trace_capacity = 0;
thread_local int g_trace_count = 0;

const std::vector<KernelEntry>& table() {
  static const std::vector<KernelEntry> t = [] {
    std::vector<KernelEntry> v;
    register_rows_c32(v);
    register_rows_c64(v);
    register_rows_i32(v);
    register_cols_c32(v);
    register_cols_c64(v);
    register_cols_i32(v);
    return v;
  }();
  return t;
}

// Kernels are found by (dtype, kind, K), column kernels also by segment width and
// mover, cluster kernels by their slice size (passed as col_bytes).  A planned call
// looks up tens of kernels, so the table is indexed once by that key.
uint64_t kernel_key(int dtype, int kind, int K, int col_bytes, int tma) {
  return (uint64_t)(uint32_t)dtype << 48 | (uint64_t)(uint32_t)kind << 40 |
         (uint64_t)(uint32_t)K << 32 | (uint64_t)(uint32_t)col_bytes << 8 | (uint64_t)(tma & 0xff);
}
uint64_t entry_key(const KernelEntry& e) {
  return kernel_key(e.dtype, e.kind, e.K, e.kind == KIND_COL ? e.col_bytes : e.kind == KIND_CLUSTER ? e.TB : 0,
                    e.kind == KIND_COL ? e.tma : 0);
}
const std::unordered_map<uint64_t, const KernelEntry*>& kernel_index() {
  static const std::unordered_map<uint64_t, const KernelEntry*> ix = [] {
    std::unordered_map<uint64_t, const KernelEntry*> m;
    for (const KernelEntry& e : table()) m.emplace(entry_key(e), &e);  // first entry wins
    return m;
  }();
  return ix;
}
const KernelEntry* find_kernel(int dtype, int kind, int K, int col_bytes = 0, int tma = 0) {
  const auto& ix = kernel_index();
  const auto it = ix.find(kernel_key(dtype, kind, K,
                                     kind == KIND_COL || kind == KIND_CLUSTER ? col_bytes : 0,
                                     kind == KIND_COL ? tma : 0));
  return it == ix.end() ? nullptr : it->second;
}

int elem_size(int dtype) { return dtype == FWT_C64 ? 8 : 4; }

// Whether a cluster kernel can run on the current device (cached per device).
std::mutex g_cap_mu;
std::vector<std::vector<signed char>> g_cap;  // [device][table index]: -1 unknown, 0 no, 1 yes
bool cluster_runnable(const KernelEntry* e);

// ---- plans -----------------------------------------------------------------------
// A plan is the list of Kronecker factors H_n = H_{f_last} (x) ... (x) H_{f_0}, each
// an on-chip pass over f_i consecutive index bits, lowest bits first.  Factor 0 is
// a row pass over contiguous memory, the others are column passes in place.
struct Plan {
  int nf = 0;
  int bits[3] = {0, 0, 0};
  int col_bytes = 128;  // width of the column passes' row segments
  int tma = 1;          // TMA-staged column passes: 0 never, 1 auto, 2 always
  int tma_mask = -1;    // auto, measured plans: factor f staged by TMA iff bit f is set
  const KernelEntry* cluster = nullptr;  // one-pass cluster kernel instead of the factors
};

// TMA staging pays for column tiles with many rows (long strided walks); short
// tiles are faster with plain vector loads (measured on GB300), unless a measured
// plan says otherwise for its factor f (f < 0: a pass outside the plan's factors).
// 16-byte segments exist only as TMA tiles.
int col_tma(const Plan& p, int f, int K) {
  if (p.tma == 2 || p.col_bytes == 16) return 1;
  if (p.tma == 0) return 0;
  if (p.tma_mask >= 0 && f >= 0) return (p.tma_mask >> f) & 1;
  return K >= 10 ? 1 : 0;
}

std::mutex g_plan_mu;
Plan g_override[3][31];  // nf == 0: no override
int g_col_bytes[3] = {0, 0, 0};  // column segment width per dtype; 0: chosen per plan
int default_col_bytes(int dtype) { return dtype == FWT_C64 ? 32 : 64; }
int g_use_tma = 1;                    // TMA-staged column passes: 0 never, 1 auto, 2 always
int g_use_cluster = 1;                // one-pass cluster kernels: 0 never, 1 auto, 2 from n = 14

int max_row_bits(int dtype) { return dtype == FWT_C64 ? 14 : 15; }
// column factors available for a segment width: tiles of 2^10 .. 2^15 (2^14 fp64) elements
int min_col_bits(int dtype, int cb) {
  return (dtype == FWT_C64 ? 6 : 5) + (cb == 64 ? 1 : cb == 32 ? 2 : cb == 16 ? 3 : 0);
}
int max_col_bits(int dtype, int cb) {
  return min_col_bits(dtype, cb) + (dtype == FWT_C64 ? 4 : 5);  // tiles up to 2^14 / 2^15
}

bool plan_valid(int n, int dtype, const Plan& p) {
  if (p.nf < 1 || p.nf > 3) return false;
  int sum = 0;
  for (int f = 0; f < p.nf; ++f) {
    const int k = p.bits[f];
    if (f == 0) {
      if (k <= 2) {
        if (p.nf != 1 || !find_kernel(dtype, KIND_SMALL, k)) return false;
      } else if (!find_kernel(dtype, KIND_ROW, k)) {
        return false;
      }
    } else {
      const KernelEntry* e = find_kernel(dtype, KIND_COL, k, p.col_bytes, col_tma(p, f, k));
      if (!e) return false;
      if (sum < e->TS) return false;  // a column segment must fit in one row
    }
    sum += k;
  }
  return sum == n;
}

// Splits measured faster than the general rule (GB300, a sweep of every two-factor
// split, column width and TMA mode at 2^26 elements a part for n <= 23, rechecked at
// 2^28 for n = 18..23, of every split and width at 2^28 for larger n, and of every
// fp64 three-factor split with TMA staging chosen per factor for n = 26..30).
//  * fp64 n = 15..22: a row factor of 9..12 bits and a column factor of 6..10 at 64-
//    or 128-byte segments, every column tile staged by TMA (the TMA column kernel runs
//    three CTAs an SM; the direct one two): passes of few bits are HBM-bound
//    (~6.7 TB/s), 15-25% faster than the general rule; n = 23: (12, 11) at 32 bytes.
//  * 4-byte n = 18..23: 128-byte column segments (2-4% faster; at n = 23 the 9-bit
//    column factor staged by TMA).
//  * 4-byte n = 25, 26: an 11-bit column factor at 32 bytes; from n = 27 three
//    passes with 128-byte column segments (each near 7 TB/s) beat two passes that
//    need narrow segments.
//  * fp64 from n = 25: tiles of 2^14 elements run one 512-thread CTA (or a CTA pair)
//    at about half the rate of the 2^13-element tiles, so from n = 26 three passes
//    over tiles of at most 2^13 elements win: a 12-bit row factor and two column
//    factors at 128 bytes, the middle one TMA-staged (~6.4 TB/s), the top one staged
//    where that measured faster (8-11% below the earlier per-plan TMA rule).
struct MeasuredSplit {
  bool fp64;
  int n, nf, bits[3], col_bytes;
  int tma_factors;  // column factors staged by TMA (bit f), when the TMA mode is
                    // auto; 0: the K >= 10 rule
};
constexpr MeasuredSplit kMeasuredSplits[] = {
    {true, 15, 2, {9, 6, 0}, 128, 0b10},    {true, 16, 2, {10, 6, 0}, 128, 0b10},
    {true, 17, 2, {10, 7, 0}, 128, 0b10},   {true, 18, 2, {10, 8, 0}, 128, 0b10},
    {true, 19, 2, {12, 7, 0}, 128, 0b10},   {true, 20, 2, {12, 8, 0}, 128, 0b10},
    {true, 21, 2, {12, 9, 0}, 64, 0b10},    {true, 22, 2, {12, 10, 0}, 64, 0b10},
    {true, 23, 2, {12, 11, 0}, 32, 0},
    {false, 18, 2, {12, 6, 0}, 128, 0}, {false, 19, 2, {13, 6, 0}, 128, 0},
    {false, 20, 2, {13, 7, 0}, 128, 0}, {false, 21, 2, {13, 8, 0}, 128, 0},
    {false, 22, 2, {14, 8, 0}, 128, 0}, {false, 23, 2, {14, 9, 0}, 128, 0b10},
    {false, 25, 2, {14, 11, 0}, 32, 0}, {false, 26, 2, {15, 11, 0}, 32, 0},
    {false, 27, 3, {12, 7, 8}, 128, 0}, {false, 28, 3, {13, 8, 7}, 128, 0},
    {false, 29, 3, {13, 8, 8}, 128, 0}, {false, 30, 3, {14, 8, 8}, 128, 0},
    {true, 25, 2, {14, 11, 0}, 32, 0},      {true, 26, 3, {12, 6, 8}, 128, 0b110},
    {true, 27, 3, {12, 8, 7}, 128, 0b010},  {true, 28, 3, {12, 8, 8}, 128, 0b010},
    {true, 29, 3, {12, 8, 9}, 128, 0b110},  {true, 30, 3, {12, 9, 9}, 128, 0b110},
};

Plan default_plan(int n, int dtype) {
  Plan p;
  int width;
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    width = g_col_bytes[dtype];
    p.tma = g_use_tma;
  }
  p.col_bytes = width ? width : default_col_bytes(dtype);
  if (width == 0) {
    for (const MeasuredSplit& ms : kMeasuredSplits) {
      if (ms.fp64 != (dtype == FWT_C64) || ms.n != n) continue;
      Plan q = p;
      q.nf = ms.nf;
      for (int f = 0; f < 3; ++f) q.bits[f] = ms.bits[f];
      q.col_bytes = ms.col_bytes;
      if (ms.tma_factors && q.tma == 1) q.tma_mask = ms.tma_factors;
      if (plan_valid(n, dtype, q)) return q;
    }
  }
  const int rmax = max_row_bits(dtype), cmin = min_col_bits(dtype, p.col_bytes),
            cmax = max_col_bits(dtype, p.col_bytes);
  if (n <= rmax) {
    p.nf = 1;
    p.bits[0] = n;
    return p;
  }
  // preferred row factor: 64 KiB row tiles for large n; smaller n splits near 12 + rest
  const int row_pref = n >= 22 ? (dtype == FWT_C64 ? 13 : 14) : 12;
  if (n <= rmax + cmax) {
    int a = std::min(std::max(cmin, n - row_pref), cmax);
    if (n - a > rmax) a = n - rmax;
    p.nf = 2;
    p.bits[0] = n - a;
    p.bits[1] = a;
    return p;
  }
  // three factors: a row factor and two column factors of about equal size
  const int b = std::min(row_pref, n - 2 * cmin);
  const int rest = n - b;
  p.nf = 3;
  p.bits[0] = b;
  p.bits[1] = (rest + 1) / 2;
  p.bits[2] = rest / 2;
  return p;
}

int cluster_mode() {
  std::lock_guard<std::mutex> lk(g_plan_mu);
  return g_use_cluster;
}

Plan get_plan(int n, int dtype) {
  int mode;
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    const Plan& o = g_override[dtype][n];
    if (o.nf > 0) return o;
    mode = g_use_cluster;
  }
  Plan p = default_plan(n, dtype);
  // a vector of 2^14 .. 2^18 4-byte elements in one pass on a thread-block cluster
  // (slices of 2^14, else 2^15 or 2^13).  Measured on GB300 against the factor
  // plans: faster for n = 16, 17 (clusters of 4 and 8 CTAs: 0.23 vs 0.32 ms and
  // 0.29 vs 0.32 ms at 2^26 elements), even at 15, slower at 18 (16-CTA clusters),
  // so the default uses it for n = 15 .. 17.
  const int lo_n = mode == 2 ? 14 : 15, hi_n = mode == 2 ? 18 : 17;
  if (dtype == FWT_C64 && mode > 0 && n == 14) {  // fp64: CTA pairs, 2^13-element slices
    const KernelEntry* e = find_kernel(dtype, KIND_CLUSTER, 14, 13);
    if (e && cluster_runnable(e)) p.cluster = e;
  }
  if (dtype != FWT_C64 && mode > 0 && n >= lo_n && n <= hi_n) {
    for (int tb : {14, 15, 13}) {
      if (n - tb < 1 || n - tb > 4) continue;
      const KernelEntry* e = find_kernel(dtype, KIND_CLUSTER, n, tb);
      if (e && cluster_runnable(e)) {
        p.cluster = e;
        break;
      }
    }
  }
  return p;
}

// ---- per-device set-up -------------------------------------------------------------
std::mutex g_dev_mu;
std::vector<char> g_dev_ready;
std::vector<long long> g_dev_l2;  // L2 bytes per device
std::vector<int> g_dev_sms;       // SMs per device
long long g_chunk_bytes = 0;       // -1: half the L2 of the current device; 0: off (default)

// SMs of the current device (0 before its set-up).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  return dev < (int)g_dev_sms.size() ? g_dev_sms[dev] : 0;
}

// How far ahead (in tiles) the staged kernels' L2 prefetch reaches: two tiles an SM,
// two thirds of a wave of the three-CTA-an-SM kernels (measured against one and
// more waves ahead: the fp64 n = 24 row pass 1.551 ms at two tiles an SM, 1.575 at
// three, 1.609 at four, 1.781 at six, 1.611 without prefetch).
int prefetch_ahead() { return 2 * device_sms(); }

long long chunk_budget() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_chunk_bytes >= 0) return g_chunk_bytes;
  return dev < (int)g_dev_l2.size() ? g_dev_l2[dev] / 2 : 0;
}

cudaError_t ensure_device() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if ((int)g_dev_ready.size() <= dev) g_dev_ready.resize(dev + 1, 0);
  if (g_dev_ready[dev]) return cudaSuccess;
  for (const KernelEntry& e : table()) {
    err = e.setup();
    if (err != cudaSuccess) return err;
  }
  err = setup_phase_table_c64();
  if (err != cudaSuccess) return err;
  int l2 = 0;
  err = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (err != cudaSuccess) return err;
  if ((int)g_dev_l2.size() <= dev) g_dev_l2.resize(dev + 1, 0);
  g_dev_l2[dev] = l2;
  int sms = 0;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  if ((int)g_dev_sms.size() <= dev) g_dev_sms.resize(dev + 1, 0);
  g_dev_sms[dev] = sms;
  g_dev_ready[dev] = 1;
  return cudaSuccess;
}

std::atomic<int> g_tma_promotion{128};
std::atomic<int> g_pdl{1};  // launch pass kernels with programmatic stream serialisation
std::once_flag g_encoder_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encoder = nullptr;

bool cluster_runnable(const KernelEntry* e) {
  int dev = 0;
  if (!e->capacity || cudaGetDevice(&dev) != cudaSuccess) return false;
  const size_t ix = (size_t)(e - table().data());
  std::lock_guard<std::mutex> lk(g_cap_mu);
  if ((int)g_cap.size() <= dev) g_cap.resize(dev + 1);
  if (g_cap[dev].size() < table().size()) g_cap[dev].resize(table().size(), -1);
  if (g_cap[dev][ix] < 0) {
    const bool ok = e->setup() == cudaSuccess && e->capacity() > 0;
    if (!ok) cudaGetLastError();
    g_cap[dev][ix] = ok ? 1 : 0;
  }
  return g_cap[dev][ix] == 1;
}

// floor(2^64 / sqrt(2)) = floor(sqrt(2^127)), by bitwise integer square root.
unsigned long long rsqrt2_q64() {
  const unsigned __int128 target = (unsigned __int128)1 << 127;
  unsigned __int128 r = 0;
  for (int bit = 63; bit >= 0; --bit) {
    const unsigned __int128 c = r | ((unsigned __int128)1 << bit);
    if (c * c <= target) r = c;
  }
  return (unsigned long long)r;
}

bool overlaps(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + bytes && y < x + bytes;
}
bool overlaps2(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + b_bytes && y < x + a_bytes;
}

// One launch of a pass kernel over the whole batch (or one chunk of it).
struct PassSpec {
  const KernelEntry* e;
  int L;        // column passes: log2 of the row stride
  int bits_lo;  // run-time bit-range row passes: first transformed tile bit
  int bits_k;   //   ... and how many
  uint32_t mask = 0;  // run-time row passes over a set of tile bits instead
};

// The column pass over bits [L, L + K): the plan's segment width when a tile
// shape exists for it, else another width, else (K <= 4) a wide-segment tile.
const KernelEntry* column_kernel(int dtype, int K, int L, const Plan& plan) {
  const int widths[5] = {plan.col_bytes, 128, 64, 32, 16};
  for (int cb : widths) {
    for (int tma : {col_tma(plan, -1, K), 1 - col_tma(plan, -1, K)}) {
      const KernelEntry* e = find_kernel(dtype, KIND_COL, K, cb, tma);
      if (e && L >= e->TS) return e;
    }
  }
  const int esz = elem_size(dtype);
  if (K <= 5) {  // short factors: wide segments of 2^(10-K) elements
    const KernelEntry* e = find_kernel(dtype, KIND_COL, K, (1 << (10 - K)) * esz, 0);
    if (e && L >= e->TS) return e;
  }
  return nullptr;
}

// A vector-load column kernel for K bits at row stride 2^L, preferring segments of
// `prefer` bytes, or nullptr (16-byte segments exist only as TMA tiles).
const KernelEntry* direct_column_kernel(int dtype, int K, int L, int prefer) {
  for (int cb : {prefer, 128, 64, 32}) {
    const KernelEntry* e = find_kernel(dtype, KIND_COL, K, cb, 0);
    if (e && L >= e->TS) return e;
  }
  if (K <= 5) {  // short factors: wide segments of 2^(10-K) elements
    const KernelEntry* e = find_kernel(dtype, KIND_COL, K, (1 << (10 - K)) * elem_size(dtype), 0);
    if (e && L >= e->TS) return e;
  }
  return nullptr;
}

// Column passes over bits [L, hi), in as few factors as the plan's segment width
// allows (near-equal sizes).
bool column_passes(int dtype, int L, int hi, const Plan& plan, std::vector<PassSpec>& out) {
  const int rest = hi - L;
  // fp64 column tiles of 2^14 elements run one 512-thread CTA an SM at about half
  // the rate of smaller ones: split into more factors instead (tiles <= 2^13)
  const int cmax = std::min(max_col_bits(dtype, plan.col_bytes),
                            dtype == FWT_C64 ? min_col_bits(dtype, plan.col_bytes) + 3 : 30);
  const int nf = (rest + cmax - 1) / cmax;
  for (int f = 0; f < nf; ++f) {
    const int K = rest / nf + (f < rest % nf ? 1 : 0);
    const KernelEntry* e = column_kernel(dtype, K, L, plan);
    if (!e) return false;
    out.push_back(PassSpec{e, L, 0, 0});
    L += K;
  }
  return true;
}

// Passes of the whole transform for a Kronecker plan (factor 0 = row pass).
// The kernel of a row pass over the low K bits.  fp64 row tiles of 2^14 elements
// run on a CTA pair (three CTAs an SM) rather than as one 512-thread CTA holding the
// whole tile, unless cluster kernels are off.
const KernelEntry* row_kernel(int dtype, int K) {
  if (dtype == FWT_C64 && K == 14 && cluster_mode() > 0) {
    const KernelEntry* c = find_kernel(dtype, KIND_CLUSTER, 14, 13);
    if (c && cluster_runnable(c)) return c;
  }
  return find_kernel(dtype, K <= 2 ? KIND_SMALL : KIND_ROW, K);
}

bool full_passes(int n, int dtype, const Plan& plan, std::vector<PassSpec>& out) {
  if (plan.cluster) {
    out.push_back(PassSpec{plan.cluster, 0, 0, 0});
    return true;
  }
  int L = 0;
  for (int f = 0; f < plan.nf; ++f) {
    const int K = plan.bits[f];
    PassSpec ps{nullptr, L, 0, 0};
    if (f == 0) ps.e = row_kernel(dtype, K);
    else ps.e = find_kernel(dtype, KIND_COL, K, plan.col_bytes, col_tma(plan, f, K));
    if (!ps.e) return false;
    out.push_back(ps);
    L += K;
  }
  return L == n;
}

// Passes of the transform over index bits [lo, lo + k) only.  From bit 0: a row
// pass (then column passes above the row tile); from a higher bit: column passes
// (rows 2^lo elements apart) when tile shapes exist for the factors, else a
// run-time bit-range row pass for the low part and column passes above it.
bool range_passes(int n, int dtype, int lo, int k, const Plan& plan, std::vector<PassSpec>& out) {
  const int rmax = max_row_bits(dtype);
  const int hi = lo + k;
  if (lo == 0 && k == n) return full_passes(n, dtype, plan, out);
  if (k == 0 || (hi <= rmax && (lo > 0 || k <= 2))) {  // one run-time bit-range row pass
    // tiles of at least 2^12 elements (128+ threads a CTA)
    const KernelEntry* e = find_kernel(dtype, KIND_ROWBITS, std::min(std::max(hi, 12), rmax));
    if (!e) return false;
    out.push_back(PassSpec{e, 0, lo, k});
    if (lo > 0 && k > 0) {  // prefer column passes when every factor has a tile shape
      std::vector<PassSpec> cols;
      if (column_passes(dtype, lo, hi, plan, cols)) out.swap(cols);
    }
    return true;
  }
  if (lo == 0) {  // row pass over the low bits, column passes above
    const int k0 = std::min(k, std::min(rmax, 13));
    const KernelEntry* e = find_kernel(dtype, KIND_ROW, k0);
    if (!e) return false;
    out.push_back(PassSpec{e, 0, 0, 0});
    return k0 == k || column_passes(dtype, k0, hi, plan, out);
  }
  if (column_passes(dtype, lo, hi, plan, out)) return true;
  out.clear();
  const int top = std::min(hi, rmax);  // bits [lo, top) in row tiles of 2^rmax elements
  const KernelEntry* e = find_kernel(dtype, KIND_ROWBITS, rmax);
  if (!e) return false;
  out.push_back(PassSpec{e, 0, lo, top - lo});
  return top == hi || column_passes(dtype, top, hi, plan, out);
}

// Passes of the transform over an arbitrary set of index bits (`mask`, below 2^n).
// One contiguous run is a bit range.  Otherwise the bits below the row-tile limit
// go to one run-time-mask row pass (tiles of 2^12 .. 2^rmax elements), and every
// run above it to column passes at its own stride.
bool mask_passes(int n, int dtype, uint32_t mask, const Plan& plan, std::vector<PassSpec>& out) {
  if (mask == 0) return range_passes(n, dtype, 0, 0, plan, out);
  const int lo = __builtin_ctz(mask), hi = 32 - __builtin_clz(mask);
  if (mask == (((hi >= 32 ? 0u : (1u << hi)) - 1u) & ~((1u << lo) - 1u)))
    return range_passes(n, dtype, lo, hi - lo, plan, out);
  const int rmax = max_row_bits(dtype);
  const uint32_t low = rmax >= 32 ? mask : mask & ((1u << rmax) - 1u);
  if (low) {
    const int top = 32 - __builtin_clz(low);
    const KernelEntry* e = find_kernel(dtype, KIND_ROWBITS, std::min(std::max(top, 12), rmax));
    if (!e) return false;
    PassSpec ps{e, 0, 0, 0};
    ps.mask = low;
    out.push_back(ps);
  }
  uint32_t high = mask & ~low;
  while (high) {  // each run [a, b) above the row tiles
    const int a = __builtin_ctz(high);
    int b = a;
    while (b < 32 && ((high >> b) & 1u)) ++b;
    if (!column_passes(dtype, a, b, plan, out)) return false;
    high &= b >= 32 ? 0u : ~((1u << b) - 1u);
  }
  return true;
}

// FWT_LOG set (and not "0") in the environment: every transform call prints its
// passes to stderr, one line a call (read once per process).
bool log_plans() {
  static const bool on = [] {
    const char* v = std::getenv("FWT_LOG");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

void log_plan(const char* what, int dtype, int n, int64_t batch, const std::vector<PassSpec>& passes) {
  static const char* const kDtype[3] = {"c32", "c64", "i32"};
  static const char* const kKind[6] = {"small", "row", "col", "rowbits", "phase", "cluster"};
  char line[512];
  int len = snprintf(line, sizeof line, "fwt: %s %s n=%d batch=%lld passes=%d", what,
                     kDtype[dtype], n, (long long)batch, (int)passes.size());
  for (const PassSpec& ps : passes) {
    const KernelEntry* e = ps.e;
    if (len < 0 || len >= (int)sizeof line) break;
    len += snprintf(line + len, sizeof line - len, " | %s K=%d tile=2^%d", kKind[e->kind], e->K,
                    e->TB);
    if (len < (int)sizeof line && e->kind == KIND_COL)
      len += snprintf(line + len, sizeof line - len, " stride=2^%d %dB %s", ps.L, e->col_bytes,
                      e->tma ? "tma" : "direct");
    if (len < (int)sizeof line && e->kind == KIND_CLUSTER)
      len += snprintf(line + len, sizeof line - len, " ctas=%d", 1 << e->TS);
    if (len < (int)sizeof line && e->kind == KIND_ROWBITS) {
      if (ps.mask)
        len += snprintf(line + len, sizeof line - len, " mask=0x%x", ps.mask);
      else
        len += snprintf(line + len, sizeof line - len, " bits=[%d,%d)", ps.bits_lo,
                        ps.bits_lo + ps.bits_k);
    }
  }
  fprintf(stderr, "%s\n", line);
}

int check_arrays(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out,
                 int n, int64_t batch, bool& has_im) {
  const int esz = elem_size(dtype);
  if (batch > (INT64_MAX >> n) / esz) return FWT_ERR_INVALID_ARG;
  const size_t bytes = (size_t)(((long long)batch << n) * esz);
  // pointers: real part required; imaginary part both-or-neither (NULL only for int32)
  if (!re_in || !re_out) return FWT_ERR_INVALID_ARG;
  has_im = im_in || im_out;
  if (has_im && (!im_in || !im_out)) return FWT_ERR_INVALID_ARG;
  if (!has_im && dtype != FWT_I32) return FWT_ERR_INVALID_ARG;
  const void* ptrs[4] = {re_in, im_in, re_out, im_out};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u)) return FWT_ERR_MISALIGNED;
  // outputs may coincide exactly with their own input, and with nothing else
  if (overlaps(re_out, re_in, bytes) && re_out != re_in) return FWT_ERR_INVALID_ARG;
  if (has_im) {
    if (overlaps(im_out, im_in, bytes) && im_out != im_in) return FWT_ERR_INVALID_ARG;
    if (overlaps(re_out, im_out, bytes) || overlaps(re_out, im_in, bytes) ||
        overlaps(im_out, re_in, bytes))
      return FWT_ERR_INVALID_ARG;
  }
  return FWT_OK;
}

// Runs the transform over bits [lo, lo + k) of each vector (the whole transform
// when lo = 0, k = n), scaled by 2^{-k/2} when normalising.
int run(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out, int n,
        int64_t batch, int lo, int k, int normalize, cudaStream_t stream, uint32_t mask = 0) {
  if (n < 0 || n > 30 || batch < 0 || lo < 0 || k < 0 || lo + k > n) return FWT_ERR_INVALID_ARG;
  if (mask && (n < 32 && (mask >> n) != 0)) return FWT_ERR_INVALID_ARG;
  if (dtype == FWT_I32 && normalize) return FWT_ERR_UNSUPPORTED;
  if (batch == 0) return FWT_OK;
  bool has_im = false;
  int st = check_arrays(dtype, re_in, im_in, re_out, im_out, n, batch, has_im);
  if (st != FWT_OK) return st;
  const int esz = elem_size(dtype);
  const bool whole = lo == 0 && k == n;
  cudaError_t err = ensure_device();
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    return FWT_ERR_CUDA;
  }
  Plan plan = whole ? get_plan(n, dtype) : default_plan(n, dtype);
  if (whole && !plan.cluster && !plan_valid(n, dtype, plan)) return FWT_ERR_UNSUPPORTED;
  if (plan.tma && !tensor_map_encoder()) plan.tma = 0;  // driver without the TMA encoder
  std::vector<PassSpec> passes;
  if (mask) {
    if (!mask_passes(n, dtype, mask, plan, passes)) return FWT_ERR_UNSUPPORTED;
    k = __builtin_popcount(mask);  // the normalisation counts the transformed bits
  } else if (!range_passes(n, dtype, lo, k, plan, passes)) {
    return FWT_ERR_UNSUPPORTED;
  }

  // TMA-staged column tiles run in place.  An out-of-place call whose first pass is
  // one loads that pass with 16-byte vectors where a tile shape exists for it; else
  // (16-byte segments below the row stride: TMA tiles only) a row pass over no bits
  // first copies the input into the output, and the column pass runs there in place.
  const bool call_in_place = re_in == re_out && (!has_im || im_in == im_out);
  if (!call_in_place && !passes.empty() && passes[0].e->kind == KIND_COL && passes[0].e->tma) {
    const KernelEntry* d =
        direct_column_kernel(dtype, passes[0].e->K, passes[0].L, passes[0].e->col_bytes);
    if (d) {
      passes[0].e = d;
    } else {
      const KernelEntry* copy = find_kernel(dtype, KIND_ROWBITS, 12);
      if (!copy) return FWT_ERR_UNSUPPORTED;
      passes.insert(passes.begin(), PassSpec{copy, 0, 0, 0});
    }
  }

  if (log_plans())
    log_plan(mask ? "mask" : (whole ? "transform" : "bits"), dtype, n, batch, passes);

  PassParams p{};
  const int ahead = prefetch_ahead();
  const double s = k % 2 == 0 ? std::ldexp(1.0, -k / 2) : std::ldexp(1.0, -(k - 1) / 2) / std::sqrt(2.0);
  p.scale_f64 = s;
  p.scale_f32 = (float)s;
  p.scale_exp = -(k / 2);
  p.scale_half = k % 2;
  p.rsqrt2_q64 = rsqrt2_q64();

  // L2 chunking (opt-in): a multi-pass transform runs all its passes on one
  // group of vectors before the next, so the intermediate written by a pass can
  // be read back from L2 by the next one.  A group is as many whole vectors as
  // fit the chunk budget; both parts share a launch when a vector pair fits, else
  // the parts are chunked one at a time.  On GB300 the extra, smaller launches
  // cost more than the L2 reuse saves for the specified workloads, so it is off
  // by default.
  const int ncomp_all = has_im ? 2 : 1;
  const long long vec_bytes = (long long)esz << n;
  const long long budget = chunk_budget();
  long long vpc = batch;  // vectors per chunk
  int parts_per_launch = ncomp_all;
  bool chunked = false;
  const int npass = (int)passes.size();
  if (npass >= 2 && budget > 0) {
    if ((long long)ncomp_all * vec_bytes <= budget) {
      vpc = std::max(1ll, budget / (ncomp_all * vec_bytes));
    } else if (vec_bytes <= budget) {
      parts_per_launch = 1;
      vpc = std::max(1ll, budget / vec_bytes);
    }
    chunked = vpc < batch || parts_per_launch < ncomp_all;
  }
  const void* ins[2] = {re_in, im_in};
  void* outs[2] = {re_out, im_out};
  for (int part0 = 0; part0 < ncomp_all; part0 += parts_per_launch) {
    for (long long v0 = 0; v0 < batch; v0 += vpc) {
      const long long nv = std::min(vpc, batch - v0);
      const long long off = (v0 << n) * esz;  // byte offset of the chunk
      const long long elems = nv << n;
      for (int f = 0; f < npass; ++f) {
        const PassSpec& ps = passes[f];
        const KernelEntry* e = ps.e;
        long long tiles;
        if (e->kind == KIND_SMALL) tiles = ((elems >> e->K) + 255) / 256;
        else if (e->kind == KIND_COL || e->kind == KIND_CLUSTER) tiles = elems >> e->TB;
        else tiles = (elems + (1ll << e->TB) - 1) >> e->TB;
        if (tiles > INT_MAX) return FWT_ERR_UNSUPPORTED;
        p.comp_elems = elems;
        bool in_place = true;
        for (int c = 0; c < 2; ++c) {
          const int part = part0 + (c < parts_per_launch ? c : 0);
          const char* src = (const char*)(f == 0 ? ins[part] : outs[part]);
          p.in[c] = src ? src + off : nullptr;
          p.out[c] = outs[part] ? (char*)outs[part] + off : nullptr;
          in_place &= p.in[c] == p.out[c];
        }
        if (e->tma && !in_place) return FWT_ERR_UNSUPPORTED;  // planned away above
        p.stride_log = ps.L;
        p.bits_lo = ps.bits_lo;
        p.bits_k = ps.bits_k;
        p.bits_mask = ps.mask;
        const bool last = f == npass - 1;
        p.do_scale = (normalize && last) ? 1 : 0;
        p.ld_policy = 0;                             // normal (evict-first measured slower)
        p.st_policy = last ? 1 : (chunked ? 2 : 0);  // keep intermediates for the next pass
        p.bulk = plan.tma != 0 ? 1 : 0;              // bulk-copied fp64 row tiles
        p.prefetch_ahead = ahead;
        const bool traced = g_trace_count + 2 <= g_trace_capacity;
        if (traced) {
          err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count], stream);
          if (err != cudaSuccess) {
            g_last_cuda_error = (int)err;
            return FWT_ERR_CUDA;
          }
        }
        err = e->launch(p, tiles, parts_per_launch, stream);
        if (err == cudaSuccess && traced) {
          err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count + 1], stream);
          g_trace_count += 2;
        }
        if (err != cudaSuccess) {
          g_last_cuda_error = (int)err;
          return FWT_ERR_CUDA;
        }
      }
    }
  }
  return FWT_OK;
}

// y = s * H (e^{i theta} . x), fp64: the phase element by element into the outputs
// (double sincos on the fp64 unit; fusing it into the fixed-point row pass would
// make the CTAs of both parts evaluate every sine and cosine), then the fp64
// transform in place.
int run_phase_c64(const double* re_in, const double* im_in, const double* theta,
                  int64_t theta_stride, double* re_out, double* im_out, int n, int64_t batch,
                  int normalize, cudaStream_t stream) {
  if (n < 0 || n > 30 || batch < 0 || theta_stride < 0) return FWT_ERR_INVALID_ARG;
  if (batch == 0) return FWT_OK;
  if (!im_in || !im_out || !theta) return FWT_ERR_INVALID_ARG;
  bool has_im = false;
  int st = check_arrays(FWT_C64, re_in, im_in, re_out, im_out, n, batch, has_im);
  if (st != FWT_OK) return st;
  if ((uintptr_t)theta & 15u) return FWT_ERR_MISALIGNED;
  if (n >= 1 && theta_stride % 2 != 0) return FWT_ERR_MISALIGNED;  // 16-byte angle pairs
  if (batch > 1 && theta_stride > (INT64_MAX / 8 - (1ll << n)) / (batch - 1))
    return FWT_ERR_INVALID_ARG;  // the angles' extent would overflow
  const long long th_elems = (theta_stride == 0 ? 0 : (long long)(batch - 1)) * theta_stride + (1ll << n);
  const size_t th_bytes = (size_t)th_elems * 8;
  const size_t bytes = (size_t)((long long)batch << n) * 8;
  if (overlaps2(theta, th_bytes, re_out, bytes) || overlaps2(theta, th_bytes, im_out, bytes))
    return FWT_ERR_INVALID_ARG;
  cudaError_t err = ensure_device();
  const int sms = device_sms();
  const bool traced = g_trace_count + 2 <= g_trace_capacity;
  if (err == cudaSuccess && traced)
    err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count], stream);
  if (err == cudaSuccess)
    err = launch_phase_apply_c64(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch, sms,
                                 stream);
  if (err == cudaSuccess && traced) {
    err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count + 1], stream);
    g_trace_count += 2;
  }
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    return FWT_ERR_CUDA;
  }
  return run(FWT_C64, re_out, im_out, re_out, im_out, n, batch, 0, n, normalize, stream);
}

// y = s * H (e^{i theta} . x), fp32: a fused phase + row pass over the low
// min(n, 13) bits, then in-place column passes over the rest.
int run_phase(const float* re_in, const float* im_in, const float* theta, int64_t theta_stride,
              float* re_out, float* im_out, int n, int64_t batch, int normalize,
              cudaStream_t stream) {
  if (n < 0 || n > 30 || batch < 0 || theta_stride < 0) return FWT_ERR_INVALID_ARG;
  if (batch == 0) return FWT_OK;
  if (!im_in || !im_out || !theta) return FWT_ERR_INVALID_ARG;
  bool has_im = false;
  int st = check_arrays(FWT_C32, re_in, im_in, re_out, im_out, n, batch, has_im);
  if (st != FWT_OK) return st;
  if ((uintptr_t)theta & 15u) return FWT_ERR_MISALIGNED;
  if (n >= 2 && theta_stride % 4 != 0) return FWT_ERR_MISALIGNED;  // 16-byte angle vectors
  if (batch > 1 && theta_stride > (INT64_MAX / 4 - (1ll << n)) / (batch - 1))
    return FWT_ERR_INVALID_ARG;  // the angles' extent would overflow
  const long long th_elems = (theta_stride == 0 ? 0 : (long long)(batch - 1)) * theta_stride + (1ll << n);
  const size_t th_bytes = (size_t)th_elems * 4;
  const size_t bytes = (size_t)((long long)batch << n) * 4;
  // the angles are read while the outputs are written: no overlap (either way round)
  if (overlaps2(theta, th_bytes, re_out, bytes) || overlaps2(theta, th_bytes, im_out, bytes))
    return FWT_ERR_INVALID_ARG;
  cudaError_t err = ensure_device();
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    return FWT_ERR_CUDA;
  }
  Plan plan = default_plan(n, FWT_C32);
  if (plan.tma && !tensor_map_encoder()) plan.tma = 0;
  const int k1 = std::min(n, 13);
  {
    // the fused first pass covers 13 bits, so 11- and 12-bit column factors follow;
    // at 64-byte segments they need 512-thread tiles, at 32 bytes 256 (measured 1.07
    // vs 0.82 ms at n = 24, batch 16)
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_col_bytes[FWT_C32] == 0 && n - k1 >= 11 && n - k1 <= 12) plan.col_bytes = 32;
  }
  std::vector<PassSpec> passes;
  const KernelEntry* e0 = find_kernel(FWT_C32, KIND_PHASE, k1);
  if (!e0) return FWT_ERR_UNSUPPORTED;
  passes.push_back(PassSpec{e0, 0, 0, 0});
  if (n > k1 && !column_passes(FWT_C32, k1, n, plan, passes)) return FWT_ERR_UNSUPPORTED;
  if (log_plans()) log_plan("phase", FWT_C32, n, batch, passes);

  PassParams p{};
  const double s = n % 2 == 0 ? std::ldexp(1.0, -n / 2) : std::ldexp(1.0, -(n - 1) / 2) / std::sqrt(2.0);
  p.scale_f64 = s;
  p.scale_f32 = (float)s;
  p.scale_exp = -(n / 2);
  p.scale_half = n % 2;
  p.rsqrt2_q64 = rsqrt2_q64();
  p.theta = theta;
  p.theta_stride = theta_stride;
  p.n = n;
  const long long elems = (long long)batch << n;
  p.comp_elems = elems;
  const int npass = (int)passes.size();
  for (int f = 0; f < npass; ++f) {
    const KernelEntry* e = passes[f].e;
    long long tiles;
    if (e->kind == KIND_PHASE && e->K <= 2) tiles = ((elems >> e->K) + 255) / 256;
    else if (e->kind == KIND_COL) tiles = elems >> e->TB;
    else tiles = (elems + (1ll << e->TB) - 1) >> e->TB;
    if (tiles > INT_MAX) return FWT_ERR_UNSUPPORTED;
    p.in[0] = f == 0 ? (const void*)re_in : re_out;
    p.in[1] = f == 0 ? (const void*)im_in : im_out;
    p.out[0] = re_out;
    p.out[1] = im_out;
    p.stride_log = passes[f].L;
    const bool last = f == npass - 1;
    p.do_scale = (normalize && last) ? 1 : 0;
    p.ld_policy = 0;
    p.st_policy = last ? 1 : 0;
    const bool traced = g_trace_count + 2 <= g_trace_capacity;
    if (traced) {
      err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count], stream);
      if (err != cudaSuccess) {
        g_last_cuda_error = (int)err;
        return FWT_ERR_CUDA;
      }
    }
    err = e->launch(p, tiles, 2, stream);
    if (err == cudaSuccess && traced) {
      err = cudaEventRecord((cudaEvent_t)g_trace_events[g_trace_count + 1], stream);
      g_trace_count += 2;
    }
    if (err != cudaSuccess) {
      g_last_cuda_error = (int)err;
      return FWT_ERR_CUDA;
    }
  }
  return FWT_OK;
}

}  // namespace

int tma_l2_promotion() { return g_tma_promotion.load(); }
int pdl_mode() { return g_pdl.load(std::memory_order_relaxed); }
void set_last_cuda_error(int err) { g_last_cuda_error = err; }

bool tensor_map_2d(CUtensorMap* out, CUtensorMapDataType dt, void* base, const cuuint64_t dims[2],
                   cuuint64_t row_stride_bytes, const cuuint32_t box[2], int l2_promotion) {
  struct Entry {
    bool valid;
    CUtensorMapDataType dt;
    void* base;
    cuuint64_t dims[2], stride;
    cuuint32_t box[2];
    int promo;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (Entry& e : cache)
    if (e.valid && e.dt == dt && e.base == base && e.dims[0] == dims[0] && e.dims[1] == dims[1] &&
        e.stride == row_stride_bytes && e.box[0] == box[0] && e.box[1] == box[1] &&
        e.promo == l2_promotion) {
      *out = e.map;
      return true;
    }
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const CUtensorMapL2promotion prom = l2_promotion == 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                      : l2_promotion == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                      : l2_promotion == 64  ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                                            : CU_TENSOR_MAP_L2_PROMOTION_NONE;
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(out, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, prom, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.valid = true;
  e.dt = dt;
  e.base = base;
  e.dims[0] = dims[0];
  e.dims[1] = dims[1];
  e.stride = row_stride_bytes;
  e.box[0] = box[0];
  e.box[1] = box[1];
  e.promo = l2_promotion;
  e.map = *out;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encoder_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encoder = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encoder;
}

}  // namespace fwt

namespace fwt {
namespace {
// A set of bits: one contiguous run goes the bit-range way (the whole transform
// included), anything else through mask_passes.
int run_mask(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out, int n,
             int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream) {
  if (n < 0 || n > 30) return FWT_ERR_INVALID_ARG;
  if ((mask >> n) != 0) return FWT_ERR_INVALID_ARG;
  if (mask != 0) {  // one contiguous run is a bit range (the whole transform included)
    const int lo = __builtin_ctz(mask), hi = 32 - __builtin_clz(mask);
    if (mask == (((hi >= 32 ? 0u : (1u << hi)) - 1u) & ~((1u << lo) - 1u)))
      return run(dtype, re_in, im_in, re_out, im_out, n, batch, lo, hi - lo, normalize,
                      (cudaStream_t)stream);
  }
  return run(dtype, re_in, im_in, re_out, im_out, n, batch, 0, 0, normalize,
                  (cudaStream_t)stream, mask);
}
}  // namespace
}  // namespace fwt

extern "C" {

int fwt_batched_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                    int64_t batch, int normalize, fwt_stream_t stream) {
  if (n < 0 || n > 30) return FWT_ERR_INVALID_ARG;
  return fwt::run(FWT_C32, re_in, im_in, re_out, im_out, n, batch, 0, n, normalize,
                  (cudaStream_t)stream);
}

int fwt_batched_c64(const double* re_in, const double* im_in, double* re_out, double* im_out,
                    int n, int64_t batch, int normalize, fwt_stream_t stream) {
  if (n < 0 || n > 30) return FWT_ERR_INVALID_ARG;
  return fwt::run(FWT_C64, re_in, im_in, re_out, im_out, n, batch, 0, n, normalize,
                  (cudaStream_t)stream);
}

int fwt_batched_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                    int n, int64_t batch, int normalize, fwt_stream_t stream) {
  if (n < 0 || n > 30) return FWT_ERR_INVALID_ARG;
  return fwt::run(FWT_I32, re_in, im_in, re_out, im_out, n, batch, 0, n, normalize,
                  (cudaStream_t)stream);
}

int fwt_bits_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream) {
  return fwt::run(FWT_C32, re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize,
                  (cudaStream_t)stream);
}

int fwt_bits_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream) {
  return fwt::run(FWT_C64, re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize,
                  (cudaStream_t)stream);
}

int fwt_bits_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream) {
  return fwt::run(FWT_I32, re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize,
                  (cudaStream_t)stream);
}

int fwt_mask_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream) {
  return fwt::run_mask(FWT_C32, re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream);
}

int fwt_mask_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream) {
  return fwt::run_mask(FWT_C64, re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream);
}

int fwt_mask_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream) {
  return fwt::run_mask(FWT_I32, re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream);
}

int fwt_phase_c64(const double* re_in, const double* im_in, const double* theta,
                  int64_t theta_stride, double* re_out, double* im_out, int n, int64_t batch,
                  int normalize, fwt_stream_t stream) {
  return fwt::run_phase_c64(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch,
                            normalize, (cudaStream_t)stream);
}

int fwt_phase_c32(const float* re_in, const float* im_in, const float* theta,
                  int64_t theta_stride, float* re_out, float* im_out, int n, int64_t batch,
                  int normalize, fwt_stream_t stream) {
  return fwt::run_phase(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch, normalize,
                        (cudaStream_t)stream);
}

const char* fwt_status_string(int status) {
  switch (status) {
    case FWT_OK: return "ok";
    case FWT_ERR_INVALID_ARG: return "invalid argument";
    case FWT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FWT_ERR_UNSUPPORTED: return "unsupported";
    case FWT_ERR_CUDA: return "CUDA error";
    case FWT_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int fwt_last_cuda_error(void) { return fwt::g_last_cuda_error; }

int fwt_plan_factors(int n, int dtype, int* bits, int max_factors) {
  if (n < 0 || n > 30 || dtype < 0 || dtype > 2) return -1;
  fwt::Plan p = fwt::get_plan(n, dtype);
  if (p.cluster) {  // one pass over the whole vector
    p.nf = 1;
    p.bits[0] = n;
  }
  for (int f = 0; f < p.nf && f < max_factors; ++f) bits[f] = p.bits[f];
  return p.nf;
}

int fwt_plan_passes(int n, int dtype) { return fwt_plan_factors(n, dtype, nullptr, 0); }

int fwt_set_plan(int n, int dtype, int nfactors, const int* bits) {
  if (n < 0 || n > 30 || dtype < 0 || dtype > 2 || nfactors < 0 || nfactors > 3)
    return FWT_ERR_INVALID_ARG;
  fwt::Plan p;
  p.nf = nfactors;
  int width;
  {
    std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
    width = fwt::g_col_bytes[dtype];
    p.tma = fwt::g_use_tma;
  }
  for (int f = 0; f < nfactors; ++f) {
    if (!bits) return FWT_ERR_INVALID_ARG;
    p.bits[f] = bits[f];
  }
  if (nfactors > 0) {
    // the width set for the dtype, else the first width with tiles for every factor
    bool ok = false;
    for (int cb : {width ? width : fwt::default_col_bytes(dtype), 32, 16, 64, 128}) {
      p.col_bytes = cb;
      if ((ok = fwt::plan_valid(n, dtype, p)) || width) break;
    }
    if (!ok) return FWT_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  fwt::g_override[dtype][n] = p;
  return FWT_OK;
}

int fwt_set_column_bytes(int dtype, int bytes) {
  if (dtype < 0 || dtype > 2 ||
      (bytes != 0 && bytes != 16 && bytes != 32 && bytes != 64 && bytes != 128))
    return FWT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  fwt::g_col_bytes[dtype] = bytes;
  return FWT_OK;
}

int fwt_get_column_bytes(int dtype) {
  if (dtype < 0 || dtype > 2) return -1;
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  return fwt::g_col_bytes[dtype];
}

int fwt_set_tma(int mode) {
  if (mode < 0 || mode > 2) return FWT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  fwt::g_use_tma = mode;
  return FWT_OK;
}

int fwt_set_cluster(int mode) {
  if (mode < 0 || mode > 2) return FWT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  fwt::g_use_cluster = mode;
  return FWT_OK;
}

int fwt_get_cluster(void) {
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  return fwt::g_use_cluster;
}

int fwt_set_tma_l2_promotion(int bytes) {
  if (bytes != 0 && bytes != 64 && bytes != 128 && bytes != 256) return FWT_ERR_INVALID_ARG;
  fwt::g_tma_promotion.store(bytes);
  return FWT_OK;
}

int fwt_set_pdl(int mode) {
  if (mode < 0 || mode > 1) return FWT_ERR_INVALID_ARG;
  fwt::g_pdl.store(mode);
  return FWT_OK;
}

int fwt_get_pdl(void) { return fwt::g_pdl.load(); }

int fwt_get_tma(void) {
  std::lock_guard<std::mutex> lk(fwt::g_plan_mu);
  return fwt::g_use_tma;
}

int fwt_selftest_bounded_wait(fwt_stream_t stream) {
  cudaError_t err = fwt::ensure_device();
  if (err == cudaSuccess) err = fwt::launch_bounded_wait_probe((cudaStream_t)stream);
  if (err != cudaSuccess) {
    fwt::g_last_cuda_error = (int)err;
    return FWT_ERR_CUDA;
  }
  return FWT_OK;
}

int fwt_device_status(void) {
  unsigned int e[3] = {0, 0, 0};
  cudaError_t err = fwt::read_device_error_c32(&e[0]);
  if (err == cudaSuccess) err = fwt::read_device_error_c64(&e[1]);
  if (err == cudaSuccess) err = fwt::read_device_error_i32(&e[2]);
  if (err != cudaSuccess) {
    fwt::g_last_cuda_error = (int)err;
    return FWT_ERR_CUDA;
  }
  return (e[0] | e[1] | e[2]) ? FWT_ERR_TIMEOUT : FWT_OK;
}

int fwt_set_l2_chunk_bytes(long long bytes) {
  if (bytes < -1) return FWT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(fwt::g_dev_mu);
  fwt::g_chunk_bytes = bytes;
  return FWT_OK;
}

long long fwt_get_l2_chunk_bytes(void) {
  std::lock_guard<std::mutex> lk(fwt::g_dev_mu);
  return fwt::g_chunk_bytes;
}

int fwt_trace_events(void** events, int capacity) {
  if (capacity < 0 || (capacity > 0 && !events)) return FWT_ERR_INVALID_ARG;
  fwt::g_trace_events = capacity > 0 ? events : nullptr;
  fwt::g_trace_capacity = capacity;
  fwt::g_trace_count = 0;
  return FWT_OK;
}

int fwt_trace_count(void) { return fwt::g_trace_count; }

int fwt_selfcheck(void) {
  int fails = 0;
  for (const fwt::KernelEntry& e : fwt::table()) fails += e.selfcheck();
  // the kernel index returns, for every entry's key, the first table entry with it
  for (const fwt::KernelEntry& e : fwt::table()) {
    const int cb = e.kind == fwt::KIND_COL ? e.col_bytes : e.kind == fwt::KIND_CLUSTER ? e.TB : 0;
    const fwt::KernelEntry* first = nullptr;
    for (const fwt::KernelEntry& f : fwt::table())
      if (fwt::entry_key(f) == fwt::entry_key(e)) {
        first = &f;
        break;
      }
    if (fwt::find_kernel(e.dtype, e.kind, e.K, cb, e.tma) != first) {
      fprintf(stderr, "fwt_selfcheck: kernel index disagrees with the table\n");
      ++fails;
    }
  }
  for (int dt = 0; dt < 3; ++dt)
    for (int n = 0; n <= 30; ++n)
      if (!fwt::plan_valid(n, dt, fwt::default_plan(n, dt))) {
        fprintf(stderr, "fwt_selfcheck: no valid default plan for n=%d dtype=%d\n", n, dt);
        ++fails;
      }
  return fails;
}

}  // extern "C"
