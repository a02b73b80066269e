// fp64 pass kernels: exact int64 fixed-point butterflies (IEEE fp64 for tiles with Inf/NaN).
#include "../../include/fwt.h"
#include "registry.cuh"

namespace fwt {
namespace {
template <int... Ks> void rows(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
  (v.push_back(row_entry<FWT_C64, 1, 1, Ks + 3>()), ...);
}
template <int CB, int K0, int... Ks> void cols(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
  (v.push_back(col_entry<FWT_C64, 1, 1, Ks + K0, CB, false>()), ...);
  (v.push_back(col_entry<FWT_C64, 1, 1, Ks + K0, CB, true>()), ...);
}
}  // namespace

// Reads and clears this translation unit's device error word (synchronising).
cudaError_t read_device_error_c64(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (err == cudaSuccess && *out) err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  return err;
}

void register_c64(std::vector<KernelEntry>& v) {
  v.push_back(small_entry<FWT_C64, double, ArithF64, 0>());
  v.push_back(small_entry<FWT_C64, double, ArithF64, 1>());
  v.push_back(small_entry<FWT_C64, double, ArithF64, 2>());
  rows(v, std::make_integer_sequence<int, 12>{});  // K = 3 .. 14
  cols<128, 6>(v, std::make_integer_sequence<int, 5>{});  // K = 6 .. 10
  cols<64, 7>(v, std::make_integer_sequence<int, 5>{});   // K = 7 .. 11
  cols<32, 8>(v, std::make_integer_sequence<int, 5>{});   // K = 8 .. 12
}
}  // namespace fwt
