// fp32 pass kernels (split complex fp32: each part is a real fp32 array).
#include "../../include/fwt.h"
#include "registry.cuh"

namespace fwt {
namespace {
template <int... Ks> void rows(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
  (v.push_back(row_entry<FWT_C32, 0, 2, Ks + 3>()), ...);
}
template <int CB, int K0, int... Ks> void cols(std::vector<KernelEntry>& v, std::integer_sequence<int, Ks...>) {
  (v.push_back(col_entry<FWT_C32, 0, 2, Ks + K0, CB, false>()), ...);
  (v.push_back(col_entry<FWT_C32, 0, 2, Ks + K0, CB, true>()), ...);
}
}  // namespace

// Reads and clears this translation unit's device error word (synchronising).
cudaError_t read_device_error_c32(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (err == cudaSuccess && *out) err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  return err;
}

void register_c32(std::vector<KernelEntry>& v) {
  v.push_back(small_entry<FWT_C32, float, ArithF32, 0>());
  v.push_back(small_entry<FWT_C32, float, ArithF32, 1>());
  v.push_back(small_entry<FWT_C32, float, ArithF32, 2>());
  rows(v, std::make_integer_sequence<int, 13>{});  // K = 3 .. 15
  cols<128, 5>(v, std::make_integer_sequence<int, 6>{});  // K = 5 .. 10
  cols<64, 6>(v, std::make_integer_sequence<int, 6>{});   // K = 6 .. 11
}
}  // namespace fwt
