// fp64 column passes.
#include "kernel_sets.cuh"

namespace fwt {
// Reads and clears this translation unit's device error word (synchronising).
cudaError_t read_device_error_c64(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (err == cudaSuccess && *out) err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  return err;
}

void register_cols_c64(std::vector<KernelEntry>& v) { ColSet<FWT_C64, 1, 1, 14>::add(v); }
}  // namespace fwt
