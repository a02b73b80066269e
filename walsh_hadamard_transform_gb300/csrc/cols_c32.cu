// fp32 column passes.
#include "kernel_sets.cuh"

namespace fwt {
// Reads and clears this translation unit's device error word (synchronising).
cudaError_t read_device_error_c32(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(out, g_device_error, sizeof(unsigned int));
  if (err == cudaSuccess && *out) err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  return err;
}

// Self-test of the bounded wait: one CTA waits on a barrier that expects an
// arrival nobody makes (and no copy targets), so the wait must give up after
// about a second and record kErrTmaTimeout; nothing is left in flight.
__global__ void __launch_bounds__(32) fwt_bounded_wait_probe_kernel() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  __syncwarp();
  mbar_wait_bounded(&bar, 0);
}

// Launches the bounded-wait self-test (one CTA, about one second).
cudaError_t launch_bounded_wait_probe(cudaStream_t st) {
  fwt_bounded_wait_probe_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

void register_cols_c32(std::vector<KernelEntry>& v) { ColSet<FWT_C32, 0, 2, 15>::add(v); }
}  // namespace fwt
