// fp64 row passes (int64 fixed-point butterflies).
#include <algorithm>

#include "kernel_sets.cuh"

namespace fwt {

// Diagonal phase for fp64 split complex vectors, element by element and in place
// or out of place: (re, im) <- (re cos t - im sin t, re sin t + im cos t) with
// (sin t, cos t) from the double-precision sincos.  16-byte vectors of two
// elements; a grid-stride loop over all pairs of the batch.
__global__ void __launch_bounds__(256) fwt_phase_apply_c64_kernel(
    const double* re_in, const double* im_in, const double* theta, long long theta_stride,
    double* re_out, double* im_out,
    int n, long long pairs) {
  pdl_begin();
  const long long nmask = (1ll << n) - 1;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < pairs;
       q += (long long)gridDim.x * blockDim.x) {
    const long long e = q * 2;  // first element of the pair (n >= 1: both in one vector)
    const double2 r = *reinterpret_cast<const double2*>(re_in + e);
    const double2 m = *reinterpret_cast<const double2*>(im_in + e);
    const long long t = (e >> n) * theta_stride + (e & nmask);
    const double2 th = *reinterpret_cast<const double2*>(theta + t);
    double s0, c0, s1, c1;
    sincos(th.x, &s0, &c0);
    sincos(th.y, &s1, &c1);
    *reinterpret_cast<double2*>(re_out + e) = make_double2(r.x * c0 - m.x * s0, r.y * c1 - m.y * s1);
    *reinterpret_cast<double2*>(im_out + e) = make_double2(r.x * s0 + m.x * c0, r.y * s1 + m.y * c1);
  }
}

// n = 0: one element a vector.
__global__ void __launch_bounds__(256) fwt_phase_apply_c64_scalar_kernel(
    const double* re_in, const double* im_in, const double* theta, long long theta_stride,
    double* re_out, double* im_out, long long count) {
  pdl_begin();
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < count;
       e += (long long)gridDim.x * blockDim.x) {
    double s, c;
    sincos(theta[e * theta_stride], &s, &c);
    const double r = re_in[e], m = im_in[e];
    re_out[e] = r * c - m * s;
    im_out[e] = r * s + m * c;
  }
}

cudaError_t launch_phase_apply_c64(const double* re_in, const double* im_in, const double* theta,
                                   long long theta_stride, double* re_out, double* im_out, int n,
                                   long long batch, int sms, cudaStream_t st) {
  const long long elems = batch << n;
  const long long work = n >= 1 ? elems / 2 : elems;
  const long long want = (work + 255) / 256;
  const unsigned blocks = (unsigned)std::max<long long>(1, std::min<long long>(want, (long long)sms * 8));
  if (n >= 1)
    return launch_pass(fwt_phase_apply_c64_kernel, dim3(blocks), 256, 0, st, 1, re_in, im_in, theta,
                       theta_stride, re_out, im_out, n, work);
  return launch_pass(fwt_phase_apply_c64_scalar_kernel, dim3(blocks), 256, 0, st, 1, re_in, im_in,
                     theta, theta_stride, re_out, im_out, work);
}

void register_rows_c64(std::vector<KernelEntry>& v) {
  RowSet<FWT_C64, 1, 1, double, ArithF64, 14>::add(v);
  v.push_back(cluster_entry<FWT_C64, 1, 13, 1>());  // 2^14-element vectors on CTA pairs
}
}  // namespace fwt
