// fp64 row passes (int64 fixed-point butterflies).
#include <algorithm>
#include <cmath>

#include "kernel_sets.cuh"

namespace fwt {

// ---- fp64 diagonal phase in 64-bit fixed point ------------------------------------
// (re, im) <- (re cos t - im sin t, re sin t + im cos t) for each element.  GB300's fp64
// unit runs at about 1/64 of the fp32 rate, so the sine and cosine are evaluated in
// integer arithmetic (the integer multiply-high units):
//   * the angle is reduced to a fraction of a turn u = t / (2 pi) mod 1 (64 bits): its
//     53-bit mantissa times 1/(2 pi) held to 128 bits, keeping the product's bits
//     just below the units (the Payne-Hanek idea; exact to 2^-64 turns for
//     |t| < 2^40, far more than the angle's own precision);
//   * the top 10 bits of u pick (cos, sin) of 2 pi j / 1024 from a table, and the
//     rest gives a remainder r < 2 pi / 1024 radians, whose sine and 1 - cosine come
//     from their Taylor series (r - r^3/6 + r^5/120 and r^2/2 - r^4/24: the first
//     omitted terms are below 3e-17; the cubic and higher terms need only ~30 bits
//     and use 32 x 32-bit products);
//   * the angle-addition formula, as one complex product with three multiplies,
//     gives cos t and sin t in units of 2^-62 (within 1e-16 of the exact values);
//   * the element (re, im) is scaled to 61 fraction bits below its larger exponent,
//     rotated with three 64 x 64-bit multiply-highs, and rounded once back to fp64.
// The result is within about 1e-16 of the exact rotation, relative to |x|.
// Elements with an Inf or NaN, or angles of magnitude 2^40 and more, take the fp64
// sincos instead.  The constants come from phase_constants.py (pi by Machin's
// formula).
namespace {
constexpr unsigned long long kInv2PiHi = 0x28be60db9391054aull;   // 2^128 / (2 pi), high word
constexpr unsigned long long kInv2PiLo = 0x7f09d5f47d4d3770ull;   // ... low word
constexpr unsigned long long kTwoPiQ61 = 0xc90fdaa22168c235ull;   // 2 pi * 2^61
constexpr unsigned long long kInv6Q32 = 0x2aaaaaabull;    // 2^32 / 6
constexpr unsigned long long kInv24Q32 = 0x0aaaaaabull;   // 2^32 / 24
constexpr unsigned long long kInv120Q32 = 0x02222222ull;  // 2^32 / 120
constexpr int kPhaseTableBits = 10;
constexpr int kPhaseTable = 1 << kPhaseTableBits;
}  // namespace

// cos and sin of 2 pi j / 1024 in units of 2^-62 (filled once per device on the host)
static __device__ longlong2 g_phase_table[kPhaseTable];

// y = e^{i t} x for one element in fixed point; false when the element needs the fp64
// fallback (an Inf or NaN anywhere, or |t| >= 2^40).
__device__ __forceinline__ bool phase_rotate_fixed(double t, double re, double im,
                                                   const longlong2* tab, double& out_re,
                                                   double& out_im) {
  const unsigned long long tb = (unsigned long long)__double_as_longlong(t);
  const unsigned long long br = (unsigned long long)__double_as_longlong(re);
  const unsigned long long bi = (unsigned long long)__double_as_longlong(im);
  const int te = (int)((tb >> 52) & 0x7ff), er = (int)((br >> 52) & 0x7ff),
            ei = (int)((bi >> 52) & 0x7ff);
  if (te >= 1063 || er == 0x7ff || ei == 0x7ff) return false;
  // turns: bits [s, s + 64) of mantissa * 2^128 / (2 pi), s = 1139 - exponent >= 77
  const unsigned long long tm = (tb & 0x000fffffffffffffull) | ((unsigned long long)(te != 0) << 52);
  const int s = 1139 - max(te, 1);
  const unsigned long long a1 = __umul64hi(tm, kInv2PiLo);
  const unsigned long long b0 = tm * kInv2PiHi, b1 = __umul64hi(tm, kInv2PiHi);
  const unsigned long long p1 = a1 + b0;
  const unsigned long long p2 = b1 + (p1 < a1 ? 1ull : 0ull);
  unsigned long long u = s >= 128 ? shr64(p2, (uint32_t)(s - 128))
                                  : (p2 << ((128 - s) & 63)) | shr64(p1, (uint32_t)(s - 64));
  if (tb >> 63) u = 0ull - u;  // the angle's sign: -t is 1 - u turns
  // table cell j and remainder: rho = 2^7 r (r < 2 pi / 1024 radians), units of 2^-64
  const int j = (int)(u >> (64 - kPhaseTableBits));
  const unsigned long long f = u & ((1ull << (64 - kPhaseTableBits)) - 1ull);
  const unsigned long long rho = (__umul64hi(f, kTwoPiQ61) << 10) | ((f * kTwoPiQ61) >> 54);
  const unsigned long long rho2 = __umul64hi(rho, rho);
  // the small terms need ~30 bits: 32 x 32-bit products of the top words
  const unsigned long long rho3 = (rho >> 32) * (rho2 >> 32);
  const unsigned long long rho4 = (rho2 >> 32) * (rho2 >> 32);
  const unsigned long long rho5 = (rho3 >> 32) * (rho2 >> 32);
  // sin r = r - r^3/6 + r^5/120 and 1 - cos r = r^2/2 - r^4/24 (units of 2^-64)
  const long long sin_r = (long long)((rho >> 7) - (((rho3 >> 32) * kInv6Q32) >> 21) +
                                      (((rho5 >> 32) * kInv120Q32) >> 35));
  const long long omc_r = (long long)((rho2 >> 15) - (((rho4 >> 32) * kInv24Q32) >> 28));
  // (cos t, sin t) = (c0 + i s0)(1 + w), w = -omc_r + i sin_r: three products (Gauss)
  const longlong2 cs0 = tab[j];
  const long long k1 = __mul64hi(-omc_r, cs0.x + cs0.y);
  const long long k2 = __mul64hi(cs0.x, sin_r + omc_r);
  const long long k3 = __mul64hi(cs0.y, sin_r - omc_r);
  const long long c = cs0.x + (k1 - k3), sn = cs0.y + (k1 + k2);
  // the element with 61 fraction bits below its larger exponent, rotated (units 2^-59)
  const int E = max(max(er, ei), 1);
  long long qr, qi;
  if (E >= 64) {
    // exact scaling by 2^(61 + 1023 - E) in the exponent field, then the hardware
    // convert (round to nearest); an element more than 2^1083 below the larger one
    // rounds to 0
    const unsigned long long add = (unsigned long long)(1084 - E) << 52;
    qr = er + 1084 - E >= 1 ? __double2ll_rn(__longlong_as_double((long long)(br + add))) : 0;
    qi = ei + 1084 - E >= 1 ? __double2ll_rn(__longlong_as_double((long long)(bi + add))) : 0;
  } else {  // tiny pairs (subnormal scale): integer conversion
    qr = to_fixed<TO_FIXED_ANY>((long long)br, E, 61);
    qi = to_fixed<TO_FIXED_ANY>((long long)bi, E, 61);
  }
  const long long g1 = __mul64hi(c, qr + qi), g2 = __mul64hi(qr, sn - c), g3 = __mul64hi(qi, c + sn);
  const long long yr = g1 - g3, yi = g1 + g2;
  const int e0 = E - 1023 - 59;
  if (e0 >= -1022 && e0 <= 960) {
    const long long e0_field = (long long)((unsigned long long)(long long)e0 << 52);
    out_re = __longlong_as_double(from_fixed_cvt<false>(yr, e0_field, 0));
    out_im = __longlong_as_double(from_fixed_cvt<false>(yi, e0_field, 0));
  } else {  // results near or below the subnormal range: exact integer rounding
    out_re = __longlong_as_double(from_fixed_exact(yr, e0, 0, 0));
    out_im = __longlong_as_double(from_fixed_exact(yi, e0, 0, 0));
  }
  return true;
}

// The same with the fp64 sincos (fallback for non-finite values and huge angles).
__device__ __noinline__ void phase_rotate_fp64(double t, double re, double im, double& out_re,
                                               double& out_im) {
  double s, c;
  sincos(t, &s, &c);
  out_re = re * c - im * s;
  out_im = re * s + im * c;
}

// Diagonal phase for fp64 split complex vectors, element by element and in place or
// out of place.  16-byte vectors of two elements; a grid-stride loop over all pairs of
// the batch; the table goes to shared memory first.
__global__ void __launch_bounds__(256) fwt_phase_apply_c64_kernel(
    const double* re_in, const double* im_in, const double* theta, long long theta_stride,
    double* re_out, double* im_out,
    int n, long long pairs) {
  pdl_begin();
  __shared__ longlong2 tab[kPhaseTable];
  for (int i = threadIdx.x; i < kPhaseTable; i += blockDim.x) tab[i] = g_phase_table[i];
  __syncthreads();
  const long long nmask = (1ll << n) - 1;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < pairs;
       q += (long long)gridDim.x * blockDim.x) {
    const long long e = q * 2;  // first element of the pair (n >= 1: both in one vector)
    const double2 r = *reinterpret_cast<const double2*>(re_in + e);
    const double2 m = *reinterpret_cast<const double2*>(im_in + e);
    const long long t = (e >> n) * theta_stride + (e & nmask);
    const double2 th = *reinterpret_cast<const double2*>(theta + t);
    double2 yr, yi;
    if (!phase_rotate_fixed(th.x, r.x, m.x, tab, yr.x, yi.x)) phase_rotate_fp64(th.x, r.x, m.x, yr.x, yi.x);
    if (!phase_rotate_fixed(th.y, r.y, m.y, tab, yr.y, yi.y)) phase_rotate_fp64(th.y, r.y, m.y, yr.y, yi.y);
    *reinterpret_cast<double2*>(re_out + e) = yr;
    *reinterpret_cast<double2*>(im_out + e) = yi;
  }
}

// n = 0: one element a vector.
__global__ void __launch_bounds__(256) fwt_phase_apply_c64_scalar_kernel(
    const double* re_in, const double* im_in, const double* theta, long long theta_stride,
    double* re_out, double* im_out, long long count) {
  pdl_begin();
  __shared__ longlong2 tab[kPhaseTable];
  for (int i = threadIdx.x; i < kPhaseTable; i += blockDim.x) tab[i] = g_phase_table[i];
  __syncthreads();
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < count;
       e += (long long)gridDim.x * blockDim.x) {
    const double t = theta[e * theta_stride], r = re_in[e], m = im_in[e];
    double yr, yi;
    if (!phase_rotate_fixed(t, r, m, tab, yr, yi)) phase_rotate_fp64(t, r, m, yr, yi);
    re_out[e] = yr;
    im_out[e] = yi;
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

// Fills this device's phase table: cos and sin of 2 pi j / 1024 in units of 2^-62, from
// the host's long double sine and cosine (rounded once).
cudaError_t setup_phase_table_c64() {
  const long double pi = 3.141592653589793238462643383279502884L;
  longlong2 host[kPhaseTable];
  for (int j = 0; j < kPhaseTable; ++j) {
    const long double a = pi * (long double)j / (long double)(kPhaseTable / 2);
    host[j].x = (long long)llroundl(cosl(a) * 4611686018427387904.0L);  // 2^62
    host[j].y = (long long)llroundl(sinl(a) * 4611686018427387904.0L);
  }
  return cudaMemcpyToSymbol(g_phase_table, host, sizeof host);
}

void register_rows_c64(std::vector<KernelEntry>& v) {
  RowSet<FWT_C64, 1, 1, double, ArithF64, 14>::add(v);
  v.push_back(cluster_entry<FWT_C64, 1, 13, 1>());  // 2^14-element vectors on CTA pairs
}
}  // namespace fwt
