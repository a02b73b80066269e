/*
 * A plain C99 program that uses the library through include/fwt.h alone: the header
 * must compile as C, the library must link into a C program, and the calls must
 * behave as the header states.
 *
 *   c_consumer cpu   argument checks, status strings, plans, the tile self-check
 *                    (no CUDA call is made)
 *   c_consumer gpu   transforms on device memory from cudaMalloc and on host
 *                    arrays, checked against closed forms of the sign rule
 *                    y[k] = s * sum_i (-1)^popc(k & i) x[i]
 *                    ("[QDP] [feature] Pr4 kronecker fwt", section "How")
 *
 * Closed forms used (exact, no reference implementation needed):
 *   - x = e_j (one 1 at index j): y[k] = s (-1)^popc(k & j), every k;
 *   - bit range [lo, lo + nb) on x = e_j: y[k] = 2^(-nb/2) (-1)^popc(k & j & R) when k
 *     agrees with j outside R = the range's bits, else 0;
 *   - integer x: y[k] for sampled k, summed directly from the definition.
 * Exit status 0 when every check passes; each failure is printed.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fwt.h"

#ifdef FWT_CONSUMER_CUDA
#include <cuda_runtime_api.h>
#endif

static int g_failures = 0;

#define CHECK(cond, ...)                                       \
  do {                                                         \
    if (!(cond)) {                                             \
      ++g_failures;                                            \
      fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__);     \
      fprintf(stderr, __VA_ARGS__);                            \
      fputc('\n', stderr);                                     \
    }                                                          \
  } while (0)

static int cpu_checks(void) {
  /* fake, 16-byte aligned addresses: validation never dereferences them */
  float* a = (float*)(uintptr_t)0x10000;
  float* b = (float*)(uintptr_t)0x40010000;
  float* c = (float*)(uintptr_t)0x80010000;
  float* d = (float*)(uintptr_t)0xc0010000;
  int bits[3] = {0, 0, 0};

  CHECK(strcmp(fwt_status_string(FWT_OK), "ok") == 0, "status string of FWT_OK");
  CHECK(fwt_status_string(12345) != NULL, "status string of an unknown code");
  CHECK(fwt_batched_c32(a, b, c, d, 31, 1, 1, NULL) == FWT_ERR_INVALID_ARG, "n = 31");
  CHECK(fwt_batched_c32(a, b, c, d, -1, 1, 1, NULL) == FWT_ERR_INVALID_ARG, "n = -1");
  CHECK(fwt_batched_c32(a, b, c, d, 4, -1, 1, NULL) == FWT_ERR_INVALID_ARG, "batch < 0");
  CHECK(fwt_batched_c32(NULL, NULL, NULL, NULL, 4, 0, 1, NULL) == FWT_OK, "empty batch");
  CHECK(fwt_batched_c32(a + 1, b, c, d, 4, 1, 1, NULL) == FWT_ERR_MISALIGNED, "misaligned");
  CHECK(fwt_batched_c32(a, b, a + 4, d, 4, 1, 1, NULL) == FWT_ERR_INVALID_ARG, "overlap");
  CHECK(fwt_batched_i32((const int32_t*)a, NULL, (int32_t*)c, NULL, 4, 1, 1, NULL) ==
            FWT_ERR_UNSUPPORTED,
        "int32 with normalisation");
  CHECK(fwt_bits_c64((const double*)a, (const double*)b, (double*)c, (double*)d, 10, 1, 6, 5, 1,
                     NULL) == FWT_ERR_INVALID_ARG,
        "bit range beyond n");
  CHECK(fwt_mask_c32(a, b, c, d, 10, 1, 1u << 10, 1, NULL) == FWT_ERR_INVALID_ARG,
        "mask beyond n");
  CHECK(fwt_host_c32(a, b, c, d, 4, 1, 1, NULL, 0, NULL) == FWT_ERR_INVALID_ARG,
        "host entry without workspace");
  CHECK(fwt_plan_passes(24, FWT_C64) == 2, "fp64 n = 24 plan passes");
  CHECK(fwt_plan_factors(24, FWT_C64, bits, 3) == 2 && bits[0] + bits[1] == 24,
        "fp64 n = 24 plan factors");
  CHECK(fwt_plan_passes(31, FWT_C32) == -1, "plan of n = 31");
  CHECK(fwt_host_workspace_bytes(FWT_C32, 20, 16, 1) > 0, "host workspace size");
  CHECK(fwt_host_workspace_bytes(FWT_C32, 31, 16, 1) == 0, "host workspace size of n = 31");
  CHECK(fwt_selfcheck() == 0, "tile self-check");
  return g_failures;
}

#ifdef FWT_CONSUMER_CUDA

static int popc64(uint64_t v) {
  int c = 0;
  while (v) {
    v &= v - 1;
    ++c;
  }
  return c;
}

#define CUDA_OK(call)                                                            \
  do {                                                                           \
    cudaError_t e_ = (call);                                                     \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, \
              __LINE__);                                                         \
      exit(2);                                                                   \
    }                                                                            \
  } while (0)

/* one 1 at index js[v] in vector v of a batch-major array */
static void deltas_f32(float* x, int n, int batch, const uint64_t* js) {
  const size_t N = (size_t)1 << n;
  memset(x, 0, N * (size_t)batch * sizeof(float));
  for (int v = 0; v < batch; ++v) x[(size_t)v * N + js[v]] = 1.0f;
}
static void deltas_f64(double* x, int n, int batch, const uint64_t* js) {
  const size_t N = (size_t)1 << n;
  memset(x, 0, N * (size_t)batch * sizeof(double));
  for (int v = 0; v < batch; ++v) x[(size_t)v * N + js[v]] = 1.0;
}

/* y = s (-1)^popc(k & j) for x = e_j, compared exactly (s a power of two) */
static int check_sign_rows_f32(const float* y, int n, int batch, const uint64_t* js, float s,
                               const char* what) {
  const size_t N = (size_t)1 << n;
  int bad = 0;
  for (int v = 0; v < batch; ++v)
    for (size_t k = 0; k < N; ++k) {
      const float want = (popc64(k & js[v]) & 1) ? -s : s;
      if (y[(size_t)v * N + k] != want && bad++ < 3)
        fprintf(stderr, "%s: vector %d, k = %zu: %g, expected %g\n", what, v, k,
                (double)y[(size_t)v * N + k], (double)want);
    }
  CHECK(bad == 0, "%s: %d wrong elements", what, bad);
  return bad;
}
static int check_sign_rows_f64(const double* y, int n, int batch, const uint64_t* js, double s,
                               double rel, const char* what) {
  const size_t N = (size_t)1 << n;
  int bad = 0;
  for (int v = 0; v < batch; ++v)
    for (size_t k = 0; k < N; ++k) {
      const double want = (popc64(k & js[v]) & 1) ? -s : s;
      if (fabs(y[(size_t)v * N + k] - want) > rel * s && bad++ < 3)
        fprintf(stderr, "%s: vector %d, k = %zu: %.17g, expected %.17g\n", what, v, k,
                y[(size_t)v * N + k], want);
    }
  CHECK(bad == 0, "%s: %d wrong elements", what, bad);
  return bad;
}

static void gpu_c32(cudaStream_t st) {
  /* one tile (n = 12), a one-pass cluster size (n = 16), two passes (n = 20) */
  const int ns[3] = {12, 16, 20};
  for (int t = 0; t < 3; ++t) {
    const int n = ns[t], batch = 3;
    const size_t N = (size_t)1 << n, bytes = N * batch * sizeof(float);
    const uint64_t jre[3] = {0, N - 1, (N / 3) | 1}, jim[3] = {5, N / 2, N - 2};
    float *hre = (float*)malloc(bytes), *him = (float*)malloc(bytes);
    float *dre, *dim, *ore, *oim;
    char what[64];
    CUDA_OK(cudaMalloc((void**)&dre, bytes));
    CUDA_OK(cudaMalloc((void**)&dim, bytes));
    CUDA_OK(cudaMalloc((void**)&ore, bytes));
    CUDA_OK(cudaMalloc((void**)&oim, bytes));
    deltas_f32(hre, n, batch, jre);
    deltas_f32(him, n, batch, jim);
    CUDA_OK(cudaMemcpy(dre, hre, bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dim, him, bytes, cudaMemcpyHostToDevice));
    CHECK(fwt_batched_c32(dre, dim, ore, oim, n, batch, 1, (fwt_stream_t)st) == FWT_OK,
          "fwt_batched_c32 n = %d", n);
    CUDA_OK(cudaStreamSynchronize(st));
    CUDA_OK(cudaMemcpy(hre, ore, bytes, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(him, oim, bytes, cudaMemcpyDeviceToHost));
    snprintf(what, sizeof what, "c32 n = %d re", n);
    check_sign_rows_f32(hre, n, batch, jre, ldexpf(1.0f, -n / 2), what);
    snprintf(what, sizeof what, "c32 n = %d im", n);
    check_sign_rows_f32(him, n, batch, jim, ldexpf(1.0f, -n / 2), what);
    /* in place, unnormalised: a second transform gives 2^n e_j back (H H = 2^n I) */
    CHECK(fwt_batched_c32(ore, oim, ore, oim, n, batch, 0, (fwt_stream_t)st) == FWT_OK,
          "in-place fwt_batched_c32 n = %d", n);
    CUDA_OK(cudaStreamSynchronize(st));
    CUDA_OK(cudaMemcpy(hre, ore, bytes, cudaMemcpyDeviceToHost));
    {
      int bad = 0;
      const float want_one = ldexpf(1.0f, n - n / 2);
      for (int v = 0; v < batch; ++v)
        for (size_t k = 0; k < N; ++k)
          bad += hre[(size_t)v * N + k] != (k == jre[v] ? want_one : 0.0f);
      CHECK(bad == 0, "c32 n = %d: H H e_j != 2^n e_j at %d elements", n, bad);
    }
    cudaFree(dre);
    cudaFree(dim);
    cudaFree(ore);
    cudaFree(oim);
    free(hre);
    free(him);
  }
}

static void gpu_c64(cudaStream_t st) {
  /* the two-pass fp64 plan at n = 24 (one vector), and an odd n (s = 2^-6.5) */
  const int ns[2] = {24, 13};
  for (int t = 0; t < 2; ++t) {
    const int n = ns[t], batch = t == 0 ? 1 : 4;
    const size_t N = (size_t)1 << n, bytes = N * batch * sizeof(double);
    const uint64_t jre[4] = {N - 1, 7, 0, N / 2 + 1}, jim[4] = {123457 % N, 1, N - 1, 2};
    double *hre = (double*)malloc(bytes), *him = (double*)malloc(bytes);
    double *dre, *dim;
    char what[64];
    const double s = (n & 1) ? ldexp(sqrt(0.5), -(n / 2)) : ldexp(1.0, -(n / 2));
    CUDA_OK(cudaMalloc((void**)&dre, bytes));
    CUDA_OK(cudaMalloc((void**)&dim, bytes));
    deltas_f64(hre, n, batch, jre);
    deltas_f64(him, n, batch, jim);
    CUDA_OK(cudaMemcpy(dre, hre, bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dim, him, bytes, cudaMemcpyHostToDevice));
    CHECK(fwt_batched_c64(dre, dim, dre, dim, n, batch, 1, (fwt_stream_t)st) == FWT_OK,
          "fwt_batched_c64 n = %d", n);
    CUDA_OK(cudaStreamSynchronize(st));
    CUDA_OK(cudaMemcpy(hre, dre, bytes, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(him, dim, bytes, cudaMemcpyDeviceToHost));
    /* Even n: every intermediate is a power of two, so the result is exact.  Odd n: the
       butterflies run in fixed point with 61 - 13 = 48 fraction bits below the tile's
       largest element, and the division by sqrt 2 is truncated at that scale, so each
       element may be off by a few units of 2^-48 relative (measured: 2e-15); 1e-13 is
       well inside the 1e-12 relative L2 error the header states. */
    snprintf(what, sizeof what, "c64 n = %d re", n);
    check_sign_rows_f64(hre, n, batch, jre, s, (n & 1) ? 1e-13 : 0.0, what);
    snprintf(what, sizeof what, "c64 n = %d im", n);
    check_sign_rows_f64(him, n, batch, jim, s, (n & 1) ? 1e-13 : 0.0, what);
    cudaFree(dre);
    cudaFree(dim);
    free(hre);
    free(him);
  }
}

static void gpu_i32(cudaStream_t st) {
  /* real-only int32 at n = 18 (two passes): sampled outputs summed from the definition */
  const int n = 18, batch = 2;
  const size_t N = (size_t)1 << n, bytes = N * batch * sizeof(int32_t);
  int32_t *hx = (int32_t*)malloc(bytes), *hy = (int32_t*)malloc(bytes);
  int32_t* dx;
  uint32_t state = 12345u;
  const size_t ks[6] = {0, 1, 2, 77777, N / 2, N - 1};
  for (size_t i = 0; i < N * batch; ++i) {
    state = state * 1664525u + 1013904223u; /* a linear congruential sequence */
    hx[i] = (int32_t)(state >> 28) - 8;     /* values in [-8, 8) */
  }
  CUDA_OK(cudaMalloc((void**)&dx, bytes));
  CUDA_OK(cudaMemcpy(dx, hx, bytes, cudaMemcpyHostToDevice));
  CHECK(fwt_batched_i32(dx, NULL, dx, NULL, n, batch, 0, (fwt_stream_t)st) == FWT_OK,
        "fwt_batched_i32 real-only in place");
  CUDA_OK(cudaStreamSynchronize(st));
  CUDA_OK(cudaMemcpy(hy, dx, bytes, cudaMemcpyDeviceToHost));
  for (int v = 0; v < batch; ++v)
    for (int q = 0; q < 6; ++q) {
      int64_t want = 0;
      for (size_t i = 0; i < N; ++i)
        want += (popc64(ks[q] & i) & 1) ? -(int64_t)hx[(size_t)v * N + i] : hx[(size_t)v * N + i];
      CHECK(hy[(size_t)v * N + ks[q]] == (int32_t)want, "int32 n = 18 vector %d k = %zu: %d vs %lld",
            v, ks[q], hy[(size_t)v * N + ks[q]], (long long)want);
    }
  cudaFree(dx);
  free(hx);
  free(hy);
}

static void gpu_bits(cudaStream_t st) {
  /* H on index bits [lo, lo + nb) of x = e_j, n = 20: a range inside the row tile
     and one above it (a strided column pass) */
  const int n = 20, batch = 2;
  const int ranges[2][2] = {{3, 7}, {16, 4}};
  const size_t N = (size_t)1 << n, bytes = N * batch * sizeof(float);
  const uint64_t js[2] = {0x5a5a5, 0xfffff};
  float *h = (float*)malloc(bytes), *dre, *dim;
  CUDA_OK(cudaMalloc((void**)&dre, bytes));
  CUDA_OK(cudaMalloc((void**)&dim, bytes));
  for (int t = 0; t < 2; ++t) {
    const int lo = ranges[t][0], nb = ranges[t][1];
    const uint64_t R = (((uint64_t)1 << nb) - 1) << lo;
    const float s = ldexpf(1.0f, -nb / 2) * ((nb & 1) ? sqrtf(0.5f) : 1.0f);
    int bad = 0;
    deltas_f32(h, n, batch, js);
    CUDA_OK(cudaMemcpy(dre, h, bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dim, h, bytes, cudaMemcpyHostToDevice));
    CHECK(fwt_bits_c32(dre, dim, dre, dim, n, batch, lo, nb, 1, (fwt_stream_t)st) == FWT_OK,
          "fwt_bits_c32 [%d, %d)", lo, lo + nb);
    CUDA_OK(cudaStreamSynchronize(st));
    CUDA_OK(cudaMemcpy(h, dre, bytes, cudaMemcpyDeviceToHost));
    for (int v = 0; v < batch; ++v)
      for (size_t k = 0; k < N; ++k) {
        const float want = ((k ^ js[v]) & ~R) ? 0.0f : ((popc64(k & js[v] & R) & 1) ? -s : s);
        const float got = h[(size_t)v * N + k];
        if (fabsf(got - want) > 1e-6f * s && bad++ < 3)
          fprintf(stderr, "bits [%d, %d) vector %d k = %zu: %g vs %g\n", lo, lo + nb, v, k,
                  (double)got, (double)want);
      }
    CHECK(bad == 0, "fwt_bits_c32 [%d, %d): %d wrong elements", lo, lo + nb, bad);
  }
  cudaFree(dre);
  cudaFree(dim);
  free(h);
}

static void gpu_host_entry(cudaStream_t st) {
  /* host arrays in and out (pageable memory), a caller-owned device workspace */
  const int n = 16, batch = 5;
  const size_t N = (size_t)1 << n, bytes = N * batch * sizeof(float);
  const uint64_t jre[5] = {0, 1, 2, 3, N - 1}, jim[5] = {N - 1, 9, 99, 999, 9999};
  const size_t ws_bytes = fwt_host_workspace_bytes(FWT_C32, n, batch, 1);
  float *re = (float*)malloc(bytes), *im = (float*)malloc(bytes);
  void* ws;
  CHECK(ws_bytes > 0, "host workspace size");
  CUDA_OK(cudaMalloc(&ws, ws_bytes));
  deltas_f32(re, n, batch, jre);
  deltas_f32(im, n, batch, jim);
  CHECK(fwt_host_c32(re, im, re, im, n, batch, 1, ws, ws_bytes, (fwt_stream_t)st) == FWT_OK,
        "fwt_host_c32");
  CUDA_OK(cudaStreamSynchronize(st));
  check_sign_rows_f32(re, n, batch, jre, ldexpf(1.0f, -n / 2), "host c32 re");
  check_sign_rows_f32(im, n, batch, jim, ldexpf(1.0f, -n / 2), "host c32 im");
  cudaFree(ws);
  free(re);
  free(im);
}

static int gpu_checks(void) {
  cudaStream_t st;
  CUDA_OK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  gpu_c32(st);
  gpu_c64(st);
  gpu_i32(st);
  gpu_bits(st);
  gpu_host_entry(st);
  CHECK(fwt_device_status() == FWT_OK, "device status word");
  CUDA_OK(cudaStreamDestroy(st));
  return g_failures;
}
#endif /* FWT_CONSUMER_CUDA */

int main(int argc, char** argv) {
  const char* mode = argc > 1 ? argv[1] : "cpu";
  int fails;
  if (strcmp(mode, "cpu") == 0) {
    fails = cpu_checks();
  } else if (strcmp(mode, "gpu") == 0) {
#ifdef FWT_CONSUMER_CUDA
    fails = gpu_checks();
#else
    fprintf(stderr, "built without the CUDA runtime\n");
    return 2;
#endif
  } else {
    fprintf(stderr, "usage: %s cpu|gpu\n", argv[0]);
    return 2;
  }
  printf("%s checks: %d failure(s)\n", mode, fails);
  return fails ? 1 : 0;
}
