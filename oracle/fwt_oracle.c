/*
 * CPU oracle for the batched Walsh-Hadamard transform.  TEST INFRASTRUCTURE ONLY:
 * nothing in the product library links, loads or calls this file.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes (per real vector x of length N = 2^n):
 *
 *     y[k] = s * sum_{i=0}^{N-1} (-1)^{popc(k & i)} x[i]
 *
 * with s = 2^{-n/2} for the normalised transform and s = 1 otherwise.  The sign
 * rule (-1)^{popc(k & i)} is the one stated in "[QDP] [feature] Pr4 kronecker
 * fwt", section "How" (naive GEMM placeholder); the scale 2^{-n/2} is the usual
 * orthonormal scaling of H_n.
 *
 * Routines:
 *   - oracle_fwt_f64 / oracle_fwt_u32: the textbook in-place butterfly network,
 *     stage h pairing entries at distance 1, 2, 4, ... with (a+b, a-b), as in the
 *     iThome "Day 18" FWT post, section "Tensor Core wants matrix
 *     multiplication" (stage 0 local pairs, stage 1 stride 2, stage 2 stride 4).
 *     Floating point runs in double; int32 runs in uint32_t so that overflow
 *     wraps modulo 2^32 (signed overflow is undefined in C).
 *   - oracle_fwt_bits_f64 / oracle_fwt_bits_u32: the same network restricted to
 *     the stages of index bits [lo, lo+nbits), i.e. I (x) H_nbits (x) I applied to
 *     each vector (a transform on a subset of qubits; the Kronecker factors of
 *     "[QDP] [feature] Pr4 kronecker fwt", deliverables: (H_{n1} (x) I) and
 *     (I (x) H_{n2})).
 *   - oracle_fwt_entry_f64 / oracle_fwt_entry_u32: one output entry straight from
 *     the definition above, O(N) per entry, for spot checks at sizes where the
 *     whole reference transform is too slow to repeat.
 *
 * No blocking, no fusion, no reordering: one stage after another over the whole
 * vector.  Threads (plain pthreads) only split the batch into whole vectors.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* s = 2^{-n/2} in double; 1 when not normalising. */
double oracle_scale(int n, int normalize) {
  if (!normalize) return 1.0;
  if (n % 2 == 0) return ldexp(1.0, -n / 2);
  return ldexp(1.0, -(n - 1) / 2) / sqrt(2.0);
}

/* Stages h = 2^lo, 2^(lo+1), ..., 2^(lo+nbits-1) of the butterfly network: the
 * transform over index bits [lo, lo+nbits) only, i.e. (I (x) H_nbits (x) I_{2^lo}) x.
 * With lo = 0 and nbits = n it is the whole transform. */
static void butterfly_bits_f64(double* x, int64_t N, int lo, int nbits) {
  for (int64_t h = (int64_t)1 << lo; h < ((int64_t)1 << (lo + nbits)); h *= 2) {
    for (int64_t i = 0; i < N; i += 2 * h) {
      for (int64_t j = i; j < i + h; ++j) {
        double u = x[j];
        double v = x[j + h];
        x[j] = u + v;
        x[j + h] = u - v;
      }
    }
  }
}

static void butterfly_bits_u32(uint32_t* x, int64_t N, int lo, int nbits) {
  for (int64_t h = (int64_t)1 << lo; h < ((int64_t)1 << (lo + nbits)); h *= 2) {
    for (int64_t i = 0; i < N; i += 2 * h) {
      for (int64_t j = i; j < i + h; ++j) {
        uint32_t u = x[j];
        uint32_t v = x[j + h];
        x[j] = u + v;
        x[j + h] = u - v;
      }
    }
  }
}

static void butterfly_f64(double* x, int64_t N) {
  for (int64_t h = 1; h < N; h *= 2) {
    for (int64_t i = 0; i < N; i += 2 * h) {
      for (int64_t j = i; j < i + h; ++j) {
        double u = x[j];
        double v = x[j + h];
        x[j] = u + v;
        x[j + h] = u - v;
      }
    }
  }
}

static void butterfly_u32(uint32_t* x, int64_t N) {
  for (int64_t h = 1; h < N; h *= 2) {
    for (int64_t i = 0; i < N; i += 2 * h) {
      for (int64_t j = i; j < i + h; ++j) {
        uint32_t u = x[j];
        uint32_t v = x[j + h];
        x[j] = u + v;
        x[j + h] = u - v;
      }
    }
  }
}

typedef struct {
  const void* x;
  void* y;
  int n;
  int64_t first, last; /* vectors [first, last) */
  double scale;
  int is_int;
  int lo, nbits; /* nbits < 0: the whole transform */
} job_t;

static void* run_job(void* arg) {
  job_t* jb = (job_t*)arg;
  int64_t N = (int64_t)1 << jb->n;
  for (int64_t b = jb->first; b < jb->last; ++b) {
    if (jb->is_int) {
      const uint32_t* src = (const uint32_t*)jb->x + b * N;
      uint32_t* dst = (uint32_t*)jb->y + b * N;
      if (dst != src) memcpy(dst, src, (size_t)N * sizeof(uint32_t));
      if (jb->nbits < 0) butterfly_u32(dst, N);
      else butterfly_bits_u32(dst, N, jb->lo, jb->nbits);
    } else {
      const double* src = (const double*)jb->x + b * N;
      double* dst = (double*)jb->y + b * N;
      if (dst != src) memcpy(dst, src, (size_t)N * sizeof(double));
      if (jb->nbits < 0) butterfly_f64(dst, N);
      else butterfly_bits_f64(dst, N, jb->lo, jb->nbits);
      if (jb->scale != 1.0)
        for (int64_t k = 0; k < N; ++k) dst[k] *= jb->scale;
    }
  }
  return NULL;
}

static int run_batch(const void* x, void* y, int n, int64_t count, double scale,
                     int is_int, int nthreads, int lo, int nbits) {
  if (n < 0 || n > 40 || count < 0 || (count > 0 && (!x || !y))) return 1;
  if (nbits >= 0 && (lo < 0 || lo + nbits > n)) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > count) nthreads = count > 0 ? (int)count : 1;
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) { free(jobs); free(tids); return 2; }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].x = x; jobs[t].y = y; jobs[t].n = n; jobs[t].scale = scale;
    jobs[t].is_int = is_int;
    jobs[t].lo = lo; jobs[t].nbits = nbits;
    jobs[t].first = count * t / nthreads;
    jobs[t].last = count * (t + 1) / nthreads;
  }
  /* A thread that could not be started has its share run on the calling thread. */
  char* started = (char*)calloc((size_t)nthreads, 1);
  if (!started) { free(jobs); free(tids); return 2; }
  for (int t = 1; t < nthreads; ++t)
    started[t] = pthread_create(&tids[t], NULL, run_job, &jobs[t]) == 0;
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t]) pthread_join(tids[t], NULL);
    else run_job(&jobs[t]);
  }
  free(started); free(jobs); free(tids);
  return 0;
}

/* count vectors of 2^n doubles, x -> y (y may equal x).  Returns 0 on success. */
int oracle_fwt_f64(const double* x, double* y, int n, int64_t count, int normalize,
                   int nthreads) {
  return run_batch(x, y, n, count, oracle_scale(n, normalize), 0, nthreads, 0, -1);
}

/* count vectors of 2^n uint32 (int32 bit patterns), wrap-around arithmetic. */
int oracle_fwt_u32(const uint32_t* x, uint32_t* y, int n, int64_t count, int nthreads) {
  return run_batch(x, y, n, count, 1.0, 1, nthreads, 0, -1);
}

/* The transform over index bits [lo, lo+nbits) of each 2^n vector (the other bits
 * untouched), scaled by 2^{-nbits/2} when normalising. */
int oracle_fwt_bits_f64(const double* x, double* y, int n, int64_t count, int lo, int nbits,
                        int normalize, int nthreads) {
  if (nbits < 0) return 1;
  return run_batch(x, y, n, count, oracle_scale(nbits, normalize), 0, nthreads, lo, nbits);
}

int oracle_fwt_bits_u32(const uint32_t* x, uint32_t* y, int n, int64_t count, int lo, int nbits,
                        int nthreads) {
  if (nbits < 0) return 1;
  return run_batch(x, y, n, count, 1.0, 1, nthreads, lo, nbits);
}

/* Parity of popc(v): XOR-fold the 64 bits down to one. */
/* IQP-style encoding step: each amplitude is first multiplied by the phase
 * e^{i theta} (theta[b * theta_stride + i] for vector b), then the complex vector
 * is transformed: y = s * H (e^{i theta} . x).  The phase step is the diagonal
 * before the transform in "[QDP] [feature] Pr4 kronecker fwt" (IQP encoding,
 * "IQP shared-mem fused" row of the benchmark table); the pages do not give the
 * angle function, so theta is an input.  cos and sin from the C library, in
 * double; then the same butterfly network as oracle_fwt_f64 on each part. */
int oracle_phase_fwt_f64(const double* re, const double* im, const double* theta,
                         int64_t theta_stride, double* re_out, double* im_out, int n,
                         int64_t count, int normalize) {
  if (n < 0 || n > 40 || count < 0) return 1;
  const int64_t N = (int64_t)1 << n;
  const double s = oracle_scale(n, normalize);
  for (int64_t b = 0; b < count; ++b) {
    const double* xr = re + b * N;
    const double* xi = im + b * N;
    const double* th = theta + b * theta_stride;
    double* yr = re_out + b * N;
    double* yi = im_out + b * N;
    for (int64_t i = 0; i < N; ++i) {
      const double c = cos(th[i]), sn = sin(th[i]);
      const double r = xr[i] * c - xi[i] * sn;
      const double m = xr[i] * sn + xi[i] * c;
      yr[i] = r;
      yi[i] = m;
    }
    butterfly_f64(yr, N);
    butterfly_f64(yi, N);
    for (int64_t k = 0; k < N; ++k) { yr[k] *= s; yi[k] *= s; }
  }
  return 0;
}

static int popc_parity(uint64_t v) {
  v ^= v >> 32; v ^= v >> 16; v ^= v >> 8; v ^= v >> 4; v ^= v >> 2; v ^= v >> 1;
  return (int)(v & 1u);
}

/* y[k] of one vector, straight from the definition, then scaled.  The 2^n signed
 * terms are added with Neumaier's compensated summation (Neumaier 1974), so the
 * sum is good to a few ulps even at n = 24, where a plain running sum of 2^24
 * terms could drift far beyond a 1e-12 relative error. */
double oracle_fwt_entry_f64(const double* x, int n, int64_t k, int normalize) {
  int64_t N = (int64_t)1 << n;
  double sum = 0.0, comp = 0.0;
  for (int64_t i = 0; i < N; ++i) {
    double t = popc_parity((uint64_t)(k & i)) ? -x[i] : x[i];
    double s2 = sum + t;
    if (fabs(sum) >= fabs(t)) comp += (sum - s2) + t;
    else comp += (t - s2) + sum;
    sum = s2;
  }
  return (sum + comp) * oracle_scale(n, normalize);
}

/* y[k] of one int32 vector from the definition, modulo 2^32. */
uint32_t oracle_fwt_entry_u32(const uint32_t* x, int n, int64_t k) {
  int64_t N = (int64_t)1 << n;
  uint32_t acc = 0;
  for (int64_t i = 0; i < N; ++i) {
    if (popc_parity((uint64_t)(k & i))) acc -= x[i];
    else acc += x[i];
  }
  return acc;
}
