/*
 * Seeded synthetic inputs, shared by the CPU oracle and the CUDA library's
 * tests and benchmark.  This file holds none of the decode method's
 * arithmetic: it only draws the random-init weights, the exit-head
 * transforms and the prompts that the workloads call for (weights
 * N(0, 0.02) in bf16, T = I + N(0, 0.01), uniform prompt tokens and lengths).
 *
 * Generator (all integer steps are exact, so every machine gets the same bits):
 *   key(seed, tid)  = mix64(seed * G + tid * 0xD1B54A32D192ED03 + 0x632BE59BD9B4E019)
 *   out_k           = mix64(key + (k + 1) * G)           k >= 0
 *   mix64           = SplitMix64's output function (Steele, Lea, Flood,
 *                     "Fast splittable pseudorandom number generators", 2014)
 *   G               = 0x9E3779B97F4A7C15
 * Normals come in pairs (Box and Muller, 1958): pair p uses out_{2p} and
 * out_{2p+1}; u1 = (hi53(out_{2p}) + 1) / 2^53 in (0, 1],
 * u2 = hi53(out_{2p+1}) / 2^53 in [0, 1);
 * z_{2p} = sqrt(-2 ln u1) cos(2 pi u2), z_{2p+1} = sqrt(-2 ln u1) sin(2 pi u2).
 * ln, sin and cos are computed here from their power series in plain IEEE
 * double arithmetic (no libm, no contraction into FMA), so the values do
 * not depend on the platform's math library.  sqrt is IEEE correctly rounded.
 * A drawn value v = base + std * z is rounded double -> float (nearest even)
 * -> bf16 (nearest even on the float bits).
 *
 * Build: cc -O2 -ffp-contract=off -fno-fast-math -fPIC -shared -pthread
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define G_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(seed * G_GOLDEN + tid * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL);
}

static inline uint64_t stream_out(uint64_t key, uint64_t k) {
  return mix64(key + (k + 1) * G_GOLDEN);
}

/* Series coefficients, filled once by plain IEEE divisions (deterministic). */
static double inv_odd[32];       /* 1/k for odd k                       */
static double inv_sin_step[20];  /* 1/((2k)(2k+1))                       */
static double inv_cos_step[20];  /* 1/((2k-1)(2k))                       */
static pthread_once_t coef_once = PTHREAD_ONCE_INIT;
static void init_coefs(void) {
  for (int k = 1; k < 32; k += 2) inv_odd[k] = 1.0 / (double)k;
  for (int k = 1; k < 20; ++k) {
    inv_sin_step[k] = 1.0 / (double)((2 * k) * (2 * k + 1));
    inv_cos_step[k] = 1.0 / (double)((2 * k - 1) * (2 * k));
  }
}

/* natural log for x in (0, 1]: x = m 2^e, m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(t) = 2 (t + t^3/3 + t^5/5 + ...), t = (m - 1) / (m + 1),
 * |t| <= 0.1716, terms to t^25. */
static double series_log(double x) {
  uint64_t b;
  memcpy(&b, &x, 8);
  int e = (int)((b >> 52) & 0x7FF) - 1023;
  uint64_t mb = (b & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL;
  double m;
  memcpy(&m, &mb, 8);
  if (m > 1.4142135623730951) {
    m = m * 0.5;
    e += 1;
  }
  double t = (m - 1.0) / (m + 1.0);
  double s = t * t;
  double acc = 0.0;
  for (int k = 25; k >= 1; k -= 2) acc = acc * s + inv_odd[k];
  double lnm = 2.0 * t * acc;
  const double ln2_hi = 0.693147180369123816490; /* high bits of ln 2 */
  const double ln2_lo = 1.90821492927058770002e-10;
  return (double)e * ln2_hi + ((double)e * ln2_lo + lnm);
}

/* sin and cos of x in [-pi, pi] from their Taylor series (terms to x^31). */
static void series_sincos(double x, double *sn, double *cs) {
  double x2 = x * x;
  double s = 0.0, c = 0.0;
  /* sin = x (1 - x^2/(2*3) (1 - x^2/(4*5) (...))), cos = 1 - x^2/(1*2) (1 - x^2/(3*4) (...)) */
  for (int k = 15; k >= 1; --k) {
    s = 1.0 - s * x2 * inv_sin_step[k];
    c = 1.0 - c * x2 * inv_cos_step[k];
  }
  *sn = x * s;
  *cs = c;
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static void normal_pair(uint64_t key, uint64_t p, double *z0, double *z1) {
  uint64_t a = stream_out(key, 2 * p);
  uint64_t b = stream_out(key, 2 * p + 1);
  double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
  double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
  double r = sqrt(-2.0 * series_log(u1));
  /* 2 pi u2 = 2 pi v + pi with v = u2 - 1/2 (exact), cos/sin flip sign */
  double v = u2 - 0.5;
  double sn, cs;
  series_sincos(6.283185307179586 * v, &sn, &cs);
  *z0 = -r * cs;
  *z1 = -r * sn;
}

typedef struct {
  uint64_t key;
  uint64_t offset;
  uint64_t begin, end; /* element range relative to offset */
  double base, stdev;
  int64_t ncols; /* > 0: add diag_add where row == col */
  double diag_add;
  uint16_t *out;
  float *outf;
} normal_job;

static inline double draw_value(const normal_job *j, uint64_t g, double z) {
  double v = j->base + j->stdev * z;
  if (j->ncols > 0 && g / (uint64_t)j->ncols == g % (uint64_t)j->ncols) v = v + j->diag_add;
  return v;
}

static inline void store_value(const normal_job *j, uint64_t i, double v) {
  float f = (float)v;
  if (j->out) j->out[i] = f32_to_bf16_rne(f);
  if (j->outf) j->outf[i] = f;
}

static void *normal_worker(void *arg) {
  normal_job *j = (normal_job *)arg;
  uint64_t i = j->begin;
  while (i < j->end) {
    uint64_t g = j->offset + i;
    double z0, z1;
    normal_pair(j->key, g >> 1, &z0, &z1);
    if ((g & 1) == 0) {
      store_value(j, i, draw_value(j, g, z0));
      if (i + 1 < j->end) store_value(j, i + 1, draw_value(j, g + 1, z1));
      i += 2;
    } else {
      store_value(j, i, draw_value(j, g, z1));
      i += 1;
    }
  }
  return 0;
}

#define MAX_THREADS 256

static void run_normal(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, double base,
                       double stdev, int64_t ncols, double diag_add, uint16_t *out, float *outf,
                       int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
  if (n < 65536) nthreads = 1;
  pthread_once(&coef_once, init_coefs);
  normal_job jobs[MAX_THREADS];
  pthread_t th[MAX_THREADS];
  uint64_t key = stream_key(seed, tid);
  uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  per = (per + 1) & ~(uint64_t)1; /* even split points keep pairs inside one worker */
  int launched = 0;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = (uint64_t)t * per, e = b + per;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (normal_job){key, offset, b, e, base, stdev, ncols, diag_add, out, outf};
    if (nthreads == 1) {
      normal_worker(&jobs[t]);
    } else {
      pthread_create(&th[t], 0, normal_worker, &jobs[t]);
      ++launched;
    }
  }
  for (int t = 0; t < launched; ++t) pthread_join(th[t], 0);
}

/* n values of base + std * N(0,1) for elements offset .. offset+n-1 of tensor
 * `tid`, rounded to bf16 bit patterns.  If ncols > 0, diag_add is added to
 * elements whose row (index / ncols) equals their column (index % ncols)
 * before rounding (used for T = I + N(0, s)). */
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, double base,
                       double stdev, int64_t ncols, double diag_add, uint16_t *out, int nthreads) {
  run_normal(seed, tid, offset, n, base, stdev, ncols, diag_add, out, 0, nthreads);
}

/* Same draws, rounded only to float (used for synthetic K/V histories). */
void synth_normal_f32(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, double base,
                      double stdev, float *out, int nthreads) {
  run_normal(seed, tid, offset, n, base, stdev, 0, 0.0, 0, out, nthreads);
}

/* n integers uniform in [lo, hi]: lo + floor(hi32(out_k) * (hi - lo + 1) / 2^32). */
void synth_uniform_int(uint64_t seed, uint64_t tid, uint64_t n, int64_t lo, int64_t hi,
                       int32_t *out) {
  uint64_t key = stream_key(seed, tid);
  uint64_t span = (uint64_t)(hi - lo + 1);
  for (uint64_t k = 0; k < n; ++k) {
    uint64_t x = stream_out(key, k) >> 32;
    out[k] = (int32_t)(lo + (int64_t)((x * span) >> 32));
  }
}

/* Raw generator words, exposed so that tests can check the SplitMix64 stream. */
void synth_raw_u64(uint64_t seed, uint64_t tid, uint64_t n, uint64_t *out) {
  uint64_t key = stream_key(seed, tid);
  for (uint64_t k = 0; k < n; ++k) out[k] = stream_out(key, k);
}

uint64_t synth_mix64(uint64_t z) { return mix64(z); }
double synth_series_log(double x) {
  pthread_once(&coef_once, init_coefs);
  return series_log(x);
}
void synth_series_sincos(double x, double *s, double *c) {
  pthread_once(&coef_once, init_coefs);
  series_sincos(x, s, c);
}
