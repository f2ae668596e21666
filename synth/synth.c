/*
 * synth.c -- seeded, counter-based synthetic input generator.
 *
 * This file produces the random inputs (activations, weights, router
 * parameters) that both the CUDA path and the CPU oracle consume.  It holds
 * none of the quantisation / matmul / routing arithmetic: only random-number
 * generation and input shaping (Gaussian draws, sparse outliers, a seeded
 * permutation, a Zipf-shaped logit bias, and a round-to-nearest-even cast to
 * bfloat16 for bf16 activations).
 *
 * Generator (counter based, so any sub-range of a tensor can be regenerated on
 * its own, e.g. a few weight rows for a sampled oracle check):
 *   key(seed, stream)  = mix64(seed ^ (stream * GAMMA))
 *   raw(seed, stream, c) = mix64(key + (c + 1) * GAMMA)      (the c-th output
 *                          of a SplitMix64 sequence started at key)
 *   mix64 is the SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable
 *   pseudorandom number generators", OOPSLA 2014).
 *   uniform53(r)       = (r >> 11) * 2^-53            in [0, 1)
 * Normal element i of a stream is the inverse normal CDF of one uniform:
 *   u = (2 * (raw(i) >> 11) + 1) * 2^-54          in (0, 1), never 0 or 1
 *   value = (float)(sigma * Phi^-1(u))
 * with Phi^-1 from P. J. Acklam's rational approximation ("An algorithm for
 * computing the inverse normal cumulative distribution function", 2003;
 * relative error below 1.15e-9): a rational function of u in the central
 * region 0.02425 <= u <= 0.97575 and of sqrt(-2 ln u) (or of 1-u) in the tails.
 * Outlier mask (independent stream): element i is an outlier when
 *   uniform53(raw_outlier(i)) < p ; its value is multiplied by `factor`.
 *
 * Parallelised with OpenMP over fixed chunks; every element depends only on
 * its own index, so the output does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ (stream * GAMMA));
}

static inline uint64_t raw_at(uint64_t key, uint64_t c) {
  return mix64(key + (c + 1ULL) * GAMMA);
}

static inline double uniform53(uint64_t r) {
  return (double)(r >> 11) * (1.0 / 9007199254740992.0);
}

uint64_t synth_raw(uint64_t seed, uint64_t stream, uint64_t counter) {
  return raw_at(stream_key(seed, stream), counter);
}

/* Inverse of the standard normal CDF (Acklam's rational approximation). */
static double inv_normal_cdf(double p) {
  static const double a[6] = {-3.969683028665376e+01, 2.209460984245205e+02,
                              -2.759285104469687e+02, 1.383577518672690e+02,
                              -3.066479806614716e+01, 2.506628277459239e+00};
  static const double b[5] = {-5.447609879822406e+01, 1.615858368580409e+02,
                              -1.556989798598866e+02, 6.680131188771972e+01,
                              -1.328068155288572e+01};
  static const double c[6] = {-7.784894002430293e-03, -3.223964580411365e-01,
                              -2.400758277161838e+00, -2.549732539343734e+00,
                              4.374664141464968e+00, 2.938163982698783e+00};
  static const double d[4] = {7.784695709041462e-03, 3.224671290700398e-01,
                              2.445134137142996e+00, 3.754408661907416e+00};
  const double plow = 0.02425, phigh = 1.0 - 0.02425;
  if (p < plow) {
    const double q = sqrt(-2.0 * log(p));
    return (((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
           ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1.0);
  }
  if (p > phigh) {
    const double q = sqrt(-2.0 * log(1.0 - p));
    return -(((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
           ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1.0);
  }
  const double q = p - 0.5, r = q * q;
  return (((((a[0] * r + a[1]) * r + a[2]) * r + a[3]) * r + a[4]) * r + a[5]) * q /
         (((((b[0] * r + b[1]) * r + b[2]) * r + b[3]) * r + b[4]) * r + 1.0);
}

/* out[t] = sigma * z[offset + t] for t < count. */
void synth_normal(uint64_t seed, uint64_t stream, uint64_t offset,
                  uint64_t count, double sigma, float *out) {
  const uint64_t key = stream_key(seed, stream);
  const int64_t n = (int64_t)count;
  #pragma omp parallel for schedule(static, 65536)
  for (int64_t t = 0; t < n; ++t) {
    const uint64_t r = raw_at(key, offset + (uint64_t)t);
    const double u = (double)(2 * (r >> 11) + 1) * (1.0 / 18014398509481984.0);
    out[t] = (float)(sigma * inv_normal_cdf(u));
  }
}

/* inout[t] *= factor where uniform(stream, offset + t) < p. Returns the
 * number of outliers applied. */
int64_t synth_outliers(uint64_t seed, uint64_t stream, uint64_t offset,
                       uint64_t count, double p, double factor, float *inout) {
  const uint64_t key = stream_key(seed, stream);
  const int64_t n = (int64_t)count;
  int64_t hits = 0;
  #pragma omp parallel for schedule(static, 65536) reduction(+ : hits)
  for (int64_t t = 0; t < n; ++t) {
    if (uniform53(raw_at(key, offset + (uint64_t)t)) < p) {
      inout[t] = (float)((double)inout[t] * factor);
      ++hits;
    }
  }
  return hits;
}

/* Round-to-nearest-even cast fp32 -> bfloat16 bit pattern (finite inputs;
 * NaN maps to a quiet NaN). */
void synth_to_bf16(const float *in, uint16_t *out, uint64_t count) {
  const int64_t n = (int64_t)count;
  #pragma omp parallel for schedule(static, 65536)
  for (int64_t t = 0; t < n; ++t) {
    union { float f; uint32_t u; } v;
    v.f = in[t];
    uint32_t u = v.u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
      out[t] = (uint16_t)((u >> 16) | 0x0040u);
    } else {
      const uint32_t lsb = (u >> 16) & 1u;
      out[t] = (uint16_t)((u + 0x7FFFu + lsb) >> 16);
    }
  }
}

/* Seeded Fisher-Yates permutation of 0..n-1 (swap partner for position i,
 * going down from n-1, is raw(stream, n-1-i) mod (i+1)). */
void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t *out) {
  const uint64_t key = stream_key(seed, stream);
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    const uint64_t r = raw_at(key, (uint64_t)(n - 1 - i));
    const int32_t j = (int32_t)(r % (uint64_t)(i + 1));
    const int32_t tmp = out[i];
    out[i] = out[j];
    out[j] = tmp;
  }
}

/* Zipf-shaped popularity bias: expert e gets rank r_e = 1 + position of e in
 * a seeded permutation, and bias[e] = -s * ln(r_e), so that exp(bias) is
 * proportional to r_e^-s. */
void synth_zipf_bias(uint64_t seed, uint64_t stream, int32_t n, double s,
                     float *bias) {
  int32_t perm[65536];
  if (n <= 0 || n > 65536) return;
  synth_permutation(seed, stream, n, perm);
  for (int32_t pos = 0; pos < n; ++pos) {
    bias[perm[pos]] = (float)(-s * log((double)(pos + 1)));
  }
}
