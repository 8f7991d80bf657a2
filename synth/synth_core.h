/*
 * synth_core.h -- seeded, counter-based generator of synthetic inputs.
 *
 * Shared by the host C build (synth_host.c, compiled with gcc
 * -ffp-contract=off) and the device build (synth_cuda.cu, compiled with
 * nvcc -fmad=false).  Every value is a pure function of
 * (seed, stream, index), so any element of any tensor can be regenerated
 * on its own, in any order, on either side, with identical bits.
 *
 * Only IEEE-754 operations that are correctly rounded on both sides are used
 * (+, -, *, /, sqrt on double; double->float conversion), never a libm or
 * CUDA transcendental, and contraction into FMA is disabled by the build
 * flags.  That is what makes the host and the device agree bit for bit.
 *
 * This file holds no arithmetic of the GRPO method: it draws random numbers.
 *
 * Methods used:
 *   - bit mixing: the SplitMix64 output function (Steele, Lea & Flood,
 *     "Fast splittable pseudorandom number generators", OOPSLA 2014),
 *     applied to a key built from (seed, stream, index, draw);
 *   - normal deviates: Marsaglia's polar method (Marsaglia & Bray 1964);
 *   - the natural log it needs: m*2^e decomposition plus the series
 *     ln m = 2 atanh((m-1)/(m+1)), written out here.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#ifdef __CUDACC__
#define SYNTH_FN __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

/* Streams: one independent sequence of draws per input tensor / purpose. */
enum {
  SYNTH_STREAM_POLICY = 1,   /* policy logits (normal) */
  SYNTH_STREAM_SPIKE = 2,    /* Bernoulli spikes added to policy logits */
  SYNTH_STREAM_REF = 3,      /* reference-logit perturbation (normal) */
  SYNTH_STREAM_ACTION = 4,   /* action ids (uniform integer) */
  SYNTH_STREAM_OLD = 5,      /* behaviour log-prob perturbation (normal) */
  SYNTH_STREAM_REWARD = 6,   /* rewards (Bernoulli or normal) */
  SYNTH_STREAM_LENGTH = 7,   /* completion lengths (uniform integer) */
  SYNTH_STREAM_GROUP = 8,    /* CSR group sizes (uniform integer) */
  SYNTH_STREAM_LOGP = 9,     /* log-probs of the logps-only workload (normal) */
  SYNTH_STREAM_REFLOGP = 10, /* reference log-prob perturbation (normal) */
  SYNTH_STREAM_HOLE = 11,    /* choice of fully-masked rows */
  SYNTH_STREAM_MISC = 12
};

enum { SYNTH_F32 = 0, SYNTH_BF16 = 1 };

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* 64 random bits for draw `draw` of element `index` in stream `stream`. */
SYNTH_FN uint64_t synth_bits(uint64_t seed, uint32_t stream, uint64_t index,
                             uint32_t draw) {
  uint64_t k = synth_mix64(seed ^ (0xD1B54A32D192ED03ull * (uint64_t)stream));
  k = synth_mix64(k ^ index);
  return synth_mix64(k + (uint64_t)draw);
}

/* Uniform double in [0, 1) with 53 random bits. */
SYNTH_FN double synth_u01(uint64_t bits) {
  return (double)(bits >> 11) * (1.0 / 9007199254740992.0);
}

/* Uniform integer in [0, n): high half of a 64x64 product (no modulo). */
SYNTH_FN uint64_t synth_below(uint64_t bits, uint64_t n) {
#ifdef __CUDA_ARCH__
  return __umul64hi(bits, n);
#else
  return (uint64_t)(((unsigned __int128)bits * (unsigned __int128)n) >> 64);
#endif
}

/* Natural log of a positive, finite, normal double.  Written from
 * ln(m 2^e) = e ln2 + 2 atanh(f), f = (m-1)/(m+1), m in [sqrt(1/2), sqrt(2)),
 * with the atanh series summed to f^23 (|f| <= 0.1716, remainder < 1e-19).
 * Accuracy is a few ulps; what matters here is that both builds give the
 * same bits, which the restriction to +,-,*,/ guarantees. */
SYNTH_FN double synth_log(double s) {
  union { double d; uint64_t u; } v;
  v.d = s;
  int e = (int)((v.u >> 52) & 0x7FF) - 1023;
  v.u = (v.u & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull; /* m in [1,2) */
  double m = v.d;
  if (m > 1.4142135623730951) { m = m * 0.5; e = e + 1; }
  double f = (m - 1.0) / (m + 1.0);
  double f2 = f * f;
  double p = 1.0 / 23.0;
  p = p * f2 + 1.0 / 21.0;
  p = p * f2 + 1.0 / 19.0;
  p = p * f2 + 1.0 / 17.0;
  p = p * f2 + 1.0 / 15.0;
  p = p * f2 + 1.0 / 13.0;
  p = p * f2 + 1.0 / 11.0;
  p = p * f2 + 1.0 / 9.0;
  p = p * f2 + 1.0 / 7.0;
  p = p * f2 + 1.0 / 5.0;
  p = p * f2 + 1.0 / 3.0;
  p = p * f2 + 1.0;
  const double ln2 = 0.69314718055994530942;
  return (double)e * ln2 + 2.0 * f * p;
}

/* Standard normal deviate for (seed, stream, index): polar method, one of
 * the pair is kept.  Draws (2j, 2j+1) form attempt j; after 64 rejected
 * attempts (probability ~1e-43) the value is 0. */
SYNTH_FN double synth_normal(uint64_t seed, uint32_t stream, uint64_t index) {
  for (uint32_t j = 0; j < 64; ++j) {
    double u = 2.0 * synth_u01(synth_bits(seed, stream, index, 2 * j)) - 1.0;
    double v = 2.0 * synth_u01(synth_bits(seed, stream, index, 2 * j + 1)) - 1.0;
    double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) {
      double q = (-2.0 * synth_log(s)) / s;
      return u * sqrt(q);
    }
  }
  return 0.0;
}

SYNTH_FN uint32_t synth_f32_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  return v.u;
}

SYNTH_FN float synth_bits_f32(uint32_t u) {
  union { float f; uint32_t u; } v;
  v.u = u;
  return v.f;
}

/* float -> bfloat16 bits, round to nearest even (inputs here are finite). */
SYNTH_FN uint16_t synth_f32_to_bf16(float f) {
  uint32_t u = synth_f32_bits(f);
  u = u + 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYNTH_FN float synth_bf16_to_f32(uint16_t h) {
  return synth_bits_f32(((uint32_t)h) << 16);
}

/* Logit value of a policy element before storage rounding:
 * sigma * N(0,1), plus spike_mag with probability spike_p. */
SYNTH_FN double synth_policy_value(uint64_t seed, uint64_t idx, double sigma,
                                   double spike_p, double spike_mag) {
  double v = sigma * synth_normal(seed, SYNTH_STREAM_POLICY, idx);
  if (spike_p > 0.0 &&
      synth_u01(synth_bits(seed, SYNTH_STREAM_SPIKE, idx, 0)) < spike_p)
    v = v + spike_mag;
  return v;
}

/* Stored policy / reference element, as the raw bits of the storage dtype
 * (f32 bits, or bf16 bits in the low 16).  The reference element is the
 * stored policy element plus ref_sigma * N(0,1), rounded again. */
SYNTH_FN uint32_t synth_logit_bits(uint64_t seed, uint64_t idx, int dtype,
                                   int is_ref, double sigma, double spike_p,
                                   double spike_mag, double ref_sigma) {
  double v = synth_policy_value(seed, idx, sigma, spike_p, spike_mag);
  float f = (float)v;
  uint32_t bits;
  double stored;
  if (dtype == SYNTH_BF16) {
    uint16_t h = synth_f32_to_bf16(f);
    bits = h;
    stored = (double)synth_bf16_to_f32(h);
  } else {
    bits = synth_f32_bits(f);
    stored = (double)f;
  }
  if (!is_ref) return bits;
  double r = stored + ref_sigma * synth_normal(seed, SYNTH_STREAM_REF, idx);
  float rf = (float)r;
  if (dtype == SYNTH_BF16) return synth_f32_to_bf16(rf);
  return synth_f32_bits(rf);
}

#endif /* SYNTH_CORE_H */
