/*
 * synth_host.c -- host (CPU) side of the seeded input generator.
 *
 * Bulk fills built on synth_core.h.  Compiled with gcc -O2 -fopenmp
 * -ffp-contract=off; the device twin in synth_cuda.cu gives identical bits.
 * Element order never changes a value (each one is a pure function of its
 * index), so the OpenMP loops are free to split the work any way.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#include "synth_core.h"

/* Logit rows: out[r, v] = element (rows[r], v) of a [*, V] tensor.
 * dtype SYNTH_F32 -> out is float[nrows*V]; SYNTH_BF16 -> uint16_t[nrows*V]. */
void synth_host_logit_rows(uint64_t seed, int dtype, int is_ref,
                           const int64_t *rows, int64_t nrows, int64_t V,
                           double sigma, double spike_p, double spike_mag,
                           double ref_sigma, void *out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    uint64_t base = (uint64_t)rows[r] * (uint64_t)V;
    for (int64_t v = 0; v < V; ++v) {
      uint32_t b = synth_logit_bits(seed, base + (uint64_t)v, dtype, is_ref,
                                    sigma, spike_p, spike_mag, ref_sigma);
      if (dtype == SYNTH_BF16)
        ((uint16_t *)out)[r * V + v] = (uint16_t)b;
      else
        ((uint32_t *)out)[r * V + v] = b;
    }
  }
}

/* out[i] = N(0,1) deviate of element start+i in `stream`. */
void synth_host_normal(uint64_t seed, uint32_t stream, int64_t start, int64_t n,
                       double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_normal(seed, stream, (uint64_t)(start + i));
}

/* out[i] = uniform [0,1) draw `draw` of element start+i in `stream`. */
void synth_host_uniform(uint64_t seed, uint32_t stream, int64_t start, int64_t n,
                        uint32_t draw, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_u01(synth_bits(seed, stream, (uint64_t)(start + i), draw));
}

/* out[i] = uniform integer in [0, bound) for element start+i in `stream`. */
void synth_host_below(uint64_t seed, uint32_t stream, int64_t start, int64_t n,
                      uint32_t draw, uint64_t bound, int64_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (int64_t)synth_below(
        synth_bits(seed, stream, (uint64_t)(start + i), draw), bound);
}
