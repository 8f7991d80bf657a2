/*
 * synth_cuda.cu -- device side of the seeded input generator.
 *
 * Fills whole logit tensors in HBM with exactly the bits synth_host.c
 * produces for the same (seed, index).  Compiled with -fmad=false so that no
 * multiply-add is contracted and every double operation is the correctly
 * rounded IEEE one, as on the host.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

__global__ void synth_logits_kernel(uint64_t seed, int dtype, int is_ref,
                                    int64_t n, double sigma, double spike_p,
                                    double spike_mag, double ref_sigma,
                                    void *out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    uint32_t b = synth_logit_bits(seed, (uint64_t)i, dtype, is_ref, sigma,
                                  spike_p, spike_mag, ref_sigma);
    if (dtype == SYNTH_BF16)
      ((uint16_t *)out)[i] = (uint16_t)b;
    else
      ((uint32_t *)out)[i] = b;
  }
}

/* Fill the first n elements (flat index 0..n-1 of a [*, V] tensor) on
 * `stream`.  Returns a cudaError_t as int. */
extern "C" int synth_cuda_logits(uint64_t seed, int dtype, int is_ref, int64_t n,
                                 double sigma, double spike_p, double spike_mag,
                                 double ref_sigma, void *out, void *stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  synth_logits_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      seed, dtype, is_ref, n, sigma, spike_p, spike_mag, ref_sigma, out);
  return (int)cudaGetLastError();
}
