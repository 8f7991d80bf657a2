// grpo_reduce.cu -- the deterministic two-level reduction of the logits path.
//
// RL-Kernel "GRPO Loss" page, "Tensor and Data Parallel", step 3: two nested
// reductions with fixed extents -- the T token slots of a sequence to one
// sequence total, then the B sequence totals to the scalar -- and the
// normaliser of "Normalizer semantics": the global active-token count (token
// mean) or the per-sequence count followed by a mean over live sequences.
//
// One CTA per sequence forms its totals; the CTA that finishes last (an
// atomic ticket, one per CTA, that nobody waits on) forms the scalar from the
// B totals.  Every sum has an order fixed by the code (thread-strided partial
// sums, xor-shuffle trees, warps in index order, sequences in index order),
// never by scheduling, so the result is bitwise reproducible.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceArgs a) {
  __shared__ double s_d[32 * 2];
  __shared__ bool s_last;
  const int64_t i = blockIdx.x;

  // level 1: sequence i.  Slots hold p + A (the policy term plus its constant
  // part, see the row kernel); the constant -A_i per token is added here.
  if (i < a.B) {
    const uint8_t* m = a.mask + i * a.T;
    const double* sp = a.slot_p + i * a.T;
    const double* sk = a.slot_k + i * a.T;
    double v[2] = {0.0, 0.0};
    for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x)
      if (m[t]) {
        v[0] += sp[t];
        v[1] += sk[t];
      }
    block_sum<double, 2>(v, s_d);
    if (threadIdx.x == 0) {
      const int L = a.L[i];
      const double P = a.split_A ? v[0] - a.A[i] * (double)L : v[0];
      a.seq[i] = P;
      a.seq[a.B + i] = v[1];
      if (a.per_seq) {
        a.per_seq[i] = (float)P;
        a.per_seq[a.B + i] = (float)v[1];
        a.per_seq[2 * a.B + i] = (float)L;
      }
      __threadfence();
      const unsigned ticket = atomicAdd(&a.hdr->done_ctas, 1u);
      s_last = ticket == gridDim.x - 1;
    }
  } else if (threadIdx.x == 0) {
    s_last = true;  // B == 0: a single CTA writes the zero loss
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // level 2: the scalar, over the B sequence totals in index order
  double u[2] = {0.0, 0.0};
  seq_totals(a.seq, a.L, a.B, a.reduction, u);
  block_sum<double, 2>(u, s_d);
  if (threadIdx.x == 0) {
    // N = active tokens, S = live sequences, as prep counted them
    const long long N = a.B > 0 ? a.hdr->N : 0, S = a.B > 0 ? a.hdr->S : 0;
    const double den = a.reduction == GRPO_TOKEN_MEAN      ? (double)(N > 0 ? N : 1)
                       : a.reduction == GRPO_SEQUENCE_MEAN ? (double)(S > 0 ? S : 1)
                                                           : (double)a.norm_c;
    const double P = u[0] / den, K = u[1] / den;
    float o0 = (float)(P + (double)a.beta * K), o1 = (float)P, o2 = (float)K;
    if (((volatile unsigned*)&a.hdr->status)[0] != 0u) o0 = o1 = o2 = NAN;
    a.out3[0] = o0;
    a.out3[1] = o1;
    a.out3[2] = o2;
    if (a.counts_out)  // every row kernel CTA added its counts before this launch
      for (int j = 0; j < 3; ++j) a.counts_out[j] = a.hdr->clip[j];
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  const int64_t grid = a.B > 0 ? a.B : 1;
  reduce_kernel<<<(unsigned)grid, kReduceThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
