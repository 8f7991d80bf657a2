// grpo_reduce.cu -- the deterministic two-level reduction of the logits path.
//
// RL-Kernel "GRPO Loss" page, "Tensor and Data Parallel", step 3: two nested
// reductions with fixed extents -- the T token slots of a sequence to one
// sequence total, then the B sequence totals to the scalar -- and the
// normaliser of "Normalizer semantics": the global active-token count (token
// mean) or the per-sequence count followed by a mean over live sequences.
// The summation order is fixed by the code (lane-strided partial sums, an
// xor-shuffle tree, a fixed warp order), never by scheduling, so the result
// is bitwise reproducible.  Single CTA: the per-token slots are B*T doubles,
// a few hundred kilobytes for vocabulary-sized rows.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceArgs a) {
  __shared__ double s_d[32 * 3];
  __shared__ long long s_l[64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;

  long long ns[2] = {0, 0};
  for (int64_t i = threadIdx.x; i < a.B; i += blockDim.x) {
    int L = a.L[i];
    ns[0] += L;
    ns[1] += L > 0;
  }
  block_sum<long long, 2>(ns, s_l);
  const long long N = ns[0], S = ns[1];

  // level 1: warp w owns sequences w, w + nw, ...; its lanes take the token
  // slots t = lane, lane + 32, ... in order, then an xor-shuffle tree gives
  // the sequence totals P_i, K_i.  Lane 0 folds them, in sequence order, into
  // this warp's share of the scalar numerator.
  double pol = 0.0, kl = 0.0;
  for (int64_t i = warp; i < a.B; i += nw) {
    const uint8_t* m = a.mask + i * a.T;
    const double* sp = a.slot_p + i * a.T;
    const double* sk = a.slot_k + i * a.T;
    double P = 0.0, K = 0.0;
    for (int64_t t = lane; t < a.T; t += 32)
      if (m[t]) {
        P += sp[t];
        K += sk[t];
      }
    P = warp_sum(P);
    K = warp_sum(K);
    const int L = a.L[i];
    P -= a.A[i] * (double)L;  // slots hold p + A: the constant -A per token, summed here
    if (lane == 0) {
      if (a.per_seq) {
        a.per_seq[i] = (float)P;
        a.per_seq[a.B + i] = (float)K;
        a.per_seq[2 * a.B + i] = (float)L;
      }
      if (a.reduction == GRPO_TOKEN_MEAN) {
        pol += P;
        kl += K;
      } else if (L > 0) {
        pol += P / (double)L;
        kl += K / (double)L;
      }
    }
  }
  // level 2: warps in fixed order
  __syncthreads();
  if (lane == 0) {
    s_d[warp] = pol;
    s_d[32 + warp] = kl;
  }
  __syncthreads();
  if (warp == 0) {
    double p = lane < nw ? s_d[lane] : 0.0;
    double k = lane < nw ? s_d[32 + lane] : 0.0;
    p = warp_sum(p);
    k = warp_sum(k);
    if (lane == 0) {
      const double den = a.reduction == GRPO_TOKEN_MEAN ? (double)(N > 0 ? N : 1)
                                                        : (double)(S > 0 ? S : 1);
      const double P = p / den, K = k / den;
      float o0 = (float)(P + (double)a.beta * K), o1 = (float)P, o2 = (float)K;
      if (a.hdr->status != 0u) o0 = o1 = o2 = NAN;
      a.out3[0] = o0;
      a.out3[1] = o1;
      a.out3[2] = o2;
    }
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  reduce_kernel<<<1, kReduceThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
