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
//
// Sequence sharding (same page, steps 2-6): a shard call writes its
// sequences' totals and stops; finalize_kernel forms the scalar from the
// totals of all shards, concatenated in shard order, with the same
// final_scalar code the unsharded last CTA runs -- the same bits at any
// degree.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceArgs a) {
  __shared__ double s_d[32 * 2];
  __shared__ unsigned s_u[3 * 32];
  __shared__ double s_em;
  __shared__ FinalSmem s_fin;
  __shared__ bool s_last;
  const int64_t i = blockIdx.x;

  // level 1: sequence i.  Slots hold the policy term plus A for the clipped
  // surrogate (see the row kernel); the constant -A_i per token is added here.
  if (i < a.B) {
    const uint8_t* m = a.mask + i * a.T;
    const double* sp = a.slot_p + i * a.T;
    double* sk = a.slot_k + i * a.T;
    const int L = a.L[i];
    double v[2] = {0.0, 0.0};
    unsigned nc[3] = {0u, 0u, 0u};
    if (a.from_slots) {
      // The slots hold logp and d = ref_logp - logp (GSPO's first sweep, or
      // the vocab-parallel merge).  GSPO: rho_i first (a fixed-order sum over
      // the sequence), used by every token in place of its own ratio.  Then
      // every token's terms in double, and w = dL/dlogp.
      double em_seq = 0.0;
      if (a.var.seq_ratio) {
        double s1[1] = {0.0};
        for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x)
          if (m[t]) s1[0] += sp[t] - (double)a.old[i * a.T + t];
        block_sum<double, 1>(s1, s_d);
        if (threadIdx.x == 0) s_em = L > 0 ? expm1(s1[0] / (double)L) : 0.0;
        __syncthreads();
        em_seq = s_em;
      }
      const double A = a.A[i];
      const unsigned long long N = a.NS[0], S = a.NS[1];
      const double c = a.reduction == GRPO_TOKEN_MEAN ? 1.0 / (double)(N > 0 ? N : 1)
                       : a.reduction == GRPO_SEQUENCE_MEAN
                           ? (L > 0 ? 1.0 / ((double)(S > 0 ? S : 1) * (double)L) : 0.0)
                           : 1.0 / (double)a.norm_c;
      double* wo = a.w_out ? a.w_out + i * a.T : sk;
      for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x)
        if (m[t]) {
          const double lp = sp[t], d = sk[t], emd = expm1(d);
          const double em = a.var.seq_ratio ? em_seq : expm1(lp - (double)a.old[i * a.T + t]);
          const TokEpi<double> te = token_epilogue<double>(em, lp, d, emd, emd - d, true, A, a.var);
          v[0] += te.q;
          v[1] += te.k;
          wo[t] = (double)a.grad_scale * c * te.g;
          if (te.clip == 1) ++nc[0];
          else if (te.clip == 2) ++nc[1];
          else if (te.clip == 3) ++nc[2];
        }
    } else {
      for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x)
        if (m[t]) {
          v[0] += sp[t];
          v[1] += sk[t];
        }
    }
    block_sum<double, 2>(v, s_d);
    if (a.from_slots && a.counts_out) block_sum<unsigned, 3>(nc, s_u);
    if (threadIdx.x == 0) {
      const double P = a.split_A ? v[0] - a.A[i] * (double)L : v[0];
      put_total(a.seq + i, P, v[1], L);
      if (a.per_seq) {
        a.per_seq[i] = (float)P;
        a.per_seq[a.B + i] = (float)v[1];
        a.per_seq[2 * a.B + i] = (float)L;
      }
      if (a.from_slots && a.counts_out) add_clip_counts(a.hdr, nc);
      __threadfence();
      const unsigned ticket = atomicAdd(&a.hdr->done_ctas, 1u);
      s_last = ticket == gridDim.x - 1;
    }
  } else if (threadIdx.x == 0) {
    s_last = true;  // B == 0: a single CTA
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the clip counts: the row kernel added its before this launch, the GSPO
  // step above before each CTA's ticket
  if (threadIdx.x == 0 && a.counts_out)
    for (int j = 0; j < 3; ++j) a.counts_out[j] = __ldcg(&a.hdr->clip[j]);
  if (a.shard) return;  // the scalar comes from grpo_loss_finalize over all shards' totals

  // level 2: the scalar, over the B sequence records in index order
  const bool bad = ((volatile unsigned*)&a.hdr->status)[0] != 0u;
  final_scalar(a.seq, a.B, a.B > 0 ? a.NS[0] : 0ull, a.B > 0 ? a.NS[1] : 0ull, a.reduction,
               a.norm_c, a.beta, bad, a.out3, s_fin);
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  const int64_t grid = a.B > 0 ? a.B : 1;
  reduce_kernel<<<(unsigned)grid, kReduceThreads, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kFinalThreads) finalize_kernel(const SeqTotal* recs, int64_t B,
                                                                const unsigned long long* NS,
                                                                int reduction, float norm_c,
                                                                float beta, float* out3) {
  __shared__ FinalSmem s_fin;
  final_scalar(recs, B, B > 0 ? NS[0] : 0ull, B > 0 ? NS[1] : 0ull, reduction, norm_c, beta,
               false, out3, s_fin);
}

cudaError_t launch_finalize(const SeqTotal* recs, int64_t B, const unsigned long long* NS,
                            int reduction, float norm_c, float beta, float* out3, cudaStream_t s) {
  finalize_kernel<<<1, kFinalThreads, 0, s>>>(recs, B, NS, reduction, norm_c, beta, out3);
  return cudaGetLastError();
}

}  // namespace grpo
