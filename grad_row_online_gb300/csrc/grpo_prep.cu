// grpo_prep.cu -- group-normalised advantages and per-sequence active-token
// counts, in one launch of 8-warp CTAs: the first ceil(G/8) CTAs give one
// warp to each group, the rest (when counting) one warp to the mask of each
// sequence.  In a shard call the groups span the whole batch (Bg sequences;
// advantages are replicated) while the masks are the shard's B sequences.
// The warp-level scan and group statistics (grpo_groups.cuh) are shared with
// the one-launch form of the logps kernel.
//
// The mask scan yields L_i = sum_t mask[i,t] and the totals behind both
// normalisers (RL-Kernel "GRPO Loss", "Normalizer semantics"):
// N = sum_i L_i and S = #{i: L_i > 0}, added with integer atomics (one per
// CTA), which are exact in any order.
#include "grpo_groups.cuh"

namespace grpo {

static constexpr int kPrepWarps = 8;
static constexpr int kPrepThreads = 32 * kPrepWarps;

// Advantages of one group, by one warp.
__device__ void warp_group(const PrepArgs& a, int64_t g, int lane) {
  int64_t lo, hi;
  if (!group_bounds(a.bounds, a.spp, a.G, a.Bg, g, lo, hi) && lane == 0)
    atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_CSR);
  const GroupStats gs = warp_group_stats(a.rewards, lo, hi, a.adv_eps, a.eps_add, lane);
  if (gs.nonfinite > 0 && lane == 0) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_NONFINITE_REWARD);
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const double Ai = group_adv(gs, __ldg(a.rewards + i));
    a.A[i] = Ai;
    if (a.Aff) {
      const float hi = (float)Ai;
      a.Aff[i] = make_float2(hi, (float)(Ai - (double)hi));
    }
    if (a.adv_out && i >= a.seq_begin && i < a.seq_begin + a.B)
      a.adv_out[i - a.seq_begin] = (float)Ai;
  }
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepArgs a) {
  __shared__ int s_L[kPrepWarps];
  // a dependent kernel launched with programmatic stream serialization (the
  // logps kernel) may start its prologue now; it waits for this grid's
  // completion (griddepcontrol.wait) before reading anything written here
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t group_ctas = (a.G + kPrepWarps - 1) / kPrepWarps;
  if ((int64_t)blockIdx.x < group_ctas) {
    const int64_t g = (int64_t)blockIdx.x * kPrepWarps + warp;
    if (g < a.G) warp_group(a, g, lane);
    return;
  }
  // active-token counts: one warp per sequence, one pair of atomics per CTA
  const int64_t i = ((int64_t)blockIdx.x - group_ctas) * kPrepWarps + warp;
  int L = 0;
  if (i < a.B) {
    const SeqScan sc = warp_scan(a.mask + i * a.T, a.T, lane);
    L = sc.count;
    if (lane == 0) {
      if (a.L) a.L[i] = L;
      if (a.range) a.range[i] = L > 0 ? make_int2(sc.first, sc.last + 1) : make_int2(0, 0);
    }
  }
  if (lane == 0) s_L[warp] = L;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long n = 0, s = 0;
#pragma unroll
    for (int k = 0; k < kPrepWarps; ++k) {
      n += (unsigned long long)s_L[k];
      s += s_L[k] > 0;
    }
    if (n) atomicAdd(&a.NS[0], n);
    if (s) atomicAdd(&a.NS[1], s);
  }
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  const int64_t grid = (a.G + kPrepWarps - 1) / kPrepWarps +
                       (a.count ? (a.B + kPrepWarps - 1) / kPrepWarps : 0);
  if (grid <= 0) return cudaSuccess;
  prep_kernel<<<(unsigned)grid, kPrepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
