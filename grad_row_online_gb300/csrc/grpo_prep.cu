// grpo_prep.cu -- group-normalised advantages and per-sequence active-token
// counts, in one launch: CTAs [0, G) take a group each, CTAs [G, G+B) the
// mask of one sequence each.
//
// RL-Kernel "GRPO Loss" page, "Accuracy": advantages are the group's rewards
// minus their mean over the population standard deviation clamped at
// adv_eps; "Group specification": uniform samples_per_prompt groups or CSR
// group_boundaries.  dockyard_rl "GRPO and the clipped policy-gradient
// loss", "Advantage estimation": a group whose rewards are all equal has
// zero advantage -- taken literally here (max == min gives A = 0 exactly).
// The mask scan yields L_i = sum_t mask[i,t], the counts behind both
// normalisers ("Normalizer semantics").
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepArgs a) {
  __shared__ double s_red[32 * 3];
  __shared__ float s_fred[32];
  __shared__ int s_bad;
  if ((int64_t)blockIdx.x >= a.G) {  // active-token count of one sequence
    const int64_t i = blockIdx.x - a.G;
    const uint8_t* m = a.mask + i * a.T;
    int cnt = 0;
    const uintptr_t addr = (uintptr_t)m;
    int64_t head = (int64_t)((16 - (addr & 15)) & 15);
    if (head > a.T) head = a.T;
    const int64_t nvec = (a.T - head) / 16;
    const int64_t tail0 = head + nvec * 16;
    for (int64_t t = threadIdx.x; t < head; t += blockDim.x) cnt += m[t] != 0;
    for (int64_t t = tail0 + threadIdx.x; t < a.T; t += blockDim.x) cnt += m[t] != 0;
    const uint4* mv = reinterpret_cast<const uint4*>(m + head);
    for (int64_t k = threadIdx.x; k < nvec; k += blockDim.x) {
      const uint4 v = __ldg(mv + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // count nonzero bytes: set the top bit of each nonzero byte
        const uint32_t x = w[q];
        const uint32_t nz = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x;
        cnt += __popc(nz & 0x80808080u);
      }
    }
    int c1[1] = {cnt};
    block_sum<int, 1>(c1, reinterpret_cast<int*>(s_red));
    if (threadIdx.x == 0) a.L[i] = c1[0];
    return;
  }
  const int64_t g = blockIdx.x;

  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();

  int64_t lo, hi;
  if (a.bounds == nullptr) {
    lo = g * (int64_t)a.spp;
    hi = lo + a.spp;
  } else {
    lo = a.bounds[g];
    hi = a.bounds[g + 1];
    if (threadIdx.x == 0) {
      bool bad = !(lo >= 0 && hi > lo && hi <= a.B);
      if (g == 0 && lo != 0) bad = true;
      if (g == a.G - 1 && hi != a.B) bad = true;
      if (bad) {
        atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_CSR);
        s_bad = 1;
      }
    }
    __syncthreads();
    if (s_bad) {
      // keep every index in range; the outputs are NaN through the status word
      lo = lo < 0 ? 0 : (lo > a.B ? a.B : lo);
      hi = hi < lo ? lo : (hi > a.B ? a.B : hi);
    }
  }
  const int64_t n = hi - lo;

  // ---- mean, max, min (fixed-order block sums) ----
  double acc[3] = {0.0, 0.0, 0.0};  // sum, non-finite count, unused
  float mx = -INFINITY, mn = INFINITY;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    float r = __ldg(a.rewards + i);
    if (!isfinite(r)) acc[1] += 1.0;
    acc[0] += (double)r;
    mx = fmaxf(mx, r);
    mn = fminf(mn, r);
  }
  block_sum<double, 3>(acc, s_red);
  const float gmax = block_max(mx, s_fred);
  const float gmin = -block_max(-mn, s_fred);
  if (acc[1] > 0.0 && threadIdx.x == 0)
    atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_NONFINITE_REWARD);
  const double mean = n > 0 ? acc[0] / (double)n : 0.0;

  // ---- population variance ----
  double ss[1] = {0.0};
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    double d = (double)__ldg(a.rewards + i) - mean;
    ss[0] += d * d;
  }
  block_sum<double, 1>(ss, s_red);
  const double sd = n > 0 ? sqrt(ss[0] / (double)n) : 0.0;
  const double eps = (double)a.adv_eps;
  const double den = a.eps_add ? sd + eps : (sd > eps ? sd : eps);
  const bool degenerate = !(gmax > gmin);

  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    double Ai = degenerate ? 0.0 : ((double)__ldg(a.rewards + i) - mean) / den;
    a.A[i] = Ai;
    if (a.adv_out) a.adv_out[i] = (float)Ai;
  }

}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  const int64_t grid = a.G + (a.count ? a.B : 0);
  if (grid <= 0) return cudaSuccess;
  prep_kernel<<<(unsigned)grid, kPrepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
