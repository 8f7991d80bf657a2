// grpo_prep.cu -- group-normalised advantages and per-sequence active-token
// counts, in one launch of 8-warp CTAs: the first ceil(G/8) CTAs give one
// warp to each group, the rest (when counting) one warp to the mask of each
// sequence.  In a shard call the groups span the whole batch (Bg sequences;
// advantages are replicated) while the masks are the shard's B sequences.
//
// RL-Kernel "GRPO Loss" page, "Accuracy": advantages are the group's rewards
// minus their mean over the population standard deviation clamped at
// adv_eps; "Group specification": uniform samples_per_prompt groups or CSR
// group_boundaries.  dockyard_rl "GRPO and the clipped policy-gradient
// loss", "Advantage estimation": a group whose rewards are all equal has
// zero advantage -- taken literally here (max == min gives A = 0 exactly).
// The mask scan yields L_i = sum_t mask[i,t] and the totals behind both
// normalisers ("Normalizer semantics"): N = sum_i L_i and S = #{i: L_i > 0},
// added with integer atomics (one per CTA), which are exact in any order.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kPrepWarps = 8;
static constexpr int kPrepThreads = 32 * kPrepWarps;

// Nonzero bytes of a 32-bit word are found through their top bits: the top
// bit of each nonzero byte is set by (x & 0x7F) + 0x7F or by x itself.

// Active tokens of one sequence, scanned by one warp: the count and the
// first and last active positions (-1 when there are none); every lane gets
// them.
struct SeqScan {
  int count, first, last;
};
__device__ __forceinline__ void scan_word(uint32_t x, int pos, SeqScan& s) {
  const uint32_t nz = (((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x) & 0x80808080u;
  s.count += __popc(nz);
  if (nz) {
    s.first = min(s.first, pos + ((__ffs(nz) - 1) >> 3));
    s.last = max(s.last, pos + ((31 - __clz(nz)) >> 3));
  }
}
__device__ __forceinline__ SeqScan warp_scan(const uint8_t* m, int64_t T, int lane) {
  SeqScan s{0, 0x7FFFFFFF, -1};
  const uintptr_t addr = (uintptr_t)m;
  int64_t head = (int64_t)((16 - (addr & 15)) & 15);
  if (head > T) head = T;
  const int64_t nvec = (T - head) / 16;
  const int64_t tail0 = head + nvec * 16;
  for (int64_t t = lane; t < head; t += 32)
    if (m[t]) { ++s.count; s.first = min(s.first, (int)t); s.last = max(s.last, (int)t); }
  for (int64_t t = tail0 + lane; t < T; t += 32)
    if (m[t]) { ++s.count; s.first = min(s.first, (int)t); s.last = max(s.last, (int)t); }
  const uint4* mv = reinterpret_cast<const uint4*>(m + head);
#pragma unroll 8
  for (int64_t k = lane; k < nvec; k += 32) {
    const uint4 v = __ldg(mv + k);
    const int pos = (int)(head + 16 * k);
    scan_word(v.x, pos, s);
    scan_word(v.y, pos + 4, s);
    scan_word(v.z, pos + 8, s);
    scan_word(v.w, pos + 12, s);
  }
  s.count = warp_sum(s.count);
  s.first = __reduce_min_sync(0xFFFFFFFFu, s.first);
  s.last = __reduce_max_sync(0xFFFFFFFFu, s.last);
  return s;
}

// Advantages of one group, by one warp.  Every sum runs over the lanes'
// strided elements in index order and then a fixed xor tree.
__device__ void warp_group(const PrepArgs& a, int64_t g, int lane) {
  int64_t lo, hi;
  if (a.bounds == nullptr) {
    lo = g * (int64_t)a.spp;
    hi = lo + a.spp;
  } else {
    lo = a.bounds[g];
    hi = a.bounds[g + 1];
    bool bad = !(lo >= 0 && hi > lo && hi <= a.Bg);
    if (g == 0 && lo != 0) bad = true;
    if (g == a.G - 1 && hi != a.Bg) bad = true;
    if (bad) {
      if (lane == 0) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_CSR);
      // keep every index in range; the outputs are NaN through the status word
      lo = lo < 0 ? 0 : (lo > a.Bg ? a.Bg : lo);
      hi = hi < lo ? lo : (hi > a.Bg ? a.Bg : hi);
    }
  }
  const int64_t n = hi - lo;

  double sum = 0.0;
  int nonfinite = 0;
  float mx = -INFINITY, mn = INFINITY;
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const float r = __ldg(a.rewards + i);
    nonfinite += !isfinite(r);
    sum += (double)r;
    mx = fmaxf(mx, r);
    mn = fminf(mn, r);
  }
  sum = warp_sum(sum);
  nonfinite = warp_sum(nonfinite);
  mx = warp_max(mx);
  mn = -warp_max(-mn);
  if (nonfinite > 0 && lane == 0) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_NONFINITE_REWARD);
  const double mean = n > 0 ? sum / (double)n : 0.0;

  double ss = 0.0;  // population variance
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const double d = (double)__ldg(a.rewards + i) - mean;
    ss += d * d;
  }
  ss = warp_sum(ss);
  const double sd = n > 0 ? sqrt(ss / (double)n) : 0.0;
  const double eps = (double)a.adv_eps;
  const double den = a.eps_add ? sd + eps : (sd > eps ? sd : eps);
  const bool degenerate = !(mx > mn);

  for (int64_t i = lo + lane; i < hi; i += 32) {
    const double Ai = degenerate ? 0.0 : ((double)__ldg(a.rewards + i) - mean) / den;
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
