// grpo_groups.cuh -- warp-level pieces shared by the separate advantage /
// count pass (grpo_prep.cu) and the one-launch form of the logps kernel
// (grpo_logps.cu): the mask scan of one sequence and the advantage
// statistics of one group, so that both forms compute the same bits.
//
// RL-Kernel "GRPO Loss" page, "Accuracy": advantages are the group's rewards
// minus their mean over the population standard deviation clamped at
// adv_eps; "Group specification": uniform samples_per_prompt groups or CSR
// group_boundaries.  dockyard_rl "GRPO and the clipped policy-gradient
// loss", "Advantage estimation": a group whose rewards are all equal has
// zero advantage -- taken literally here (max == min gives A = 0 exactly).
#pragma once

#include "grpo_internal.cuh"

namespace grpo {

// Active tokens of one sequence, scanned by one warp: the count and the
// first and last active positions relative to the scanned piece (first =
// INT_MAX, last = -1 when there are none); every lane gets them.
// Nonzero bytes of a 32-bit word are found through their top bits: the top
// bit of each nonzero byte is set by (x & 0x7F) + 0x7F or by x itself.
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
  // rounds of kScanBatch 16-byte words per lane, all loaded before any is
  // scanned: a piece of up to 2 KB per warp costs one memory round trip
  constexpr int kScanBatch = 4;
  const uint4* mv = reinterpret_cast<const uint4*>(m + head);
  for (int64_t k0 = lane; k0 < nvec; k0 += 32 * kScanBatch) {
    uint4 v[kScanBatch];
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      const int64_t k = k0 + 32 * u;
      v[u] = k < nvec ? __ldg(mv + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      const int pos = (int)(head + 16 * (k0 + 32 * u));
      scan_word(v[u].x, pos, s);
      scan_word(v[u].y, pos + 4, s);
      scan_word(v[u].z, pos + 8, s);
      scan_word(v[u].w, pos + 12, s);
    }
  }
  s.count = warp_sum(s.count);
  s.first = __reduce_min_sync(0xFFFFFFFFu, s.first);
  s.last = __reduce_max_sync(0xFFFFFFFFu, s.last);
  return s;
}

// The sequences [lo, hi) of group g: uniform groups of spp, or the CSR
// entries, checked against the batch of Bg sequences (boundaries[0] = 0,
// boundaries[G] = Bg, strictly increasing).  A bad group is clamped into
// range and reported by the return value.
__device__ __forceinline__ bool group_bounds(const int64_t* bounds, int32_t spp, int64_t G,
                                             int64_t Bg, int64_t g, int64_t& lo, int64_t& hi) {
  if (bounds == nullptr) {
    lo = g * (int64_t)spp;
    hi = lo + spp;
    return true;
  }
  lo = bounds[g];
  hi = bounds[g + 1];
  bool bad = !(lo >= 0 && hi > lo && hi <= Bg);
  if (g == 0 && lo != 0) bad = true;
  if (g == G - 1 && hi != Bg) bad = true;
  if (bad) {  // keep every index in range; the outputs are NaN through the status word
    lo = lo < 0 ? 0 : (lo > Bg ? Bg : lo);
    hi = hi < lo ? lo : (hi > Bg ? Bg : hi);
  }
  return !bad;
}

// The group holding sequence gb of a CSR batch, by one warp: each round
// probes 32 boundaries evenly over [g0, g1) (bounds[g0] <= gb < bounds[g1]
// when the boundaries are valid) and keeps the last probe at or below gb,
// shrinking the range to a 32nd.  Any input ends inside [0, G).
__device__ __forceinline__ int64_t warp_find_group(const int64_t* bounds, int64_t G, int64_t gb,
                                                   int lane) {
  int64_t g0 = 0, g1 = G;
  while (g1 - g0 > 1) {
    const int64_t step = (g1 - g0 + 31) / 32;
    const int64_t p = g0 + (int64_t)lane * step;
    const bool le = p < g1 && __ldg(bounds + p) <= gb;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, le);
    const int k = m ? 31 - __clz((int)m) : 0;
    g0 += (int64_t)k * step;
    g1 = min(g0 + step, g1);
  }
  return g0;
}

// One group's statistics, by one warp, in float-pair arithmetic (about 46
// significant bits: the double-precision units of GB300 are a small
// fraction of its fp32 rate, and a dozen dependent double operations with
// divisions and a square root held the one-launch logps kernel for
// microseconds).  Every sum runs over the lanes' strided elements in index
// order, then the fixed xor tree; lane 0's result is broadcast, so every
// lane holds the same statistics.
struct GroupStats {
  FF mean, den;
  bool degenerate;  // max == min: every advantage of the group is 0
  int nonfinite;    // non-finite rewards in the group
};
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = __fmaf_rn(a.hi, b.hi, -p);
  return fast_two_sum(p, __fadd_rn(e, __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi))));
}
// sqrt of a non-negative float pair: the fp32 root, then one Newton
// correction from the exact residual a - s^2.
__device__ __forceinline__ FF ff_sqrt(FF a) {
  if (!(a.hi > 0.f)) return {0.f, 0.f};
  const float s = __fsqrt_rn(a.hi);
  const float p = __fmul_rn(s, s);
  const float e = __fmaf_rn(s, s, -p);
  const float r = __fadd_rn(__fsub_rn(__fsub_rn(a.hi, p), e), a.lo);
  return fast_two_sum(s, __fdiv_rn(r, __fmul_rn(2.f, s)));
}
__device__ __forceinline__ FF ff_bcast0(FF v) {
  return {__shfl_sync(0xFFFFFFFFu, v.hi, 0), __shfl_sync(0xFFFFFFFFu, v.lo, 0)};
}
__device__ __forceinline__ GroupStats warp_group_stats(const float* rewards, int64_t lo,
                                                       int64_t hi, float adv_eps, int eps_add,
                                                       int lane) {
  const int64_t n = hi - lo;
  FF sum = {0.f, 0.f};
  int nonfinite = 0;
  float mx = -INFINITY, mn = INFINITY;
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const float r = __ldg(rewards + i);
    nonfinite += !isfinite(r);
    sum = ff_add(sum, FF{r, 0.f});
    mx = fmaxf(mx, r);
    mn = fminf(mn, r);
  }
  sum = ff_bcast0(warp_sum_ff2(sum));
  GroupStats g;
  g.nonfinite = warp_sum(nonfinite);
  mx = warp_max(mx);
  mn = -warp_max(-mn);
  const FF nf = ff_from_u64((unsigned long long)(n > 0 ? n : 1));
  g.mean = n > 0 ? ff_div(sum, nf) : FF{0.f, 0.f};

  FF ss = {0.f, 0.f};  // population variance
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const FF d = ff_add(FF{__ldg(rewards + i), 0.f}, ff_neg(g.mean));
    ss = ff_add(ss, ff_mul(d, d));
  }
  ss = ff_bcast0(warp_sum_ff2(ss));
  const FF sd = n > 0 ? ff_sqrt(ff_div(ss, nf)) : FF{0.f, 0.f};
  const FF eps = {adv_eps, 0.f};
  if (eps_add) {
    g.den = ff_add(sd, eps);
  } else {  // max(sd, eps)
    const bool above = sd.hi > adv_eps || (sd.hi == adv_eps && sd.lo > 0.f);
    g.den = above ? sd : eps;
  }
  g.degenerate = !(mx > mn);
  return g;
}

// The advantage of a reward r of the group, as a double (the float pair's
// exact sum).
__device__ __forceinline__ double group_adv(const GroupStats& g, float r) {
  if (g.degenerate) return 0.0;
  const FF a = ff_div(ff_add(FF{r, 0.f}, ff_neg(g.mean)), g.den);
  return (double)a.hi + (double)a.lo;
}

}  // namespace grpo
