// grpo_rows_common.cuh -- the per-row arithmetic of the fused row kernel
// (grpo_rows.cu): geometry of a row, the block combine of the online
// normalisers, the row finish (fast: fp32 / float-float; precise: double),
// and the gradient element.
#pragma once

#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kRowThreads = 256;
static constexpr int kRowBlocksPerSM = 4;
static constexpr int kUnroll = 4;        // 16-byte vectors in flight per thread, one row
static constexpr int kPairUnroll = 3;    // ... per row when policy and reference stream together
static constexpr int kGradUnroll = 4;    // ... in the gradient sweep
static constexpr bool kReverseSweep2 = true;
// The first kPolicySmemBytes of the policy row are kept in shared memory
// between the sweeps: with sweep 2 back to front they are the lines read
// longest ago, the ones L2 would have lost.
static constexpr int kPolicySmemBytes = 44 * 1024;
static constexpr int kPolicySmemVecs = kPolicySmemBytes / 16;
// Tensor memory as a second kept slice.  Nothing on this path is a
// contraction, so the SM's 256 KB of tensor memory (128 lanes x 512 columns
// of 32 bits) is free: each CTA allocates kTmemCols columns (all of it at
// four CTAs per SM) and keeps there the policy vectors that follow the shared
// memory slice, kTmemVecs per thread (64 KB per row).  A warp may touch only
// the 32 lanes of its quadrant (warp index mod 4), so warps w and w + 4 split
// the columns: thread t of warp w keeps its vectors in lane 32 (w mod 4) + t,
// columns (w / 4) kTmemCols / 2 + 4 i.  The vectors of a thread are
// t + kRowThreads j (the sweeps' order); shared memory holds j < kSmemJ,
// tensor memory kSmemJ <= j < kSmemJ + kTmemVecs.
static constexpr int kTmemCols = 128;
static constexpr int kTmemVecs = kTmemCols / 2 / 4;
static constexpr int kSmemJ = kPolicySmemVecs / kRowThreads;
static_assert(kPolicySmemVecs % kRowThreads == 0, "the shared slice must end on a sweep step");
static_assert(kRowThreads == 256, "two warps per tensor-memory lane quadrant");
static_assert(kTmemVecs % 2 == 0, "tensor memory is read back two vectors at a time");
// Refinement.  The fast logsumexp of a row has an absolute error below
// kFastErrBound (the normaliser's relative error, below 2^-19, plus the
// float-float finish's ~1e-7).  An element of the fp32 gradient stays within
// one ulp + 1e-9 of the exact value when (that error) x (the sensitivity of
// the element to the logsumexp) stays below kTau, which leaves ~2e-10 for
// the roundings of w and p_v.  The policy row is refined when its
// sensitivity |w| + |dw/dlogp| crosses the line, the reference row when
// |dw/dref_logp| = |grad_scale c beta e^d| does.
static constexpr float kFastErrBound = 2.2e-6f;
static constexpr float kTau = 8.0e-10f;
static constexpr float kElemPrecise = 0x1p-12f;

struct RowScalars {
  double lse_p, w;
  double q, k, logp;  // q = policy term + A (the constant -A is summed per sequence)
  float LL;           // logsumexp of the policy row in base 2: p_v = 2^(x_v log2e - LL)
  float wneg;         // -w as float
  float ga;           // gradient at the action element
  int precise;      // bit 0: policy row refined, bit 1: reference row refined
  int clip;         // 0, or the clip that bound: 1 upper, 2 lower, 3 dual
  double dlr;       // ref_logp - logp
};

// --------------------------------------------------------- tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(d),
               "r"(ncols)
               : "memory");
}
// A kernel that may allocate tensor memory gets another CTA on an SM only
// once the resident ones have given up the right to allocate (measured: a
// CTA that never does runs alone on its SM), so every CTA of such a kernel
// gives it up at once, whether it allocated or not.
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// this thread's lane and first column in a CTA's allocation `base` whose
// warps w and w + 4 share a lane quadrant, `half` columns each
__device__ __forceinline__ uint32_t tmem_thread_base(uint32_t base, uint32_t half) {
  const uint32_t warp = threadIdx.x >> 5;
  return base + ((warp & 3u) << 21) + (warp >> 2) * half;
}
// one 16-byte vector into 4 columns of this thread's lane (warp-collective)
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4& v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// two vectors (8 columns) of this thread's lane back, waited for in the same
// statement so no use of the registers can be scheduled before the data lands
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint4 (&v)[2]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0].x), "=r"(v[0].y), "=r"(v[0].z), "=r"(v[0].w), "=r"(v[1].x), "=r"(v[1].y),
        "=r"(v[1].z), "=r"(v[1].w)
      : "r"(taddr)
      : "memory");
}

// vector geometry of a row: `head` scalars up to the first 16-byte boundary,
// `nvec` 16-byte vectors, then `tail` scalars
template <typename T>
struct Geom {
  int head, tail;
  int64_t nvec, t0;
  __device__ Geom(const T* p, int64_t V) {
    constexpr int VEC = Storage<T>::kVec;
    const uintptr_t addr = (uintptr_t)p;
    int64_t h = (int64_t)(((16 - (addr & 15)) & 15) / sizeof(T));
    if (h > V) h = V;
    head = (int)h;
    nvec = (V - h) / VEC;
    t0 = h + nvec * VEC;
    tail = (int)(V - t0);
  }
};

// ln 2 as a float pair
constexpr float kLn2Hi = 0.693147182464599609375f;
constexpr float kLn2Lo = -1.904654323148236e-09f;

__device__ __forceinline__ FF ff_mul_ln2(FF a) {
  const float ph = __fmul_rn(a.hi, kLn2Hi);
  float pl = __fmaf_rn(a.hi, kLn2Hi, -ph);
  pl = __fmaf_rn(a.hi, kLn2Lo, pl);
  pl = __fmaf_rn(a.lo, kLn2Hi, pl);
  return fast_two_sum(ph, pl);
}

// log2 of a positive float pair: exact exponent + log2f of the mantissa in
// [1,2) (absolute error ~6e-8) + the first-order term of the low part.
__device__ __forceinline__ FF log2_ff(FF z) {
  int e;
  const float m = frexpf(z.hi, &e);  // z.hi = m 2^e, m in [0.5, 1)
  const float l = log2f(__fmul_rn(m, 2.0f));
  const float corr = __fmul_rn(__fdiv_rn(z.lo, z.hi), kLog2e);
  FF r = two_sum((float)(e - 1), l);
  r.lo = __fadd_rn(r.lo, corr);
  return fast_two_sum(r.hi, r.lo);
}

// k3 = e^d - d - 1 in fp32: a short series where e^d - 1 and d nearly
// cancel, expm1f elsewhere (em = expm1f(d)).
__device__ __forceinline__ float k3_from(float d, float em) {
  if (fabsf(d) < 0.0625f) {
    float q = __fmaf_rn(d, 1.0f / 720.0f, 1.0f / 120.0f);
    q = __fmaf_rn(d, q, 1.0f / 24.0f);
    q = __fmaf_rn(d, q, 1.0f / 6.0f);
    q = __fmaf_rn(d, q, 0.5f);
    return __fmul_rn(__fmul_rn(d, d), q);
  }
  return __fsub_rn(em, d);
}

// ------------------------------------------------------------- the combine
// Block combine of the per-thread normalisers of the policy (a) and reference
// (b) slices.  Every thread gets the maxima; warp 0 gets the two sums
// Z = sum_v 2^(x_v log2e - ML), ML = fl(M log2e), as float pairs.  Fixed
// order: xor-shuffle trees, warps in index order.  Contains __syncthreads().
__device__ __forceinline__ void combine_ff(const OnlineLse& a, const OnlineLse& b, float* fs,
                                           FF* zs, float& Ma, float& Mb, FF& Za, FF& Zb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  float ma = warp_max(a.m), mb = warp_max(b.m);
  if (lane == 0) { fs[warp] = ma; fs[32 + warp] = mb; }
  __syncthreads();
  ma = warp_max(lane < nw ? fs[lane] : -INFINITY);
  mb = warp_max(lane < nw ? fs[32 + lane] : -INFINITY);
  Ma = ma;
  Mb = mb;
  const float MLa = __fmul_rn(ma, kLog2e), MLb = __fmul_rn(mb, kLog2e);
  const float za = a.m == -INFINITY ? 0.f
                                    : __fmul_rn(__fsub_rn(a.s, a.c), ex2_fast(__fsub_rn(a.mL, MLa)));
  const float zb = b.m == -INFINITY ? 0.f
                                    : __fmul_rn(__fsub_rn(b.s, b.c), ex2_fast(__fsub_rn(b.mL, MLb)));
  const FF wa = warp_sum_ff(za), wb = warp_sum_ff(zb);
  if (lane == 0) { zs[warp] = wa; zs[32 + warp] = wb; }
  __syncthreads();
  if (warp == 0) {
    Za = warp_sum_ff2(lane < nw ? zs[lane] : FF{0.f, 0.f});
    Zb = warp_sum_ff2(lane < nw ? zs[32 + lane] : FF{0.f, 0.f});
  }
}

// --------------------------------------------------------- the fast finish
// One thread, fp32 and float-float.  Inputs: the policy / reference rows'
// logsumexp in base 2 as ML + log2(Z), the action logits xa / ya, the
// behaviour log-prob o, the advantage A and the token weight c.
__device__ __forceinline__ RowScalars finish_fast(const RowArgs& a, float MLp, FF Zp, float MLr,
                                                  FF Zr, float xa, float ya, float o, float A,
                                                  float c, bool want_grad) {
  RowScalars r;
  const FF Pp = ff_add(FF{MLp, 0.f}, log2_ff(Zp));  // logsumexp / ln2
  const FF Pr = ff_add(FF{MLr, 0.f}, log2_ff(Zr));
  const FF lse_p = ff_mul_ln2(Pp);
  const FF lp = ff_add(FF{xa, 0.f}, ff_neg(lse_p));            // log pi(a)
  const FF lpo = ff_add(two_sum(xa, -o), ff_neg(lse_p));       // log pi(a) - old
  const FF dl = ff_mul_ln2(ff_add(Pr, ff_neg(Pp)));            // lse_r - lse_p
  const float d = ff_float(ff_add(two_sum(ya, -xa), ff_neg(dl)));  // ref_logp - logp
  const float lpf = ff_float(lp);
  const float rm1 = expm1f(ff_float(lpo));  // r - 1
  const float emd = expm1f(d);
  const float emlp = expm1f(lpf);
  const float ratio = __fadd_rn(1.0f, rm1);
  const TokEpi<float> t = token_epilogue<float>(rm1, lpf, d, emd, k3_from(d, emd), true, A, a.var);
  const float gc = __fmul_rn(a.grad_scale, c);
  const float w = __fmul_rn(gc, t.g);
  r.lse_p = (double)lse_p.hi + (double)lse_p.lo;
  r.q = (double)t.q;
  r.k = (double)t.k;
  r.logp = (double)lp.hi + (double)lp.lo;
  r.w = (double)w;
  r.wneg = -w;
  r.LL = ff_float(Pp);
  r.ga = -__fmul_rn(w, emlp);
  r.precise = 0;
  r.clip = t.clip;
  r.dlr = (double)d;
  if (want_grad && a.precise_ok) {
    // sensitivities of w to the two rows' logsumexp: the KL part's slope
    // (both rows), the policy part's |A| r (policy row), w itself (p_a)
    const float s_ref = fabsf(gc) * a.beta * kl_slope(a.var.kl_type, emd);
    const float s_pol = fabsf(w) + fabsf(gc) * fabsf(A) * ratio + s_ref;
    r.precise = (s_pol * kFastErrBound > kTau ? 1 : 0) | (s_ref * kFastErrBound > kTau ? 2 : 0);
    // k1's value is d itself (and k2's gradient is d): an error in one row's
    // logsumexp enters the KL term at full weight and, summed over tokens of
    // either sign, is not damped; refining the policy row alone would leave
    // the reference row's rounding in d uncancelled, so both rows go together
    if ((r.precise & 1) && a.var.kl_type != GRPO_KL_K3) r.precise |= 2;
  }
  return r;
}

// ------------------------------------------------------ the precise finish
// Run by all 32 lanes of warp 0; the result is valid in lane 0.  The rows'
// logsumexp are base + log(z), in double; the transcendentals run on separate
// lanes (GB300's double rate is low, its latency high).
static __device__ __forceinline__ RowScalars finish_precise(const RowArgs& a, double base_p,
                                                            double z_p, double base_r, double z_r,
                                                            float xa, float ya, float o, double A,
                                                            double c) {
  const int lane = threadIdx.x & 31;
  xa = __shfl_sync(0xFFFFFFFFu, xa, 0);
  ya = __shfl_sync(0xFFFFFFFFu, ya, 0);
  o = __shfl_sync(0xFFFFFFFFu, o, 0);
  const double lz = log(lane == 1 ? z_r : z_p);
  const double lse_p = base_p + __shfl_sync(0xFFFFFFFFu, lz, 0);
  const double lse_r = base_r + __shfl_sync(0xFFFFFFFFu, lz, 1);
  const double lp = (double)xa - lse_p;
  const double lr = (double)ya - lse_r;
  const double d = lr - lp;
  const double arg = lane == 0 ? lp - (double)o : (lane == 1 ? d : lp);
  const double em = expm1(arg);
  const double rm1 = __shfl_sync(0xFFFFFFFFu, em, 0);
  const double emd = __shfl_sync(0xFFFFFFFFu, em, 1);
  const double emlp = __shfl_sync(0xFFFFFFFFu, em, 2);
  RowScalars r;
  const TokEpi<double> t = token_epilogue<double>(rm1, lp, d, emd, emd - d, true, A, a.var);
  const double w = (double)a.grad_scale * c * t.g;
  r.lse_p = lse_p;
  r.q = t.q;
  r.k = t.k;
  r.logp = lp;
  r.w = w;
  r.wneg = (float)(-w);
  r.LL = (float)(lse_p * (double)kLog2e);
  r.ga = (float)(-w * emlp);
  r.precise = 1;
  r.clip = t.clip;
  r.dlr = d;
  return r;
}

// ---------------------------------------------------------------- sweep 2
// -w softmax_v; in a refined row, elements above kElemPrecise in double
template <bool kPrecise>
__device__ __forceinline__ float grad_elem(float x, const RowScalars& rs) {
  const float p = ex2_fast(__fmaf_rn(x, kLog2e, -rs.LL));
  float g = __fmul_rn(rs.wneg, p);
  if (kPrecise && fabsf(g) > kElemPrecise) g = (float)(-rs.w * exp((double)x - rs.lse_p));
  return g;
}
// the element v of a row (the action element is w (1 - p_a))
template <bool kPrecise>
__device__ __forceinline__ float grad_at(float x, int64_t v, const RowScalars& rs, int64_t act) {
  return v == act ? rs.ga : grad_elem<kPrecise>(x, rs);
}

}  // namespace grpo
