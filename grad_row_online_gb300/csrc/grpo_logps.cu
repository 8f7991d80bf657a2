// grpo_logps.cu -- the GRPO loss from per-token log-probs (no vocabulary).
//
// grpo.cpp README, "CUDA": the selected-token GRPO loss over [tokens] log
// probs, reduced inside each block (never with per-token atomics); RL-Kernel
// "GRPO Loss" page, "Accuracy" for the per-token terms and "Tensor and Data
// Parallel" for the two nested reductions (token slots -> sequence totals ->
// scalar).
//
// One CTA per sequence evaluates each active token's policy and KL terms
// once, writes dL/dlogp for every slot (0 on masked ones) and forms the
// sequence's totals in a fixed order; the CTA that finishes last (an atomic
// ticket that nobody waits on) forms the scalar from the B totals in index
// order.  When every sequence's CTA fits on the GPU at once the kernel is one
// cooperative launch that also does the advantage / count pass: each CTA
// scans its own mask row and forms its own advantage, and the CTAs meet at a
// grid barrier for the batch counts N and S; otherwise (or on request) that
// pass runs first as its own kernel.  The whole cost is one pass over logps /
// old_logps / ref_logps / mask plus the gradient write.
//
// Arithmetic: fp32 per token, Kahan sums per thread, float pairs (two_sum)
// for every sum above that.  No fp64 on the common path: GB300's fp64 pipe
// is a small fraction of its fp32 rate, and a few dozen fp64 operations per
// CTA measurably lengthened this kernel.
#include <atomic>

#include "grpo_groups.cuh"

namespace grpo {

static constexpr int kLogpsThreads = 128;
static_assert(kLogpsThreads >= kFinalThreads, "the last CTA runs final_scalar");
static constexpr float kWPrecise = 0x1p-11f;

// e^d - 1 and k3 = e^d - d - 1 together.  With Q(d) = sum_{n>=2} d^(n-2)/n!,
// e^d - 1 = d + d^2 Q(d) and k3 = d^2 Q(d).
//
// Q_poly: Q through its d^7/9! term.  For |d| < 1/2 the first omitted term,
// d^8/10!, is below 2e-9 of Q, so Q_poly is Q to fp32 rounding.
__device__ __forceinline__ float Q_poly(float d) {
  float q = __fmaf_rn(d, 1.0f / 362880.0f, 1.0f / 40320.0f);
  q = __fmaf_rn(d, q, 1.0f / 5040.0f);
  q = __fmaf_rn(d, q, 1.0f / 720.0f);
  q = __fmaf_rn(d, q, 1.0f / 120.0f);
  q = __fmaf_rn(d, q, 1.0f / 24.0f);
  q = __fmaf_rn(d, q, 1.0f / 6.0f);
  return __fmaf_rn(d, q, 0.5f);
}

struct Em {
  float em;  // e^d - 1
  float k3;  // e^d - d - 1
};
// Any d: Q_poly inside |d| < 1/2, the library expm1f outside (where
// k3 = (e^d - 1) - d no longer cancels).
__device__ __forceinline__ Em expm1_k3(float d) {
  Em r;
  if (fabsf(d) < 0.5f) {
    const float q = Q_poly(d), d2 = __fmul_rn(d, d);
    r.k3 = __fmul_rn(d2, q);
    r.em = __fmaf_rn(d2, q, d);
  } else {
    r.em = expm1f(d);
    r.k3 = __fsub_rn(r.em, d);
  }
  return r;
}

// One token on the general path: the ratio and the KL argument through
// expm1_k3 (accurate near 0), then the variant's epilogue.  For the clipped
// surrogate p = -A - min((r-1)A, (clip(r)-1)A): the constant -A enters once
// per sequence, as -A_i L_i in float pairs from the float-pair advantage
// (with a full mask the A_i of a group cancel there, which an fp32 A rounded
// per token would break).
// (em_seq: GSPO's rho_i - 1 for the whole sequence, used in place of the
// token's own ratio when the call asks for sequence-level ratios.)
__device__ __forceinline__ TokEpi<float> tok_terms(float lp, float o, float rf, float A,
                                                   const LogpsArgs& a, float em_seq) {
  const float em = a.var.seq_ratio ? em_seq : expm1_k3(__fsub_rn(lp, o)).em;  // r - 1
  const float d = a.ref ? __fsub_rn(rf, lp) : 0.0f;
  const Em kd = expm1_k3(d);
  return token_epilogue<float>(em, lp, d, kd.em, kd.k3, a.ref != nullptr, A, a.var);
}

// dL/dlogp in double, for tokens whose gradient is large enough that the
// fp32 evaluation could be off by more than its rounding allowance.  Rare,
// so it also forms the token weight c itself.
struct SeqCtx {
  float A, gc;        // advantage and grad_scale * c, rounded to fp32
  double Ad;          // the advantage
  int64_t b;          // the sequence
  int L;              // its active tokens
  unsigned long long N, S;
  float em_seq;       // GSPO: rho_i - 1 (fp32 and double)
  double em_seq_d;
};
// The sequence's constants the precise path needs, in shared memory (set
// once per CTA before the token loop): the rare call then takes three
// floats, and neither a per-thread struct nor the kernel's arguments need an
// address (either would give the kernel a stack frame).
struct PreciseCtx {
  double A, em_seq;  // the advantage; GSPO: rho_i - 1
  unsigned long long N, S;
  int L, reduction;
  float norm_c, grad_scale;
  Variant var;
  bool has_ref;
};
__shared__ PreciseCtx g_pc;
__device__ __noinline__ float w_precise(float lp, float o, float rf) {
  const PreciseCtx& p = g_pc;
  // the token weight c: 1/max(N,1), 1/(max(S,1) L) or 1/C
  const double c = p.reduction == GRPO_TOKEN_MEAN ? 1.0 / (double)(p.N > 0 ? p.N : 1)
                   : p.reduction == GRPO_SEQUENCE_MEAN
                       ? 1.0 / ((double)(p.S > 0 ? p.S : 1) * (double)p.L)
                       : 1.0 / (double)p.norm_c;
  const double em = p.var.seq_ratio ? p.em_seq : expm1((double)lp - (double)o);
  const double d = p.has_ref ? (double)rf - (double)lp : 0.0;
  const double emd = expm1(d);
  const TokEpi<double> t =
      token_epilogue<double>(em, (double)lp, d, emd, emd - d, p.has_ref, p.A, p.var);
  return (float)((double)p.grad_scale * c * t.g);
}

__device__ __forceinline__ void kahan(float& s, float& c, float x) {
  const float y = __fsub_rn(x, c);
  const float t = __fadd_rn(s, y);
  c = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}
// Two Kahan sums side by side on packed fp32x2 (the policy and KL terms):
// the same IEEE operations as two calls of kahan(), a - b formed as
// fma(b, -1, a) (one rounding, as a subtraction).
__device__ __forceinline__ void kahan2(float2& s, float2& c, float2 x) {
  const float2 m1 = make_float2(-1.f, -1.f);
  const float2 y = __ffma2_rn(c, m1, x);
  const float2 t = __fadd2_rn(s, y);
  c = __ffma2_rn(y, m1, __ffma2_rn(s, m1, t));
  s = t;
}

__device__ __forceinline__ bool vec_ok(const LogpsArgs& a) {
  const uintptr_t m = (uintptr_t)a.logps | (uintptr_t)a.old | (uintptr_t)a.ref | (uintptr_t)a.grad;
  return (a.T % 4 == 0) && ((m & 15) == 0) && (((uintptr_t)a.mask & 3) == 0);
}

// Per-thread sums: q and k each as a Kahan pair.  A vector's four active
// tokens are added in fp32 first and enter the Kahan sum once.
struct Acc {
  float2 s = {0.f, 0.f}, c = {0.f, 0.f};  // Kahan sums of (q, k) and their compensations
  unsigned nc[3] = {0u, 0u, 0u};  // clipped tokens: upper, lower, dual
  // (constant indices only, so the counters stay in registers)
  __device__ __forceinline__ void count(int clip, unsigned n = 1u) {
    if (clip == 1) nc[0] += n;
    else if (clip == 2) nc[1] += n;
    else if (clip == 3) nc[2] += n;
  }
};

__device__ __forceinline__ float token_w(float lp, float o, float rf, const TokEpi<float>& t,
                                         const SeqCtx& x, const LogpsArgs& a) {
  float w = __fmul_rn(x.gc, t.g);
  if (fabsf(w) > kWPrecise) w = w_precise(lp, o, rf);
  return w;
}

// Per-CTA constants of the fast path.  With s = sign(A) (+1 for A = 0) and
// lim = eps_hi (A > 0) or eps_lo (A <= 0):
//   min(rA, clip(r)A) = A + |A| min(s(r-1), lim)    (so q = -|A| min(s em, lim))
//   the token is clipped  <=>  s em > lim
// which is the clipped-surrogate case split with the sign of A taken out.
struct FastCtx {
  bool on;     // the call's loss is the default variant (clipped surrogate, k3)
  int clip_kind;  // how a clipped token counts: 1 upper (A > 0), 2 lower (A < 0), 0 not
  float2 s2, neg_absA2, negA2, gc2, neg_beta2, beta2;
  float lim;
  float lo, hi;  // CISPO: the bounds on r - 1, -eps_lo and eps_hi
  float dlo;     // the dual clip's floor on s(r - 1): -(c - 1) when A < 0, else -inf
  float g2_max;  // (kWPrecise / gc)^2: a vector whose sum of g^2 stays below
                 // it has every |w| <= kWPrecise
};

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Q_poly on two lanes with packed fp32x2 arithmetic.
__device__ __forceinline__ float2 Q_poly2(float2 d) {
  float2 q = __ffma2_rn(d, f2(1.0f / 362880.0f), f2(1.0f / 40320.0f));
  q = __ffma2_rn(d, q, f2(1.0f / 5040.0f));
  q = __ffma2_rn(d, q, f2(1.0f / 720.0f));
  q = __ffma2_rn(d, q, f2(1.0f / 120.0f));
  q = __ffma2_rn(d, q, f2(1.0f / 24.0f));
  q = __ffma2_rn(d, q, f2(1.0f / 6.0f));
  return __ffma2_rn(d, q, f2(0.5f));
}

// Two active tokens on the fast path (every operation but the clip on
// packed fp32x2).  Accumulates q and k, and the sums behind the range check.
// kKL: the KL estimator, 0 k3 (the default; k = e^d - d - 1 from the
// polynomial, its gradient -(e^d - 1)), 1 k1 (k = -d, gradient 1), 2 k2
// (k = d^2 / 2, gradient -d); d = ref_logp - logp, and only k3 puts d under
// the polynomial's range check.  kDual: the dual clip on negative-advantage
// tokens, min(s(r-1), lim) held at or above dlo = -(c-1) (A < 0; -inf
// otherwise), so that q = -|A| max(min(s(r-1), lim), dlo), and the policy
// gradient is 0 where s(r-1) < dlo too (counted apart, in ndual).
template <bool kCount, int kKL, bool kDual>
__device__ __forceinline__ float2 pair_fast(float2 lp, float2 od, float2 rf, bool has_ref,
                                            const FastCtx& f, float2& vq, float2& vk,
                                            float2& d2sum, float2& g2sum, int& nclip,
                                            int& ndual) {
  const float2 dp = __ffma2_rn(od, f2(-1.f), lp);  // logp - old
  const float2 Qp = Q_poly2(dp), ddp = __fmul2_rn(dp, dp);
  const float2 em = __ffma2_rn(ddp, Qp, dp);       // r - 1
  const float2 dr = has_ref ? __ffma2_rn(lp, f2(-1.f), rf) : f2(0.f);  // ref - logp
  float2 k, ddr = f2(0.f), emr = f2(0.f);
  if (kKL == 0) {
    const float2 Qr = Q_poly2(dr);
    ddr = __fmul2_rn(dr, dr);
    k = __fmul2_rn(ddr, Qr);                       // k3
    emr = __ffma2_rn(ddr, Qr, dr);                 // e^(ref-logp) - 1
  } else if (kKL == 1) {
    k = __fmul2_rn(dr, f2(-1.f));                  // k1 = -d
  } else {
    k = __fmul2_rn(__fmul2_rn(dr, dr), f2(0.5f));  // k2 = d^2 / 2
  }
  const float2 se = __fmul2_rn(f.s2, em);
  float2 mn = make_float2(fminf(se.x, f.lim), fminf(se.y, f.lim));
  if (kDual) mn = make_float2(fmaxf(mn.x, f.dlo), fmaxf(mn.y, f.dlo));
  const float2 q = __fmul2_rn(f.neg_absA2, mn);
  float2 gp = __fmul2_rn(f.negA2, __fadd2_rn(em, f2(1.f)));  // -A r
  const bool cx = se.x > f.lim, cy = se.y > f.lim;
  const bool dx = kDual && se.x < f.dlo, dy = kDual && se.y < f.dlo;
  gp.x = (cx || dx) ? 0.f : gp.x;
  gp.y = (cy || dy) ? 0.f : gp.y;
  if (kCount) {
    nclip += (int)cx + (int)cy;
    if (kDual) ndual += (int)dx + (int)dy;
  }
  const float2 g = kKL == 0 ? __ffma2_rn(f.neg_beta2, emr, gp)
                 : kKL == 1 ? __fadd2_rn(gp, f.beta2)
                            : __ffma2_rn(f.neg_beta2, dr, gp);
  vq = __fadd2_rn(vq, q);
  vk = __fadd2_rn(vk, k);
  d2sum = __fadd2_rn(d2sum, kKL == 0 ? __fadd2_rn(ddp, ddr) : ddp);
  g2sum = __ffma2_rn(g, g, g2sum);
  return __fmul2_rn(f.gc2, g);
}

// CISPO with k3 on two active tokens (packed fp32x2 but for the clip): the
// weight clip(r) behind the stop-gradient gives p = -A clip(r) logp and the
// policy gradient -A clip(r); every token keeps it.
template <bool kCount>
__device__ __forceinline__ float2 pair_cispo(float2 lp, float2 od, float2 rf, bool has_ref,
                                             const FastCtx& f, float2& vq, float2& vk,
                                             float2& d2sum, float2& g2sum, int (&nclip)[2]) {
  const float2 dp = __ffma2_rn(od, f2(-1.f), lp);  // logp - old
  const float2 Qp = Q_poly2(dp), ddp = __fmul2_rn(dp, dp);
  const float2 em = __ffma2_rn(ddp, Qp, dp);       // r - 1
  const float2 dr = has_ref ? __ffma2_rn(lp, f2(-1.f), rf) : f2(0.f);  // ref - logp
  const float2 Qr = Q_poly2(dr), ddr = __fmul2_rn(dr, dr);
  const float2 k = __fmul2_rn(ddr, Qr);            // k3
  const float2 emr = __ffma2_rn(ddr, Qr, dr);      // e^(ref-logp) - 1
  const float2 emc = make_float2(fminf(fmaxf(em.x, f.lo), f.hi), fminf(fmaxf(em.y, f.lo), f.hi));
  const float2 gp = __fmul2_rn(f.negA2, __fadd2_rn(f2(1.f), emc));  // -A clip(r)
  const float2 q = __fmul2_rn(gp, lp);
  if (kCount) {
    nclip[0] += (int)(em.x > f.hi) + (int)(em.y > f.hi);
    nclip[1] += (int)(em.x < f.lo) + (int)(em.y < f.lo);
  }
  const float2 g = __ffma2_rn(f.neg_beta2, emr, gp);
  vq = __fadd2_rn(vq, q);
  vk = __fadd2_rn(vk, k);
  d2sum = __fadd2_rn(d2sum, __fadd2_rn(ddp, ddr));
  g2sum = __ffma2_rn(g, g, g2sum);
  return __fmul2_rn(f.gc2, g);
}
template <bool kCount>
__device__ __forceinline__ bool vec_cispo(const float4& l4, const float4& o4, const float4& r4,
                                          bool has_ref, const FastCtx& f, float4& w, float& vq,
                                          float& vk, int (&nclip)[2]) {
  float2 sq = f2(0.f), sk = f2(0.f), d2 = f2(0.f), g2 = f2(0.f);
  nclip[0] = nclip[1] = 0;
  const float2 w01 = pair_cispo<kCount>(make_float2(l4.x, l4.y), make_float2(o4.x, o4.y),
                                        make_float2(r4.x, r4.y), has_ref, f, sq, sk, d2, g2, nclip);
  const float2 w23 = pair_cispo<kCount>(make_float2(l4.z, l4.w), make_float2(o4.z, o4.w),
                                        make_float2(r4.z, r4.w), has_ref, f, sq, sk, d2, g2, nclip);
  w = make_float4(w01.x, w01.y, w23.x, w23.y);
  vq = __fadd_rn(sq.x, sq.y);
  vk = __fadd_rn(sk.x, sk.y);
  return __fadd_rn(d2.x, d2.y) < 0.25f && __fadd_rn(g2.x, g2.y) <= f.g2_max;
}

// One vector of four active slots on the fast path.  Returns false when a
// token needs the general path: a log ratio outside |d| < 1/2 (caught by
// the vector's sum of d^2 reaching 1/4), or a gradient above kWPrecise
// (caught by its sum of g^2); NaNs fail the check too.
template <bool kCount, int kKL, bool kDual>
__device__ __forceinline__ bool vec_fast(const float4& l4, const float4& o4, const float4& r4,
                                         bool has_ref, const FastCtx& f, float4& w,
                                         float& vq, float& vk, int& nclip, int& ndual) {
  float2 sq = f2(0.f), sk = f2(0.f), d2 = f2(0.f), g2 = f2(0.f);
  nclip = 0;
  ndual = 0;
  const float2 w01 = pair_fast<kCount, kKL, kDual>(
      make_float2(l4.x, l4.y), make_float2(o4.x, o4.y), make_float2(r4.x, r4.y), has_ref, f, sq,
      sk, d2, g2, nclip, ndual);
  const float2 w23 = pair_fast<kCount, kKL, kDual>(
      make_float2(l4.z, l4.w), make_float2(o4.z, o4.w), make_float2(r4.z, r4.w), has_ref, f, sq,
      sk, d2, g2, nclip, ndual);
  w = make_float4(w01.x, w01.y, w23.x, w23.y);
  vq = __fadd_rn(sq.x, sq.y);
  vk = __fadd_rn(sk.x, sk.y);
  return __fadd_rn(d2.x, d2.y) < 0.25f && __fadd_rn(g2.x, g2.y) <= f.g2_max;
}

// One vector of four active slots on the fast path for the other loss
// variants (k1 / k2 KL, the dual clip, CISPO, GSPO's sequence ratio): the
// same packed polynomials give e^(logp - old) - 1 (GSPO: the sequence's
// rho - 1 instead), e^d - 1 and k3, then each token takes the variant's
// epilogue in fp32, unrolled.  Same range checks as vec_fast (|d| < 1/2 for
// every argument taken from the polynomial, every |w| <= kWPrecise); the
// clip counts are returned, to be added only when the vector passes.
__device__ __forceinline__ bool vec_fast_variant(const float4& l4, const float4& o4,
                                                 const float4& r4, bool has_ref,
                                                 const SeqCtx& x, const LogpsArgs& a,
                                                 float4& w, float& vq, float& vk,
                                                 unsigned (&nc)[3]) {
  const float lp[4] = {l4.x, l4.y, l4.z, l4.w};
  float em[4], d[4], emd[4], k3[4];
  float2 d2 = f2(0.f);
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const float2 l2 = p ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
    float2 e2 = f2(x.em_seq);
    if (!a.var.seq_ratio) {
      const float2 o2 = p ? make_float2(o4.z, o4.w) : make_float2(o4.x, o4.y);
      const float2 dp = __ffma2_rn(o2, f2(-1.f), l2);  // logp - old
      const float2 Qp = Q_poly2(dp), ddp = __fmul2_rn(dp, dp);
      e2 = __ffma2_rn(ddp, Qp, dp);
      d2 = __fadd2_rn(d2, ddp);
    }
    float2 dr = f2(0.f), k2 = f2(0.f), er = f2(0.f);
    if (has_ref) {
      const float2 r2 = p ? make_float2(r4.z, r4.w) : make_float2(r4.x, r4.y);
      dr = __ffma2_rn(l2, f2(-1.f), r2);  // ref - logp
      const float2 Qr = Q_poly2(dr), ddr = __fmul2_rn(dr, dr);
      k2 = __fmul2_rn(ddr, Qr);
      er = __ffma2_rn(ddr, Qr, dr);
      d2 = __fadd2_rn(d2, ddr);
    }
    em[2 * p] = e2.x;
    em[2 * p + 1] = e2.y;
    d[2 * p] = dr.x;
    d[2 * p + 1] = dr.y;
    emd[2 * p] = er.x;
    emd[2 * p + 1] = er.y;
    k3[2 * p] = k2.x;
    k3[2 * p + 1] = k2.y;
  }
  vq = 0.f;
  vk = 0.f;
  nc[0] = nc[1] = nc[2] = 0u;
  bool small = true;
  float wj[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const TokEpi<float> t = token_epilogue<float>(em[j], lp[j], d[j], emd[j], k3[j], has_ref,
                                                  x.A, a.var);
    vq = __fadd_rn(vq, t.q);
    vk = __fadd_rn(vk, t.k);
    nc[0] += t.clip == 1;
    nc[1] += t.clip == 2;
    nc[2] += t.clip == 3;
    wj[j] = __fmul_rn(x.gc, t.g);
    small = small && fabsf(wj[j]) <= kWPrecise;
  }
  w = make_float4(wj[0], wj[1], wj[2], wj[3]);
  return __fadd_rn(d2.x, d2.y) < 0.25f && small;
}

enum : int { kModeDefault = 0, kModeVariant = 1, kModeGspo = 2, kModeK1 = 3, kModeK2 = 4,
             kModeCispo = 5, kModeDual = 6 };
// The clipped surrogate without the dual clip or sequence ratios, with the KL
// estimator of the mode: the packed fast path of vec_fast.
__host__ __device__ constexpr int mode_kl(int mode) {
  return mode == kModeK1 ? 1 : (mode == kModeK2 ? 2 : 0);
}
__host__ __device__ constexpr bool mode_packed(int mode) {
  return mode == kModeDefault || mode == kModeK1 || mode == kModeK2 || mode == kModeDual;
}
// Modes whose general-path vectors wait for the end of the token loop.
__host__ __device__ constexpr bool mode_defers(int mode) { return mode != kModeVariant; }

// GSPO with the clipped surrogate and k3: every token of the sequence shares
// the ratio rho_i, so its policy term q, policy gradient and clip are the
// sequence's constants (token_epilogue at r - 1 = rho_i - 1, once per CTA);
// per token only the KL term and its gradient remain: k3 and e^d - 1 from
// the packed polynomial, g = g_pol - beta (e^d - 1).
struct GspoCtx {
  bool on;
  float q;        // the policy term of every token
  int clip;       // its clip (counted per token, as the general path does)
  float2 gpol2, neg_beta2, gc2;
};
__device__ __forceinline__ bool vec_fast_gspo(const float4& l4, const float4& r4, bool has_ref,
                                              const GspoCtx& gs, float4& w, float& vq,
                                              float& vk) {
  float2 d2 = f2(0.f);
  float k[4];
  float2 wv[2];
  bool small = true;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const float2 l2 = p ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
    const float2 r2 = p ? make_float2(r4.z, r4.w) : make_float2(r4.x, r4.y);
    const float2 dr = has_ref ? __ffma2_rn(l2, f2(-1.f), r2) : f2(0.f);  // ref - logp
    const float2 Qr = Q_poly2(dr), ddr = __fmul2_rn(dr, dr);
    const float2 kk = __fmul2_rn(ddr, Qr);        // k3
    const float2 emr = __ffma2_rn(ddr, Qr, dr);   // e^(ref-logp) - 1
    d2 = __fadd2_rn(d2, ddr);
    wv[p] = __fmul2_rn(gs.gc2, __ffma2_rn(gs.neg_beta2, emr, gs.gpol2));
    small = small && fabsf(wv[p].x) <= kWPrecise && fabsf(wv[p].y) <= kWPrecise;
    k[2 * p] = kk.x;
    k[2 * p + 1] = kk.y;
  }
  w = make_float4(wv[0].x, wv[0].y, wv[1].x, wv[1].y);
  // the four tokens' terms added in token order, as the general path adds them
  vq = __fadd_rn(__fadd_rn(__fadd_rn(gs.q, gs.q), gs.q), gs.q);
  vk = __fadd_rn(__fadd_rn(__fadd_rn(k[0], k[1]), k[2]), k[3]);
  return __fadd_rn(d2.x, d2.y) < 0.25f && small;
}

// Every byte of a mask word nonzero.
__device__ __forceinline__ bool all_active(uint32_t mw) {
  return ((((mw & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | mw) & 0x80808080u) == 0x80808080u;
}

// The same vector on the general path, token by token.
__device__ __forceinline__ void vec_general(uint32_t mw, const float4& l4, const float4& o4,
                                            const float4& r4, const SeqCtx& x,
                                            const LogpsArgs& a, float4& w, float& vq,
                                            float& vk, Acc& acc) {
  // the token loop is kept rolled (code size); its operands and results are
  // picked by selects on the loop counter, so nothing goes to local memory
  float w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;
  vq = 0.f;
  vk = 0.f;
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    if ((mw >> (8 * j)) & 0xFFu) {
      const float lp = j == 0 ? l4.x : j == 1 ? l4.y : j == 2 ? l4.z : l4.w;
      const float od = j == 0 ? o4.x : j == 1 ? o4.y : j == 2 ? o4.z : o4.w;
      const float rf = j == 0 ? r4.x : j == 1 ? r4.y : j == 2 ? r4.z : r4.w;
      const TokEpi<float> t = tok_terms(lp, od, rf, x.A, a, x.em_seq);
      vq = __fadd_rn(vq, t.q);
      vk = __fadd_rn(vk, t.k);
      acc.count(t.clip);
      const float wj = token_w(lp, od, rf, t, x, a);
      w0 = j == 0 ? wj : w0;
      w1 = j == 1 ? wj : w1;
      w2 = j == 2 ? wj : w2;
      w3 = j == 3 ? wj : w3;
    }
  }
  w = make_float4(w0, w1, w2, w3);
}

// One vector of four slots in the token loop: its gradient, and its q / k
// sums into the thread's Kahan pairs.  Fully active vectors take a fast path
// when its range check passes; fully masked ones give zeros.  Any other
// vector: an instantiation with a packed path of its own (every mode but
// kModeVariant) returns false, and the thread records it and evaluates it on
// the general path after the loop (deferred_list), so that loop holds no
// general-path code, call or double arithmetic; the shared variants'
// instantiation (whose loop measured faster with it) takes the general path
// in place.
template <int kMode, bool kCount>
__device__ __forceinline__ bool process_vec(uint32_t mw, const float4& l, const float4& o,
                                            const float4& r, bool has_ref, const FastCtx& f,
                                            const GspoCtx& gs, const SeqCtx& x,
                                            const LogpsArgs& a, Acc& acc, float4& w) {
  w = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mw == 0u) return true;
  float vq, vk;
  int nclip, ndual;
  int ncl2[2];
  unsigned nc[3];
  if (mode_packed(kMode) && all_active(mw) &&
      vec_fast<kCount, mode_kl(kMode), kMode == kModeDual>(l, o, r, has_ref, f, w, vq, vk, nclip,
                                                           ndual)) {
    if (kCount) {
      acc.count(f.clip_kind, (unsigned)nclip);
      if (kMode == kModeDual) acc.nc[2] += (unsigned)ndual;
    }
  } else if (kMode == kModeGspo && all_active(mw) && vec_fast_gspo(l, r, has_ref, gs, w, vq, vk)) {
    if (gs.clip) acc.count(gs.clip, 4u);
  } else if (kMode == kModeCispo && all_active(mw) &&
             vec_cispo<kCount>(l, o, r, has_ref, f, w, vq, vk, ncl2)) {
    if (kCount) {
      acc.nc[0] += (unsigned)ncl2[0];
      acc.nc[1] += (unsigned)ncl2[1];
    }
  } else if (kMode == kModeVariant && all_active(mw) &&
             vec_fast_variant(l, o, r, has_ref, x, a, w, vq, vk, nc)) {
    acc.nc[0] += nc[0];
    acc.nc[1] += nc[1];
    acc.nc[2] += nc[2];
  } else if (mode_defers(kMode)) {
    return false;
  } else {
    vec_general(mw, l, o, r, x, a, w, vq, vk, acc);
  }
  kahan2(acc.s, acc.c, make_float2(vq, vk));
  return true;
}

// The vectors a thread leaves to the general path, in the order it met them:
// entry k of thread t at list[t * m + k], m = ceil(vectors of the row / 128)
// (the most any thread meets), in the workspace's token-slot area of the
// sequence (16 bytes per slot; at most T / 4 + 127 entries are used, below
// its 4 T words).  Each thread reads back only its own entries.
// (Only the count lives in a register through the loop; the address is
// formed from the kernel's arguments when a vector is recorded.)
__device__ __forceinline__ uint32_t* deferred_list(const LogpsArgs& a, int64_t b) {
  const int64_t m = (a.T / 4 + kLogpsThreads - 1) / kLogpsThreads;
  return a.defer + b * 4 * a.T + (int64_t)threadIdx.x * m;
}

// ---- staging through shared memory with bulk asynchronous copies ----
// A sequence's row is cut into chunks of kChunk tokens from slot 0; the
// chunks that hold its active tokens move through shared memory (logps,
// old, ref and the mask bytes: four cp.async.bulk copies completing on one
// mbarrier), kDepth of them in flight while one is evaluated.  (Requesting
// chunks before the mask scan, or prefetching the whole active range into
// L2 once it is known, measured slower: the flood of requests delays the
// mask scan and the grid barrier behind it.)
static constexpr int kChunkVecs = 2;  // float4 vectors per thread per chunk
static constexpr int kChunk = 4 * kLogpsThreads * kChunkVecs;
static constexpr int kDepth = 2;
static constexpr unsigned long long kWaitNs = 200000000ull;  // 0.2 s per bounded wait
static constexpr uint32_t kWaitRounds = 1u << 26;  // and never more try_wait rounds than this

struct Stage {
  float4 lp[kChunk / 4];
  float4 od[kChunk / 4];
  float4 rf[kChunk / 4];
  uint32_t mk[kChunk / 4];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for a phase of `bar`: false if it did not complete within
// kWaitNs (read from the global timer every 16 rounds) or kWaitRounds rounds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < kWaitRounds; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

// Staging applies when every copy is 16-byte aligned: float rows on 16-byte
// boundaries with T % 16 == 0 puts each 16-token chunk start on a 64-byte
// (data) and 16-byte (mask) boundary.
__device__ __forceinline__ bool staged_ok(const LogpsArgs& a) {
  const uintptr_t m = (uintptr_t)a.logps | (uintptr_t)a.old | (uintptr_t)a.ref |
                      (uintptr_t)a.grad | (uintptr_t)a.mask;
  return (a.fused || a.range != nullptr) && (a.T % 16 == 0) && ((m & 15) == 0);
}

// The grid barrier of the one-launch form (a cooperative launch: every CTA
// that holds a sequence is resident).  A CTA arrives with one relaxed 64-bit
// add of (1 << 52) + ([L > 0] << 41) + L to the header's word: the word is
// the barrier and the batch counts at once, so no other data crosses CTAs
// and no memory fence is needed (under a saturated memory system a fence
// costs microseconds).  B <= 4095 CTAs, S <= B < 2^11 and N <= B T < 2^41
// fit their fields.  The wait polls the word, bounded like the copy waits
// (false if it ran out).
static constexpr int kArriveShift = 52, kLiveShift = 41;
__device__ __forceinline__ void grid_arrive(unsigned long long* c, int L) {
  const unsigned long long v =
      (1ull << kArriveShift) + ((unsigned long long)(L > 0) << kLiveShift) + (unsigned long long)L;
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(c), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool grid_wait(const unsigned long long* c, unsigned expected,
                                          unsigned long long& word) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < kWaitRounds; ++i) {
    word = ld_relaxed(c);
    if ((unsigned)(word >> kArriveShift) >= expected) return true;
    __nanosleep(100);  // fewer polls of the one word every CTA adds to
    if ((i & 15u) == 15u && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

// kMode: the call's loss is the default variant (clipped surrogate, k3:
// kModeDefault), the clipped surrogate with k1 or k2 (kModeK1, kModeK2: the
// same packed path with the other KL term), the clipped surrogate with the
// dual clip and k3 (kModeDual), CISPO with k3 (kModeCispo), GSPO
// with the clipped surrogate and k3 (kModeGspo), or any other variant
// (kModeVariant); kCount: the call wants the clip counters.
// Each form is its own instantiation, so that another's fast path does not
// cost it registers or instructions.
template <int kMode, bool kCount>
__global__ void __launch_bounds__(kLogpsThreads, 7) logps_kernel(const LogpsArgs a) {
  __shared__ FF s_ff[2][kLogpsThreads / 32];
  __shared__ unsigned s_nc[3][kLogpsThreads / 32];
  __shared__ FinalSmem s_fin;
  __shared__ double s_em[1];
  __shared__ bool s_last;
  __shared__ __align__(16) Stage s_st[kDepth];
  __shared__ __align__(8) uint64_t s_full[kDepth];
  __shared__ int s_scan[3][kLogpsThreads / 32];
  __shared__ double s_adv;
  __shared__ float2 s_aff;
  __shared__ int s_L;
  __shared__ int2 s_rg;
  __shared__ unsigned long long s_NS[2];
  const int64_t b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first();  // every input byte is read once
  const int64_t base = b * a.T;
  const bool has_ref = a.ref != nullptr;
  const bool staged = staged_ok(a);
  const uint32_t nref = has_ref ? 1u : 0u;
  // GSPO's tokens use the sequence's ratio, so the token loop needs no
  // behaviour log-probs (its pre-pass reads them); its stages skip them
  const uint32_t nold = a.var.seq_ratio ? 0u : 1u;
  // the test hook GRPO_FLAG_TEST_STALLED_COPY: the first copy of sequence 0
  // expects 16 bytes more than it delivers, so its wait runs out
  const uint32_t stall = ((a.flags & GRPO_FLAG_TEST_STALLED_COPY) && b == 0) ? 16u : 0u;
  // the staged path's active range ends at slot hi16 (the last active slot + 1,
  // rounded up to 16 slots)
  int hi16 = 0;  // slots within a sequence are 32-bit (T <= 2^30)
  // chunk c of the row, up to hi16, into the stage of the k-th chunk taken
  // (one thread)
  auto issue = [&](int c, int k) {
    const int64_t st = (int64_t)c * kChunk;
    const uint32_t len = (uint32_t)min((int64_t)kChunk, (int64_t)hi16 - st);
    Stage& S = s_st[k % kDepth];
    uint64_t* bar = &s_full[k % kDepth];
    mbar_expect_tx(bar, len * (4u * (1u + nold + nref) + 1u) + (k == 0 ? stall : 0u));
    bulk_g2s(S.lp, a.logps + base + st, 4u * len, bar, pol);
    if (nold) bulk_g2s(S.od, a.old + base + st, 4u * len, bar, pol);
    if (has_ref) bulk_g2s(S.rf, a.ref + base + st, 4u * len, bar, pol);
    bulk_g2s(S.mk, a.mask + base + st, len, bar, pol);
  };
  if (threadIdx.x == 0) {
    for (int d = 0; d < kDepth; ++d) mbar_init(&s_full[d], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // launched as a programmatic dependent of prep: everything above overlaps
  // prep's tail; prep's outputs (counts, advantages, ranges) are read below
  // (in the one-launch form there is no prep and this returns at once)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (b < a.B) {
    SeqCtx x;
    x.b = b;
    // The staged path takes the chunks [c_lo, c_hi) that hold active tokens
    // (the last one only up to hi16), the k-th of them (chunk c_lo + k) in
    // stage k % kDepth; the gradient slots outside [c_lo kChunk, hi16) are
    // zero-stored.
    int c_lo = 0, c_hi = 0, nlive = 0;
    auto geometry = [&](int2 rg) {
      c_lo = rg.y > rg.x ? rg.x / kChunk : 0;
      c_hi = rg.y > rg.x ? (rg.y + kChunk - 1) / kChunk : 0;
      hi16 = rg.y > rg.x ? (int)min((int64_t)((rg.y + 15) & ~15), a.T) : 0;
      if (!staged) c_lo = c_hi = 0, hi16 = 0;
      nlive = c_hi - c_lo;
    };
    auto first_copies = [&]() {  // one thread
      for (int k = 0; k < nlive && k < kDepth; ++k) issue(c_lo + k, k);
    };
    // slots outside the evaluated chunks hold no active token
    float4* grow = reinterpret_cast<float4*>(a.grad + base);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    auto zero_outside = [&](int t, int nt) {
      if (!staged || !a.grad) return;
      const int64_t v_lo = (int64_t)c_lo * (kChunk / 4);
      const int64_t v_hi = hi16 / 4;
      for (int64_t v = t; v < v_lo; v += nt) grow[v] = z4;
      for (int64_t v = v_hi + t; v < a.T / 4; v += nt) grow[v] = z4;
    };
    if (a.fused) {
      // warp 0 forms this sequence's advantage from its group while warps 1-3
      // scan the mask row, arrive at the grid barrier with the counts,
      // request the first chunks and zero the slots outside the evaluated
      // chunks
      if (warp == 0) {
        const int64_t gb = a.seq_begin + b;
        const int64_t g = a.bounds ? warp_find_group(a.bounds, a.G, gb, lane) : gb / a.spp;
        int64_t glo, ghi;
        group_bounds(a.bounds, a.spp, a.G, a.Bg, g, glo, ghi);
        const GroupStats gs = warp_group_stats(a.rewards, glo, ghi, a.adv_eps, a.eps_add, lane);
        if (lane == 0) {
          const double Ai = group_adv(gs, __ldg(a.rewards + gb));
          const float hi32 = (float)Ai;
          s_adv = Ai;
          s_aff = make_float2(hi32, (float)(Ai - (double)hi32));
          if (a.adv_out) a.adv_out[b] = hi32;
        }
      } else {
        // warp 1 + p scans piece p of three (a multiple of 16 slots each);
        // the integer counts combine exactly, each warp forming the same
        // range from the three records
        constexpr int kScanWarps = kLogpsThreads / 32 - 1;
        const int p = warp - 1;
        const int64_t q = (a.T + 16 * kScanWarps - 1) / (16 * kScanWarps) * 16;
        const int64_t t0 = min((int64_t)p * q, a.T), t1 = min(t0 + q, a.T);
        const SeqScan sc = warp_scan(a.mask + base + t0, t1 - t0, lane);
        if (lane == 0) {
          s_scan[0][p] = sc.count;
          s_scan[1][p] = sc.count ? (int)t0 + sc.first : 0x7FFFFFFF;
          s_scan[2][p] = sc.count ? (int)t0 + sc.last : -1;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kScanWarps) : "memory");
        int L = 0, first = 0x7FFFFFFF, last = -1;
#pragma unroll
        for (int k = 0; k < kScanWarps; ++k) {
          L += s_scan[0][k];
          first = min(first, s_scan[1][k]);
          last = max(last, s_scan[2][k]);
        }
        const int2 rg = L > 0 ? make_int2(first, last + 1) : make_int2(0, 0);
        geometry(rg);
        if (threadIdx.x == 32) {
          s_L = L;
          s_rg = rg;
          if (!a.shard) grid_arrive(&a.hdr->arrive, L);  // a shard call is given the batch's counts
        }
        if (threadIdx.x == 64 && staged) first_copies();
        zero_outside((int)threadIdx.x - 32, kLogpsThreads - 32);
        if (warp == kScanWarps) {
          // every group is checked once over the grid, as the separate pass
          // does: its boundaries, and its rewards for non-finite values
          for (int64_t g = blockIdx.x; g < a.G; g += gridDim.x) {
            int64_t glo, ghi;
            const bool ok = group_bounds(a.bounds, a.spp, a.G, a.Bg, g, glo, ghi);
            int nf = 0;
            for (int64_t i = glo + lane; i < ghi; i += 32) nf += !isfinite(__ldg(a.rewards + i));
            nf = warp_sum(nf);
            if (lane == 0 && !ok) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_CSR);
            if (lane == 0 && nf) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_NONFINITE_REWARD);
          }
        }
      }
      __syncthreads();
      x.L = s_L;
      if (warp == 0) geometry(s_rg);
    } else {
      x.L = a.L[b];
      geometry(a.range ? a.range[b] : make_int2(0, (int)a.T));
      if (staged && threadIdx.x == 0) first_copies();
      zero_outside((int)threadIdx.x, kLogpsThreads);
    }

    x.em_seq = 0.f;
    x.em_seq_d = 0.0;
    if (a.var.seq_ratio) {
      // GSPO: rho_i = exp(mean over the active tokens of logp - old), before
      // any token's term (Kahan sums per thread, float pairs across the CTA)
      float ss = 0.f, sc = 0.f;
      if (vec_ok(a)) {
        // 4-slot vectors of the evaluated chunks (the whole row off the
        // staged path), four per thread in flight, read whole (masked slots
        // are loaded but never used); each thread adds its vectors in order
        const uint32_t* mrow = reinterpret_cast<const uint32_t*>(a.mask + base);
        const float4* lrow = reinterpret_cast<const float4*>(a.logps + base);
        const float4* orow = reinterpret_cast<const float4*>(a.old + base);
        auto add4 = [&](uint32_t mw, const float4& l, const float4& o) {
          const float d[4] = {__fsub_rn(l.x, o.x), __fsub_rn(l.y, o.y), __fsub_rn(l.z, o.z),
                              __fsub_rn(l.w, o.w)};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((mw >> (8 * j)) & 0xFFu) kahan(ss, sc, d[j]);
        };
        const int64_t v1 = staged ? hi16 / 4 : a.T / 4;
        int64_t v = (staged ? (int64_t)c_lo * (kChunk / 4) : 0) + threadIdx.x;
        constexpr int kPre = 4;  // vectors per thread in flight
        for (; v < v1; v += kPre * kLogpsThreads) {
          uint32_t m[kPre];
          float4 l[kPre], o[kPre];
#pragma unroll
          for (int u = 0; u < kPre; ++u) {
            const int64_t vu = v + u * kLogpsThreads;
            m[u] = vu < v1 ? __ldg(mrow + vu) : 0u;
            l[u] = vu < v1 ? __ldg(lrow + vu) : make_float4(0.f, 0.f, 0.f, 0.f);
            o[u] = vu < v1 ? __ldg(orow + vu) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kPre; ++u) add4(m[u], l[u], o[u]);
        }
      } else {
        for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x)
          if (a.mask[base + t]) kahan(ss, sc, __fsub_rn(a.logps[base + t], a.old[base + t]));
      }
      const FF wsum = warp_sum_ff2(FF{ss, -sc});
      if (lane == 0) s_ff[0][warp] = wsum;
      __syncthreads();
      if (threadIdx.x == 0) {
        FF tot = s_ff[0][0];
        for (int k = 1; k < kLogpsThreads / 32; ++k) tot = ff_add(tot, s_ff[0][k]);
        const double em = x.L > 0 ? expm1(((double)tot.hi + (double)tot.lo) / (double)x.L) : 0.0;
        s_em[0] = em;
      }
      __syncthreads();
      x.em_seq_d = s_em[0];
      x.em_seq = (float)x.em_seq_d;
    }

    // the batch counts: complete once every CTA has arrived (the test hook
    // GRPO_FLAG_TEST_STALLED_BARRIER makes CTA 0 wait for one arrival more
    // than there are, so its wait runs out)
    if (threadIdx.x == 0) {
      if (a.fused && !a.shard) {
        const unsigned extra = ((a.flags & GRPO_FLAG_TEST_STALLED_BARRIER) && b == 0) ? 1u : 0u;
        unsigned long long word = 0ull;
        if (!grid_wait(&a.hdr->arrive, (unsigned)a.B + extra, word))
          atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_TIMEOUT);
        s_NS[0] = word & ((1ull << kLiveShift) - 1ull);
        s_NS[1] = (word >> kLiveShift) & ((1ull << (kArriveShift - kLiveShift)) - 1ull);
      } else if (a.fused) {
        s_NS[0] = a.NS[0];
        s_NS[1] = a.NS[1];
      } else {
        s_NS[0] = a.NS[0];
        s_NS[1] = a.NS[1];
        s_adv = a.A[b];
        s_aff = a.Aff[b];
      }
      g_pc = PreciseCtx{s_adv, x.em_seq_d, s_NS[0], s_NS[1], x.L, a.reduction, a.norm_c,
                        a.grad_scale, a.var, has_ref};
    }
    __syncthreads();
    x.N = s_NS[0];
    x.S = s_NS[1];
    x.Ad = s_adv;
    const float2 Ab = s_aff;
    x.A = Ab.x;
    // grad_scale * c in fp32: c = 1/max(N,1), 1/(max(S,1) L_b) or 1/C; the
    // products and quotient are rounded in fp32, well inside the gradient's
    // rounding allowance
    const float den =
        a.reduction == GRPO_TOKEN_MEAN      ? __ull2float_rn(x.N > 0 ? x.N : 1)
        : a.reduction == GRPO_SEQUENCE_MEAN ? __fmul_rn(__ull2float_rn(x.S > 0 ? x.S : 1), (float)x.L)
                                            : a.norm_c;
    x.gc = x.L > 0 ? __fdiv_rn(a.grad_scale, den) : 0.f;
    FastCtx f;
    f.on = mode_packed(kMode);
    f.clip_kind = x.A > 0.f ? 1 : (x.A < 0.f ? 2 : 0);
    const float sgn = x.A > 0.f ? 1.f : -1.f;
    f.s2 = f2(sgn);
    f.neg_absA2 = f2(-fabsf(x.A));
    f.negA2 = f2(-x.A);
    f.gc2 = f2(x.gc);
    f.neg_beta2 = f2(-a.beta);
    f.beta2 = f2(a.beta);
    f.lim = x.A > 0.f ? a.eps_hi : a.eps_lo;
    f.lo = -a.eps_lo;
    f.hi = a.eps_hi;
    f.dlo = a.var.dual_c > 0.f && x.A < 0.f ? -__fsub_rn(a.var.dual_c, 1.f) : -INFINITY;
    {
      const float gm = x.gc > 0.f ? __fdiv_rn(kWPrecise, x.gc) : INFINITY;
      f.g2_max = __fmul_rn(gm, gm);
    }
    GspoCtx gs;
    gs.on = kMode == kModeGspo;
    {
      // the policy part at the sequence's ratio (no KL part: has_ref false)
      const TokEpi<float> t0 = token_epilogue<float>(x.em_seq, 0.f, 0.f, 0.f, 0.f, false, x.A,
                                                     a.var);
      gs.q = t0.q;
      gs.clip = t0.clip;
      gs.gpol2 = f2(t0.g);
      gs.neg_beta2 = f2(-a.beta);
      gs.gc2 = f2(x.gc);
    }
    Acc acc;
    int n_def = 0;  // vectors this thread left to the general path
    if (staged) {
      // A wait that runs out (never expected outside the test hook) is
      // recorded; the CTA then issues no further copy, still waits for the
      // copies already issued (bounded), and skips the arithmetic -- the loss
      // outputs become NaN through the status word.
      // One CTA-wide barrier per chunk: past it, every thread is done with
      // the (k-1)-th chunk, whose stage is then refilled with the
      // (k-1+kDepth)-th.  Every thread counts the chunks requested so far (the
      // decisions are the same everywhere: `stalled` is taken CTA-wide).
      bool stalled = false;
      int issued = nlive < kDepth ? nlive : kDepth;
      for (int k = 0; k < issued; ++k) {
        const int slot = k % kDepth;
        const int64_t st = (int64_t)(c_lo + k) * kChunk;
        const int len = min(kChunk, hi16 - (c_lo + k) * kChunk);
        // warp 0 waits for the copies (the other warps sleep in the CTA
        // barrier, leaving the issue slots to the warps still computing)
        const bool ready = warp != 0 || mbar_wait(&s_full[slot], (uint32_t)(k / kDepth) & 1u);
        stalled = __syncthreads_or(!ready) || stalled;  // one decision for the CTA
        if (!stalled && k >= 1 && k - 1 + kDepth < nlive) {
          if (threadIdx.x == 0) issue(c_lo + k - 1 + kDepth, k - 1 + kDepth);
          issued = k + kDepth;
        }
        if (!stalled) {
          const Stage& S = s_st[slot];
#pragma unroll
          for (int u = 0; u < kChunkVecs; ++u) {
            const int v = threadIdx.x + u * kLogpsThreads;
            if (4 * v < len) {
              float4 w;
              if (process_vec<kMode, kCount>(S.mk[v], S.lp[v], S.od[v],
                                                has_ref ? S.rf[v] : z4, has_ref, f, gs, x, a,
                                                acc, w)) {
                if (a.grad) grow[st / 4 + v] = w;
              } else {
                deferred_list(a, b)[n_def++] = (uint32_t)(st / 4 + v);
              }
            }
          }
        }
      }
      if (stalled && threadIdx.x == 0) atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_TIMEOUT);
    } else if (vec_ok(a)) {
      const int64_t nv = a.T / 4;
      const uint32_t* mrow = reinterpret_cast<const uint32_t*>(a.mask + base);
      const float4* lrow = reinterpret_cast<const float4*>(a.logps + base);
      const float4* orow = reinterpret_cast<const float4*>(a.old + base);
      const float4* rrow = reinterpret_cast<const float4*>(a.ref + base);
      float4* grow = reinterpret_cast<float4*>(a.grad + base);
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      // Software pipeline, one vector per thread per iteration: the data of
      // vector v+1 (whose mask word arrived an iteration earlier) and the
      // mask word of v+2 are in flight while v is evaluated.  Masked vectors
      // are not read.
      constexpr int kS = kLogpsThreads;
      int64_t v = threadIdx.x;
      uint32_t m0 = v < nv ? __ldg(mrow + v) : 0u;
      uint32_t m1 = v + kS < nv ? __ldg(mrow + v + kS) : 0u;
      float4 l0 = z4, o0 = z4, r0 = z4;
      if (m0 != 0u) {
        l0 = __ldg(lrow + v);
        o0 = __ldg(orow + v);
        if (a.ref) r0 = __ldg(rrow + v);
      }
      for (; v < nv; v += kS) {
        float4 l1 = z4, o1 = z4, r1 = z4;
        if (m1 != 0u) {
          l1 = __ldg(lrow + v + kS);
          o1 = __ldg(orow + v + kS);
          if (a.ref) r1 = __ldg(rrow + v + kS);
        }
        const uint32_t m2 = v + 2 * kS < nv ? __ldg(mrow + v + 2 * kS) : 0u;
        float4 w;
        if (process_vec<kMode, kCount>(m0, l0, o0, r0, has_ref, f, gs, x, a, acc, w)) {
          if (a.grad) grow[v] = w;
        } else {
          deferred_list(a, b)[n_def++] = (uint32_t)v;
        }
        m0 = m1;
        m1 = m2;
        l0 = l1;
        o0 = o1;
        r0 = r1;
      }
    } else {
      // the scalar loop (rows that break the vector paths' rules): every
      // token on the general path
      for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x) {
        float w = 0.f;
        if (a.mask[base + t]) {
          const float lp = a.logps[base + t], o = a.old[base + t];
          const float rf = a.ref ? a.ref[base + t] : 0.f;
          const TokEpi<float> tt = tok_terms(lp, o, rf, x.A, a, x.em_seq);
          kahan2(acc.s, acc.c, make_float2(tt.q, tt.k));
          acc.count(tt.clip);
          w = token_w(lp, o, rf, tt, x, a);
        }
        if (a.grad) a.grad[base + t] = w;
      }
    }
    // the vectors this thread left to the general path, in the order it met
    // them (vector paths only: both need vec_ok's alignment)
    for (int k = 0; k < n_def; ++k) {
      const int64_t v = deferred_list(a, b)[k];
      const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(a.mask + base) + v);
      const float4 l4 = __ldg(reinterpret_cast<const float4*>(a.logps + base) + v);
      const float4 o4 = __ldg(reinterpret_cast<const float4*>(a.old + base) + v);
      const float4 r4 = has_ref ? __ldg(reinterpret_cast<const float4*>(a.ref + base) + v) : z4;
      float vq, vk;
      float4 w;
      vec_general(mw, l4, o4, r4, x, a, w, vq, vk, acc);
      kahan2(acc.s, acc.c, make_float2(vq, vk));
      if (a.grad) reinterpret_cast<float4*>(a.grad + base)[v] = w;
    }
    // the sequence's totals as float pairs: threads' Kahan sums, a fixed
    // xor tree per warp, warps in index order
    FF fq = warp_sum_ff2(FF{acc.s.x, -acc.c.x}), fk = warp_sum_ff2(FF{acc.s.y, -acc.c.y});
    unsigned nc[3] = {0u, 0u, 0u};
    if (a.counts_out) {
#pragma unroll
      for (int j = 0; j < 3; ++j) nc[j] = warp_sum(acc.nc[j]);
    }
    if (lane == 0) {
      s_ff[0][warp] = fq;
      s_ff[1][warp] = fk;
#pragma unroll
      for (int j = 0; j < 3; ++j) s_nc[j][warp] = nc[j];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      fq = s_ff[0][0];
      fk = s_ff[1][0];
#pragma unroll
      for (int k = 1; k < kLogpsThreads / 32; ++k) {
        fq = ff_add(fq, s_ff[0][k]);
        fk = ff_add(fk, s_ff[1][k]);
      }
      // P_b = sum q - A_b L_b for the clipped surrogate (the product exact
      // up to ~2^-48 relative); CISPO's q is the policy term itself
      const FF P = a.var.splits_A() ? ff_add(fq, ff_neg(ff_scale(FF{Ab.x, Ab.y}, (float)x.L))) : fq;
      put_total(a.seq + b, P, fk, x.L);
      if (a.per_seq) {
        a.per_seq[b] = ff_float(P);
        a.per_seq[a.B + b] = ff_float(fk);
        a.per_seq[2 * a.B + b] = (float)x.L;
      }
      if (a.counts_out) {
        unsigned n[3];
        for (int j = 0; j < 3; ++j) {
          n[j] = 0u;
          for (int k = 0; k < kLogpsThreads / 32; ++k) n[j] += s_nc[j][k];
        }
        add_clip_counts(a.hdr, n);
      }
      // the ticket: a release (this thread wrote the record and added the
      // clip counts) and, for the CTA that takes the last one, an acquire
      s_last = atom_add_acq_rel(&a.hdr->done_ctas, 1u) == gridDim.x - 1;
    }
  } else if (threadIdx.x == 0) {
    s_last = true;  // B == 0: a single CTA writes the zero loss
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0 && a.counts_out)  // every CTA added its counts before its ticket
    for (int j = 0; j < 3; ++j) a.counts_out[j] = __ldcg(&a.hdr->clip[j]);
  // the status of the call (every CTA set its bits before its ticket)
  const unsigned status = ((volatile unsigned*)&a.hdr->status)[0];
  if (!a.shard) {  // a shard's scalar comes from grpo_loss_finalize over all shards' totals
    // the scalar over the B sequence records, in index order
    final_scalar_ff<8>(a.seq, a.B, a.B > 0 ? s_NS[0] : 0ull, a.B > 0 ? s_NS[1] : 0ull,
                       a.reduction, a.norm_c, a.beta, status != 0u, a.out3, s_fin);
  }
  // every other CTA has taken its ticket, so nothing reads the counters any
  // more: leave the header clean for the next call (GRPO_FLAG_WORKSPACE_CLEAN),
  // the status bits moved to last_status
  if (threadIdx.x == 0) {
    WsHeader* h = a.hdr;
    h->last_status = status;
    h->status = 0u;
    h->done_ctas = 0u;
    h->N = 0ull;
    h->S = 0ull;
    h->clip[0] = h->clip[1] = h->clip[2] = 0ull;
    h->arrive = 0ull;
  }
}

// seven 27 KB CTAs per SM need the largest shared-memory carveout; the
// attribute, and the resident-CTA count it gives, are taken once per device
// (setting or querying them again costs host time)
static constexpr int kMaxDevices = 64;
static std::atomic<long long> g_capacity[kMaxDevices];  // 0: not yet known

static cudaError_t prepare_device(int dev, int64_t* cap) {
  const int d = dev & (kMaxDevices - 1);
  long long c = g_capacity[d].load(std::memory_order_acquire);
  if (c == 0) {
    cudaError_t e = cudaSuccess;
    for (auto k : {logps_kernel<kModeDefault, false>, logps_kernel<kModeDefault, true>,
                   logps_kernel<kModeVariant, false>, logps_kernel<kModeVariant, true>,
                   logps_kernel<kModeGspo, false>, logps_kernel<kModeGspo, true>,
                   logps_kernel<kModeK1, false>, logps_kernel<kModeK1, true>,
                   logps_kernel<kModeK2, false>, logps_kernel<kModeK2, true>,
                   logps_kernel<kModeCispo, false>, logps_kernel<kModeCispo, true>,
                   logps_kernel<kModeDual, false>, logps_kernel<kModeDual, true>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0, coop = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, logps_kernel<kModeDefault, false>, kLogpsThreads,
                                                           0)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
      return e;
    c = coop ? (long long)per_sm * sms : 0;
    if (c > (1ll << (64 - kArriveShift)) - 1) c = (1ll << (64 - kArriveShift)) - 1;  // the arrival field
    g_capacity[d].store(c > 0 ? c : -1, std::memory_order_release);  // -1: none
  }
  *cap = c > 0 ? c : 0;
  return cudaSuccess;
}

cudaError_t logps_fused_capacity(int64_t* cap) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return prepare_device(dev, cap);
}

cudaError_t launch_logps(const LogpsArgs& a, const grpo_profile_t* prof, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int64_t cap = 0;
  if ((e = prepare_device(dev, &cap)) != cudaSuccess) return e;
  const int64_t grid = a.B > 0 ? a.B : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kLogpsThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (a.fused) {
    // every CTA resident at once: the grid barrier's precondition
    if (grid > cap) return cudaErrorCooperativeLaunchTooLarge;
    if (a.flags & GRPO_FLAG_OVERLAP_LAUNCH) {
      // the caller vouches for residency (include/grpo.h); dispatch early
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
    } else {
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
    }
    cfg.numAttrs = 1;
  } else if (!(prof && (prof->start || prof->stop))) {
    // programmatic dependent launch: the CTAs may start while prep finishes
    // (a launch timed alone between events is an ordinary one)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  if (prof && prof->start) cudaEventRecord((cudaEvent_t)prof->start, s);
  const bool count = a.counts_out != nullptr;
  const bool gspo = a.var.seq_ratio && a.var.kl_type == GRPO_KL_K3 &&
                    a.var.surrogate == GRPO_SURROGATE_CLIP;
  const bool plain_clip = a.var.surrogate == GRPO_SURROGATE_CLIP && a.var.dual_c == 0.f &&
                          !a.var.seq_ratio;
  if (a.var.is_default())
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeDefault, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeDefault, false>, a);
  else if (plain_clip && a.var.kl_type == GRPO_KL_K1)
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeK1, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeK1, false>, a);
  else if (plain_clip && a.var.kl_type == GRPO_KL_K2)
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeK2, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeK2, false>, a);
  else if (a.var.surrogate == GRPO_SURROGATE_CLIP && a.var.dual_c > 0.f && !a.var.seq_ratio &&
           a.var.kl_type == GRPO_KL_K3)
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeDual, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeDual, false>, a);
  else if (a.var.surrogate == GRPO_SURROGATE_CISPO && a.var.kl_type == GRPO_KL_K3 &&
           !a.var.seq_ratio)
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeCispo, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeCispo, false>, a);
  else if (gspo)
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeGspo, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeGspo, false>, a);
  else
    e = count ? cudaLaunchKernelEx(&cfg, logps_kernel<kModeVariant, true>, a)
              : cudaLaunchKernelEx(&cfg, logps_kernel<kModeVariant, false>, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (prof && prof->stop) cudaEventRecord((cudaEvent_t)prof->stop, s);
  return e;
}

}  // namespace grpo
