// grpo_internal.cuh -- shared device helpers of the GB300 GRPO loss library:
// workspace layout, storage types, the two exponential paths (fast MUFU and
// precise float-float), and deterministic block reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/grpo.h"

namespace grpo {

// ----------------------------------------------------------------------------
// workspace layout (caller-owned, 256-byte aligned; nothing needs zeroing)
//   header   256 B   status word, row counter
//   L        int32 [B]        active tokens per sequence
//   A        double[B]        advantages
//   Aff      float2[B]        the same advantages as float pairs (hi, lo)
//   range    int2[B]          first active token and last active token + 1
//                             ({0, 0} for an empty sequence)
//   seq      SeqTotal[B]      per-sequence totals (the records of
//                             grpo_seq_total_t: double totals on the logits
//                             path, float pairs on the logps path)
//   slots    double[2 B T]    per-token policy / KL terms (logits path); the
//                             logps path's per-thread lists of vectors left
//                             to its general path
// ----------------------------------------------------------------------------
struct WsHeader {
  unsigned int status;             // device-detected error bits
  unsigned int done_ctas;          // reduce: CTAs finished (the last one forms the scalar)
  unsigned long long row_counter;  // rows: next row to claim
  unsigned long long row_counter2; // GSPO's second row sweep: next row to claim
  unsigned long long N;            // active tokens  (prep: integer atomics, exact)
  unsigned long long S;            // live sequences (idem)
  unsigned long long clip[3];      // clipped tokens: upper, lower, dual (integer atomics)
  // one-launch logps kernel: the grid barrier and the batch counts in one
  // word, so that one relaxed atomic per CTA carries both (bits 52-63: CTAs
  // arrived, 41-51: live sequences S, 0-40: active tokens N)
  unsigned long long arrive;
  // grpo_loss_from_logps: the status bits of the call, moved here by its
  // last CTA, which also zeroes every counter above (the header is then
  // clean for the next call)
  unsigned int last_status;
  unsigned int pad_;
};
static_assert(sizeof(WsHeader) <= 256, "the header region is 256 bytes");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t off_L, off_A, off_Aff, off_rng, off_seq, off_slots, total;
  __host__ __device__ WsLayout(int64_t B, int64_t T) {
    off_L = 256;
    off_A = off_L + align256(sizeof(int32_t) * (size_t)B);
    off_Aff = off_A + align256(sizeof(double) * (size_t)B);
    off_rng = off_Aff + align256(sizeof(float) * 2 * (size_t)B);
    off_seq = off_rng + align256(sizeof(int32_t) * 2 * (size_t)B);
    off_slots = off_seq + align256((size_t)32 * (size_t)B);
    total = off_slots + align256(sizeof(double) * 2 * (size_t)B * (size_t)T);
  }
};

// ----------------------------------------------------------------------------
// storage types: 16-byte vectors unpacked to float
// ----------------------------------------------------------------------------
template <typename T> struct Storage;
template <> struct Storage<float> {
  static constexpr int kVec = 4;
  __device__ static float load1(const float* p) { return __ldg(p); }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  __device__ static void store1(float* p, float f) { *p = f; }
};
template <> struct Storage<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static float load1(const __nv_bfloat16* p) {
    return __uint_as_float(((uint32_t)__ldg((const unsigned short*)p)) << 16);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __device__ static uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                      pack2(f[6], f[7]));
  }
  __device__ static void store1(__nv_bfloat16* p, float f) { *p = __float2bfloat16_rn(f); }
};
template <> struct Storage<__half> {
  static constexpr int kVec = 8;
  __device__ static float load1(const __half* p) {
    return __half2float(__ushort_as_half(__ldg((const unsigned short*)p)));
  }
  __device__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      float2 g = __half22float2(h);
      f[2 * k] = g.x;
      f[2 * k + 1] = g.y;
    }
  }
  __device__ static uint32_t pack2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                      pack2(f[6], f[7]));
  }
  __device__ static void store1(__half* p, float f) { *p = __float2half_rn(f); }
};

// L2 eviction-priority policies (createpolicy) and loads / stores that carry
// them: rows that will be read again are kept (evict_last), rows read or
// written for the last time go first (evict_first).
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_hint(void* p, const uint4& v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// ----------------------------------------------------------------------------
// fast path: 2^x on the MUFU unit
// ----------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;  // float nearest log2(e)
constexpr double kLn2 = 0.69314718055994530942;

__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-thread online normaliser of one row (Milakov & Gimelshein, "Online
// normalizer calculation for softmax", 2018): running maximum m, its base-2
// image mL = fl(m log2e), and the sum s (Kahan-compensated by c) of
// 2^(x log2e - mL) over the elements seen so far.
struct OnlineLse {
  float m, mL, s, c;
  __device__ void init() { m = -INFINITY; mL = -INFINITY; s = 0.f; c = 0.f; }
  template <int N>
  __device__ __forceinline__ void update(const float* x) {
    float vmax = x[0];
#pragma unroll
    for (int j = 1; j < N; ++j) vmax = fmaxf(vmax, x[j]);
    if (vmax > m) {
      float nL = __fmul_rn(vmax, kLog2e);
      float f = ex2_fast(__fsub_rn(mL, nL));
      s = __fmul_rn(s, f);
      c = __fmul_rn(c, f);
      m = vmax;
      mL = nL;
    }
    if (m == -INFINITY) return;  // nothing finite seen yet (-inf logits)
    float e[N];
#pragma unroll
    for (int j = 0; j < N; ++j) e[j] = ex2_fast(__fmaf_rn(x[j], kLog2e, -mL));
    // pairwise sum of the N terms, then one compensated add
#pragma unroll
    for (int w = 1; w < N; w *= 2)
#pragma unroll
      for (int j = 0; j + w < N; j += 2 * w) e[j] = __fadd_rn(e[j], e[j + w]);
    float y = __fsub_rn(e[0], c);
    float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
};

// ----------------------------------------------------------------------------
// precise path: exp in float-float arithmetic, Tang's table-driven method
// (P. T. P. Tang, "Table-driven implementation of the exponential function in
// IEEE floating-point arithmetic", ACM TOMS 15(2), 1989):
//   t = n ln2/64 + r, |r| <= ln2/128,  e^t = 2^(n div 64) 2^((n mod 64)/64) e^r,
// the 64 table values carried as float pairs and e^r - 1 as a short Taylor
// polynomial.  Relative error ~1e-12 for t in [-87, 0].
// ----------------------------------------------------------------------------
struct ExpTable {
  float hi[64], lo[64];  // 2^(j/64) = hi + lo
  float c1, c2, c3;      // ln2/64 = c1 + c2 + c3, c1 with 11 significant bits
  float inv;             // 64 / ln2
};

struct FF { float hi, lo; };

__device__ __forceinline__ FF two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, err};
}
__device__ __forceinline__ FF fast_two_sum(float a, float b) {  // |a| >= |b|
  float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  FF s = two_sum(a.hi, b.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ FF ff_neg(FF a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ FF ff_scale(FF a, float f) {  // a * f
  const float ph = __fmul_rn(a.hi, f);
  const float pl = __fmaf_rn(a.hi, f, -ph);
  return fast_two_sum(ph, __fmaf_rn(a.lo, f, pl));
}
__device__ __forceinline__ float ff_float(FF a) { return __fadd_rn(a.hi, a.lo); }
// a / b: the fp32 quotient of the leading parts, then one correction from
// the remainder a - q1 b (formed with an exact product).
__device__ __forceinline__ FF ff_div(FF a, FF b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  const float p = __fmul_rn(q1, b.hi);
  const float pe = __fmaf_rn(q1, b.hi, -p);
  const FF r = two_sum(a.hi, -p);
  const float rem = __fadd_rn(r.hi, __fadd_rn(__fsub_rn(r.lo, pe),
                                              __fsub_rn(a.lo, __fmul_rn(q1, b.lo))));
  return fast_two_sum(q1, __fdiv_rn(rem, b.hi));
}
// A non-negative integer below 2^48 as an exact float pair.
__device__ __forceinline__ FF ff_from_u64(unsigned long long n) {
  const float hi = __ull2float_rn(n);
  const long long rest = (long long)n - (long long)hi;
  return {hi, (float)rest};
}

// thi / tlo: the 2^(j/64) table, staged in shared memory by the caller.
__device__ __forceinline__ FF exp_ff(float t_hi, float t_lo, const float* thi,
                                     const float* tlo, const ExpTable& tb) {
  if (!(t_hi >= -87.0f)) {
    if (t_hi != t_hi) return {t_hi, 0.f};
    return {0.f, 0.f};
  }
  float nf = rintf(__fmul_rn(t_hi, tb.inv));
  int n = (int)nf;
  float r1 = __fsub_rn(t_hi, __fmul_rn(nf, tb.c1));  // exact
  float p2 = __fmul_rn(nf, tb.c2);
  float e2 = __fmaf_rn(nf, tb.c2, -p2);
  FF r = two_sum(r1, -p2);
  r.lo = __fadd_rn(r.lo, __fsub_rn(__fsub_rn(t_lo, e2), __fmul_rn(nf, tb.c3)));
  r = fast_two_sum(r.hi, r.lo);
  float rh = r.hi;
  float q = __fmaf_rn(rh, 1.0f / 120.0f, 1.0f / 24.0f);
  q = __fmaf_rn(rh, q, 1.0f / 6.0f);
  q = __fmaf_rn(rh, q, 0.5f);
  q = __fmul_rn(__fmul_rn(rh, rh), q);
  q = __fmaf_rn(rh, r.lo, q);  // cross term of r^2/2
  float s_hi = rh, s_lo = __fadd_rn(r.lo, q);
  int j = n & 63;
  int m = n >> 6;  // floor(n / 64)
  float T_hi = thi[j], T_lo = tlo[j];
  float ph = __fmul_rn(T_hi, s_hi);
  float pl = __fmaf_rn(T_hi, s_hi, -ph);
  FF e = fast_two_sum(T_hi, ph);
  float small = __fadd_rn(__fadd_rn(pl, __fmul_rn(T_hi, s_lo)),
                          __fadd_rn(T_lo, __fmul_rn(T_lo, s_hi)));
  e = fast_two_sum(e.hi, __fadd_rn(e.lo, small));
  float sc = __int_as_float((m + 127) << 23);  // 2^m, m in [-126, 0]
  return {__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc)};
}

// ----------------------------------------------------------------------------
// deterministic reductions: fixed xor-shuffle trees and a fixed warp order
// ----------------------------------------------------------------------------
// Warp sum of floats carried as float pairs (two_sum at every level): the
// result in lane 0 is the exact sum up to ~2^-46 relative, in a fixed order.
__device__ __forceinline__ FF warp_sum_ff(float v) {
  FF acc = {v, 0.f};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, acc.hi, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o);
    const FF s = two_sum(acc.hi, oh);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(__fadd_rn(s.lo, acc.lo), ol);
  }
  return acc;
}

// Warp sum of float pairs, same fixed tree; result in lane 0.
__device__ __forceinline__ FF warp_sum_ff2(FF acc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, acc.hi, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o);
    const FF s = two_sum(acc.hi, oh);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(__fadd_rn(s.lo, acc.lo), ol);
  }
  return acc;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Block-wide sum of K values per thread; every thread gets the totals.
// `scratch` holds at least 32*K elements.  Contains __syncthreads().
template <typename T, int K>
__device__ __forceinline__ void block_sum(T (&v)[K], T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) scratch[k * 32 + warp] = v[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    T x = lane < nw ? scratch[k * 32 + lane] : T(0);
    v[k] = warp_sum(x);
  }
}

// ----------------------------------------------------------------------------
// the per-token epilogue and its variants
// ----------------------------------------------------------------------------
// The loss variant of a call (dockyard_rl "One loss, many algorithms",
// "CISPO", "Reference-KL penalty"; Relax "REINFORCE++-baseline" for k2).
struct Variant {
  float eps_lo, eps_hi, beta;
  float dual_c;  // 0: off; > 1: the dual clip on negative-advantage tokens
  int kl_type;   // grpo_kl_t
  int surrogate; // grpo_surrogate_t
  int seq_ratio; // 1: GSPO, one ratio per sequence (em is then the sequence's rho - 1)
  __host__ __device__ bool is_default() const {
    return kl_type == GRPO_KL_K3 && surrogate == GRPO_SURROGATE_CLIP && dual_c == 0.f &&
           seq_ratio == 0;
  }
  // the policy term's constant -A is summed per sequence (clipped surrogate)
  __host__ __device__ bool splits_A() const { return surrogate == GRPO_SURROGATE_CLIP; }
};

template <typename F>
struct TokEpi {
  F q;       // clipped surrogate: the policy term plus A (p = q - A); CISPO: p
  F k;       // the KL estimator
  F g;       // g_pol + beta g_kl = d(p + beta k)/d logp
  int clip;  // 0, or the clip that removed / clipped the token: 1 upper, 2 lower, 3 dual
};

// One token's scalars from em = r - 1, the log-prob lp, d = ref_logp - logp,
// emd = e^d - 1 and k3 = e^d - d - 1 (the caller evaluates these three with
// the accuracy its precision needs).  Clipped surrogate:
//   p + A = -min((r-1)A, (clip(r)-1)A), and with the dual clip (A < 0)
//   p + A = -max(min(...), (c-1)A); g_pol = 0 where a clip binds, else -A r.
// CISPO: p = -A clip(r) lp, g_pol = -A clip(r).
// KL: k3 = e^d - d - 1 (g_kl = -(e^d - 1)), k1 = -d (g_kl = 1),
//     k2 = d^2/2 (g_kl = -d); no reference: k = g_kl = 0.
template <typename F>
__device__ __forceinline__ TokEpi<F> token_epilogue(F em, F lp, F d, F emd, F k3, bool has_ref,
                                                    F A, const Variant& v) {
  TokEpi<F> t;
  const F lo = -(F)v.eps_lo, hi = (F)v.eps_hi;  // bounds on r - 1
  const F emc = em < lo ? lo : (em > hi ? hi : em);
  F gpol;
  if (v.surrogate == GRPO_SURROGATE_CISPO) {
    const F rc = (F)1 + emc;
    t.q = -A * rc * lp;
    gpol = -A * rc;
    t.clip = em > hi ? 1 : (em < lo ? 2 : 0);
  } else {
    const F unc = em * A, cl = emc * A;
    F m = unc < cl ? unc : cl;
    bool dual = false;
    if (v.dual_c > 0.f && A < (F)0) {
      const F cm1 = (F)v.dual_c - (F)1;
      const F dc = cm1 * A;
      if (dc > m) m = dc;
      dual = em > cm1;
    }
    t.q = -m;
    const bool up = A > (F)0 && em > hi, down = A < (F)0 && em < lo;
    gpol = (up || down || dual) ? (F)0 : -A * (em + (F)1);
    t.clip = up ? 1 : (down ? 2 : (dual ? 3 : 0));
  }
  F gkl;
  if (!has_ref) {
    t.k = (F)0;
    gkl = (F)0;
  } else if (v.kl_type == GRPO_KL_K1) {
    t.k = -d;
    gkl = (F)1;
  } else if (v.kl_type == GRPO_KL_K2) {
    t.k = d * d * (F)0.5;
    gkl = -d;
  } else {
    t.k = k3;
    gkl = -emd;
  }
  t.g = gpol + (F)v.beta * gkl;
  return t;
}

// d g_kl / d ref_logp in magnitude (= d g_kl / d logp), for error budgets:
// e^d for k3, 0 for k1, 1 for k2.
__device__ __forceinline__ float kl_slope(int kl_type, float emd) {
  return kl_type == GRPO_KL_K1 ? 0.f : (kl_type == GRPO_KL_K2 ? 1.f : 1.f + emd);
}

// This CTA's clip counts into the workspace header (one atomic per nonzero
// count; integer sums are exact in any order).  Call with the CTA's totals
// from one thread.
__device__ __forceinline__ void add_clip_counts(WsHeader* hdr, const unsigned (&n)[3]) {
#pragma unroll
  for (int j = 0; j < 3; ++j)
    if (n[j]) atomicAdd(&hdr->clip[j], (unsigned long long)n[j]);
}

// ----------------------------------------------------------------------------
// per-sequence totals and the final scalar
// ----------------------------------------------------------------------------
// One sequence's totals (grpo_seq_total_t, 32 bytes).  kind 1: P, K as
// doubles (logits path); kind 2: P and K as float pairs in the first 16
// bytes (logps path).
struct __align__(16) SeqTotal {
  double P, K;
  long long L;
  int kind;
  int pad;
};
static_assert(sizeof(SeqTotal) == 32, "grpo_seq_total_t is 32 bytes");
enum : int { kTotalsDouble = 1, kTotalsFF = 2 };

__device__ __forceinline__ void put_total(SeqTotal* r, double P, double K, int L) {
  SeqTotal t;
  t.P = P;
  t.K = K;
  t.L = L;
  t.kind = kTotalsDouble;
  t.pad = 0;
  *r = t;
}
__device__ __forceinline__ void put_total(SeqTotal* r, FF P, FF K, int L) {
  uint4* q = reinterpret_cast<uint4*>(r);
  q[0] = make_uint4(__float_as_uint(P.hi), __float_as_uint(P.lo), __float_as_uint(K.hi),
                    __float_as_uint(K.lo));
  q[1] = make_uint4((unsigned)L, 0u, (unsigned)kTotalsFF, 0u);
}

// The final scalar from B records, by the first kFinalThreads threads of a
// CTA (every thread of the CTA calls it: it holds __syncthreads).  Each
// thread takes records j = t, t + 128, ... in index order (loads batched
// kBatch at a time, from L2: the records may come from other CTAs of the
// same launch), then a fixed xor tree per warp and the four warps in index
// order.  The token mean and the fixed constant add the totals; the sequence
// mean adds total / L over live sequences; then one division by N, S or C.
// The order depends only on the index, so an unsharded call and
// grpo_loss_finalize over the same records produce the same bits.
// kind 1 sums in double, kind 2 in float pairs; each record is read once,
// and the kind of the whole set is known after the loads (no separate read
// of the first record ahead of them).  Records of both kinds, of another
// kind, or a nonzero `bad`, give NaN outputs.  Thread 0 writes out3.
constexpr int kFinalThreads = 128;
struct FinalSmem {
  double d[2][kFinalThreads / 32];
  FF f[2][kFinalThreads / 32];
  unsigned kinds;  // bit 0: a kind-1 record, bit 1: kind 2, bit 2: another
};
// One float-pair record's contribution (the sequence mean divides by L and
// skips empty sequences: false), shared by both final forms.
__device__ __forceinline__ bool ff_record(const uint4& lo, int L, int reduction, FF& P, FF& K) {
  P = {__uint_as_float(lo.x), __uint_as_float(lo.y)};
  K = {__uint_as_float(lo.z), __uint_as_float(lo.w)};
  if (reduction == GRPO_SEQUENCE_MEAN) {
    if (L == 0) return false;
    const FF Lf = {(float)L, 0.f};
    P = ff_div(P, Lf);
    K = ff_div(K, Lf);
  }
  return true;
}
// The float-pair outputs from the warps' partial sums (thread 0).
__device__ __forceinline__ void ff_final_outputs(const FinalSmem& sm, unsigned long long N,
                                                 unsigned long long S, int reduction,
                                                 float norm_c, float beta, float& o0, float& o1,
                                                 float& o2) {
  FF P = sm.f[0][0], K = sm.f[1][0];
#pragma unroll
  for (int k = 1; k < kFinalThreads / 32; ++k) {
    P = ff_add(P, sm.f[0][k]);
    K = ff_add(K, sm.f[1][k]);
  }
  const FF den = reduction == GRPO_FIXED_CONSTANT
                     ? FF{norm_c, 0.f}
                     : ff_from_u64(reduction == GRPO_TOKEN_MEAN ? (N > 0 ? N : 1) : (S > 0 ? S : 1));
  P = ff_div(P, den);
  K = ff_div(K, den);
  o0 = ff_float(ff_add(P, ff_scale(K, beta)));
  o1 = ff_float(P);
  o2 = ff_float(K);
}

static __device__ __forceinline__ void final_scalar(const SeqTotal* recs, int64_t B, unsigned long long N,
                             unsigned long long S, int reduction, float norm_c, float beta,
                             bool bad, float* out3, FinalSmem& sm) {
  constexpr int kBatch = 4;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) sm.kinds = 0u;
  __syncthreads();
  double ud[2] = {0.0, 0.0};
  FF uf[2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (t < kFinalThreads) {
    unsigned kinds = 0u;
    for (int64_t j0 = t; j0 < B; j0 += kBatch * kFinalThreads) {
      // per record: the four totals words, the count and the kind
      uint4 lo[kBatch];
      unsigned Lk[kBatch], kk[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t j = j0 + (int64_t)k * kFinalThreads;
        const uint4* q = reinterpret_cast<const uint4*>(recs + (j < B ? j : 0));
        const unsigned* h = reinterpret_cast<const unsigned*>(q + 1);
        lo[k] = j < B ? __ldcg(q) : make_uint4(0u, 0u, 0u, 0u);
        Lk[k] = j < B ? __ldcg(h) : 0u;
        kk[k] = j < B ? __ldcg(h + 2) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int L = (int)Lk[k];
        const int rk = (int)kk[k];
        if (rk == kTotalsDouble) {
          kinds |= 1u;
          double P = __hiloint2double((int)lo[k].y, (int)lo[k].x);
          double K = __hiloint2double((int)lo[k].w, (int)lo[k].z);
          if (reduction == GRPO_SEQUENCE_MEAN) {
            if (L == 0) continue;
            P /= (double)L;
            K /= (double)L;
          }
          ud[0] += P;
          ud[1] += K;
        } else if (rk == kTotalsFF) {
          kinds |= 2u;
          FF P, K;
          if (!ff_record(lo[k], L, reduction, P, K)) continue;
          uf[0] = ff_add(uf[0], P);
          uf[1] = ff_add(uf[1], K);
        } else if (j0 + (int64_t)k * kFinalThreads < B) {
          kinds |= 4u;
        }
      }
    }
    kinds = __reduce_or_sync(0xFFFFFFFFu, kinds);
    if (lane == 0 && kinds) atomicOr(&sm.kinds, kinds);
  }
  __syncthreads();
  const unsigned ks = sm.kinds;
  const int kind = ks == 2u ? kTotalsFF : kTotalsDouble;  // no records: kind 1, zeros
  if (t < kFinalThreads) {
    if (kind == kTotalsDouble) {
      ud[0] = warp_sum(ud[0]);
      ud[1] = warp_sum(ud[1]);
      if (lane == 0) {
        sm.d[0][warp] = ud[0];
        sm.d[1][warp] = ud[1];
      }
    } else {
      uf[0] = warp_sum_ff2(uf[0]);
      uf[1] = warp_sum_ff2(uf[1]);
      if (lane == 0) {
        sm.f[0][warp] = uf[0];
        sm.f[1][warp] = uf[1];
      }
    }
  }
  __syncthreads();
  if (t != 0) return;
  float o0, o1, o2;
  if (kind == kTotalsDouble) {
    double P = sm.d[0][0], K = sm.d[1][0];
#pragma unroll
    for (int k = 1; k < kFinalThreads / 32; ++k) {
      P += sm.d[0][k];
      K += sm.d[1][k];
    }
    const double den = reduction == GRPO_TOKEN_MEAN      ? (double)(N > 0 ? N : 1)
                       : reduction == GRPO_SEQUENCE_MEAN ? (double)(S > 0 ? S : 1)
                                                         : (double)norm_c;
    P /= den;
    K /= den;
    o0 = (float)(P + (double)beta * K);
    o1 = (float)P;
    o2 = (float)K;
  } else {
    ff_final_outputs(sm, N, S, reduction, norm_c, beta, o0, o1, o2);
  }
  if (bad || (ks & 4u) || ks == 3u) o0 = o1 = o2 = NAN;
  out3[0] = o0;
  out3[1] = o1;
  out3[2] = o2;
}

// final_scalar for B records all known to be float pairs (written by the
// calling launch): the same order and arithmetic, hence the same bits, with
// kBatch records per thread in flight at once.
template <int kBatch>
static __device__ __forceinline__ void final_scalar_ff(const SeqTotal* recs, int64_t B,
                                                       unsigned long long N, unsigned long long S,
                                                       int reduction, float norm_c, float beta,
                                                       bool bad, float* out3, FinalSmem& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  FF uf[2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (t < kFinalThreads) {
    for (int64_t j0 = t; j0 < B; j0 += kBatch * kFinalThreads) {
      uint4 lo[kBatch];
      unsigned Lk[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t j = j0 + (int64_t)k * kFinalThreads;
        const uint4* q = reinterpret_cast<const uint4*>(recs + (j < B ? j : 0));
        lo[k] = j < B ? __ldcg(q) : make_uint4(0u, 0u, 0u, 0u);
        Lk[k] = j < B ? __ldcg(reinterpret_cast<const unsigned*>(q + 1)) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (j0 + (int64_t)k * kFinalThreads >= B) continue;
        FF P, K;
        if (!ff_record(lo[k], (int)Lk[k], reduction, P, K)) continue;
        uf[0] = ff_add(uf[0], P);
        uf[1] = ff_add(uf[1], K);
      }
    }
    uf[0] = warp_sum_ff2(uf[0]);
    uf[1] = warp_sum_ff2(uf[1]);
    if (lane == 0) {
      sm.f[0][warp] = uf[0];
      sm.f[1][warp] = uf[1];
    }
  }
  __syncthreads();
  if (t != 0) return;
  float o0, o1, o2;
  ff_final_outputs(sm, N, S, reduction, norm_c, beta, o0, o1, o2);
  if (bad) o0 = o1 = o2 = NAN;
  out3[0] = o0;
  out3[1] = o1;
  out3[2] = o2;
}

// ----------------------------------------------------------------------------
// kernels (defined in the .cu files)
// ----------------------------------------------------------------------------
struct PrepArgs {
  const float* rewards;   // [Bg]
  const int64_t* bounds;  // NULL -> uniform groups of spp
  int64_t B, T, G;        // B: sequences whose masks are scanned (a shard's)
  int64_t Bg;             // sequences the groups cover (the whole batch)
  int64_t seq_begin;      // the scanned sequences' first index in the batch
  unsigned long long* NS; // [2]: N and S receive the scanned counts (atomics)
  int32_t spp;
  float adv_eps;
  int eps_add;
  const uint8_t* mask;  // the completion mask (may be NULL when T == 0)
  int count;            // 1: also count active tokens per sequence into L
  double* A;
  float2* Aff;     // nullable: the advantages as float pairs
  float* adv_out;  // nullable
  int32_t* L;      // nullable: per-sequence counts (when counting)
  int2* range;     // nullable: active range per sequence (when counting)
  WsHeader* hdr;   // status word (may be NULL when G == 0)
};

struct RowArgs {
  const void* policy;
  const void* ref;
  void* grad;  // nullable
  const int64_t* actions;
  const float* old;
  const uint8_t* mask;
  const int32_t* L;
  const double* A;
  double* slot_p;
  double* slot_k;
  float* logps_out;  // nullable
  WsHeader* hdr;
  const unsigned long long* NS;  // [2]: N and S of the whole batch
  int64_t B, T, V;
  float eps_lo, eps_hi, beta, grad_scale;
  int reduction;
  unsigned flags;
  int precise_ok;  // fp32 gradient output: rows may take the precise path
  int tmem_cols;   // tensor-memory columns a row CTA keeps policy vectors in (0: none)
  ExpTable tab;
  Variant var;
  float norm_c;  // GRPO_FIXED_CONSTANT's constant
};

struct ReduceArgs {
  const uint8_t* mask;
  const int32_t* L;
  const double* A;
  SeqTotal* seq;  // [B] per-sequence totals
  const double* slot_p;
  double* slot_k;
  int64_t B, T;
  float beta;
  int reduction;
  WsHeader* hdr;
  const unsigned long long* NS;  // [2]: N and S of the whole batch
  float* out3;
  float* per_seq;  // nullable
  int split_A;      // the clipped surrogate: add -A_i L_i per sequence
  float norm_c;     // GRPO_FIXED_CONSTANT's constant
  unsigned long long* counts_out;  // nullable [3]
  int shard;        // 1: write the totals only (the scalar comes from grpo_loss_finalize)
  // from_slots (GSPO, the vocab-parallel path): the slots hold logp and
  // d = ref_logp - logp; this kernel forms the ratios (rho_i for GSPO), the
  // per-token terms and w = dL/dlogp, written to w_out (or over d)
  Variant var;
  const float* old;
  float grad_scale;
  int from_slots;
  double* w_out;  // nullable
};

// The vocabulary-parallel path (grpo_vocab.cu): a rank's slice of every row,
// [rows, Vk] from vocabulary entry v_begin on, in chunks of kVChunk.
constexpr int64_t kVChunk = 4096;
struct VocabArgs {
  const void* policy;
  const void* ref;
  const int64_t* actions;
  const uint8_t* mask;
  int64_t rows, Vk, v_begin, nck, V;  // nck: chunks of the slice (partials) or of all slices (merge)
  float4* part_p;      // [nck][rows] partial normalisers {M, Z.hi, Z.lo, 0}
  float4* part_r;
  float* act_logits;   // [2][rows]: policy and reference logit of the action
  int precise;         // fp32 logits: float-float exponentials
  ExpTable tab;
  double* slot_p;      // merge: logp
  double* slot_k;      // merge: d = ref_logp - logp
  double* lse_w;       // merge: [rows] policy logsumexp
  float* logps_out;    // nullable
  WsHeader* hdr;
};

struct LogpsArgs {
  const float* logps;
  const float* old;
  const float* ref;  // nullable
  const uint8_t* mask;
  const double* A;
  const float2* Aff;  // the advantages as float pairs
  const int2* range;  // active range per sequence
  int32_t* L;
  SeqTotal* seq;  // [B] per-sequence totals
  float* grad;  // nullable
  float* out3;
  float* per_seq;  // nullable
  WsHeader* hdr;
  int64_t B, T;
  float eps_lo, eps_hi, beta, grad_scale;
  int reduction;
  Variant var;
  float norm_c;  // GRPO_FIXED_CONSTANT's constant
  unsigned long long* counts_out;  // nullable [3]
  const unsigned long long* NS;    // [2]: N and S of the whole batch
  int shard;     // 1: write the totals only (the scalar comes from grpo_loss_finalize)
  unsigned flags;  // grpo_params_t.flags
  // One-launch form (fused = 1, a cooperative launch): each CTA scans its own
  // mask row and forms its own advantage from the groups below (as the
  // separate pass would), adds its counts to hdr->arrive and waits at the
  // grid barrier that word also is before any count is read; A, Aff, range
  // and L are unused.
  int fused;
  const float* rewards;   // [Bg]
  const int64_t* bounds;  // NULL -> uniform groups of spp
  int64_t G, Bg, seq_begin;
  int32_t spp;
  float adv_eps;
  int eps_add;
  float* adv_out;  // nullable [B]
  // the workspace's token-slot area (16 bytes per slot, unused by this
  // path's sums): each sequence's vectors left to the general path
  uint32_t* defer;
};

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
// sequences the one-launch logps kernel can take (its CTAs all resident)
cudaError_t logps_fused_capacity(int64_t* cap);
cudaError_t launch_rows(const RowArgs& a, grpo_dtype_t dt, const grpo_profile_t* prof,
                        cudaStream_t s);
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s);
cudaError_t launch_gspo_rows(const RowArgs& a, grpo_dtype_t dt, int phase,
                             const grpo_profile_t* prof, cudaStream_t s);
cudaError_t launch_vocab_partials(const VocabArgs& a, grpo_dtype_t dt, cudaStream_t s);
cudaError_t launch_vocab_merge(const VocabArgs& a, cudaStream_t s);
cudaError_t launch_vocab_grad(const RowArgs& a, grpo_dtype_t dt, int64_t v_begin,
                              const double* lse_w, cudaStream_t s);
cudaError_t launch_logps(const LogpsArgs& a, const grpo_profile_t* prof, cudaStream_t s);
cudaError_t launch_finalize(const SeqTotal* recs, int64_t B, const unsigned long long* NS,
                            int reduction, float norm_c, float beta, float* out3, cudaStream_t s);

}  // namespace grpo
