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
//   seq      double[2B]       per-sequence policy / KL totals (logits path);
//                             the logps path keeps float-pair totals there,
//                             float4 {P.hi, P.lo, K.hi, K.lo} per sequence
//   slots    double[2 B T]    per-token policy / KL terms (logits path)
// ----------------------------------------------------------------------------
struct WsHeader {
  unsigned int status;             // device-detected error bits
  unsigned int done_ctas;          // reduce: CTAs finished (the last one forms the scalar)
  unsigned long long row_counter;  // rows: next row to claim
  unsigned long long N;            // active tokens  (prep: integer atomics, exact)
  unsigned long long S;            // live sequences (idem)
  unsigned long long clip[3];      // clipped tokens: upper, lower, dual (integer atomics)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t off_L, off_A, off_Aff, off_rng, off_seq, off_slots, total;
  __host__ __device__ WsLayout(int64_t B, int64_t T) {
    off_L = 256;
    off_A = off_L + align256(sizeof(int32_t) * (size_t)B);
    off_Aff = off_A + align256(sizeof(double) * (size_t)B);
    off_rng = off_Aff + align256(sizeof(float) * 2 * (size_t)B);
    off_seq = off_rng + align256(sizeof(int32_t) * 2 * (size_t)B);
    off_slots = off_seq + align256(sizeof(double) * 2 * (size_t)B);
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

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

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

__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float x = lane < nw ? scratch[lane] : -INFINITY;
  return warp_max(x);
}

// This thread's share of the level-2 sums over the B sequence totals
// (seq[0..B) policy, seq[B..2B) KL), in a fixed order: the token mean and
// the fixed constant add the totals, the sequence mean adds total / L_i over
// live sequences.  The
// totals were written by other CTAs of the same launch (made visible by
// their __threadfence before the ticket), so they are read from L2 (ld.cg),
// eight at a time to keep the loads in flight.
__device__ __forceinline__ void seq_totals(const double* seq, const int32_t* Ls, int64_t B,
                                           int reduction, double (&u)[2]) {
  constexpr int kBatch = 8;
  const int64_t stride = blockDim.x;
  for (int64_t j0 = threadIdx.x; j0 < B; j0 += kBatch * stride) {
    double P[kBatch], K[kBatch];
    int L[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int64_t j = j0 + k * stride;
      P[k] = j < B ? __ldcg(seq + j) : 0.0;
      K[k] = j < B ? __ldcg(seq + B + j) : 0.0;
      L[k] = j < B ? __ldcg(Ls + j) : 0;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (reduction != GRPO_SEQUENCE_MEAN) {
        u[0] += P[k];
        u[1] += K[k];
      } else if (L[k] > 0) {
        u[0] += P[k] / (double)L[k];
        u[1] += K[k] / (double)L[k];
      }
    }
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
  __host__ __device__ bool is_default() const {
    return kl_type == GRPO_KL_K3 && surrogate == GRPO_SURROGATE_CLIP && dual_c == 0.f;
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
// kernels (defined in the .cu files)
// ----------------------------------------------------------------------------
struct PrepArgs {
  const float* rewards;
  const int64_t* bounds;  // NULL -> uniform groups of spp
  int64_t B, T, G;
  int32_t spp;
  float adv_eps;
  int eps_add;
  const uint8_t* mask;  // the completion mask (may be NULL when T == 0)
  int count;            // 1: also count active tokens per sequence into L
  double* A;
  float2* Aff;     // nullable: the advantages as float pairs
  float* adv_out;  // nullable
  int32_t* L;      // used when counting
  int2* range;     // nullable: active range per sequence (when counting)
  WsHeader* hdr;
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
  int64_t B, T, V;
  float eps_lo, eps_hi, beta, grad_scale;
  int reduction;
  unsigned flags;
  int precise_ok;  // fp32 gradient output: rows may take the precise path
  ExpTable tab;
  Variant var;
  float norm_c;  // GRPO_FIXED_CONSTANT's constant
};

struct ReduceArgs {
  const uint8_t* mask;
  const int32_t* L;
  const double* A;
  double* seq;  // [2B] per-sequence totals
  const double* slot_p;
  const double* slot_k;
  int64_t B, T;
  float beta;
  int reduction;
  WsHeader* hdr;
  float* out3;
  float* per_seq;  // nullable
  int split_A;      // the clipped surrogate: add -A_i L_i per sequence
  float norm_c;     // GRPO_FIXED_CONSTANT's constant
  unsigned long long* counts_out;  // nullable [3]
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
  float4* seq;  // [B] {P.hi, P.lo, K.hi, K.lo}
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
};

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_rows(const RowArgs& a, grpo_dtype_t dt, const grpo_profile_t* prof,
                        cudaStream_t s);
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s);
cudaError_t launch_logps(const LogpsArgs& a, const grpo_profile_t* prof, cudaStream_t s);

}  // namespace grpo
