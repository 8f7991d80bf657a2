// grpo_logps.cu -- the GRPO loss from per-token log-probs (no vocabulary).
//
// grpo.cpp README, "CUDA": the selected-token GRPO loss over [tokens] log
// probs, reduced inside each block (never with per-token atomics); RL-Kernel
// "GRPO Loss" page, "Accuracy" for the per-token terms and "Tensor and Data
// Parallel" for the two nested reductions (token slots -> sequence totals ->
// scalar).  Two kernels:
//   seq kernel   one CTA per sequence: the sequence's active-token count and
//                its policy / KL totals (fp32 per token, Kahan per thread,
//                double across the block, fixed order);
//   grad kernel  block 0 reduces the B sequence totals to the scalar
//                outputs; all blocks write dL/dlogp = w for every token.
// The whole cost is one pass over logps / old_logps / ref_logps / mask.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kSeqThreads = 256;
static constexpr int kGradThreads = 256;
static constexpr float kWPrecise = 0x1p-11f;

// k3 = e^d - d - 1 in fp32: a short series where e^d - 1 and d nearly
// cancel, the library expm1 elsewhere.
__device__ __forceinline__ float k3f(float d) {
  if (fabsf(d) < 0.0625f) {
    float q = __fmaf_rn(d, 1.0f / 720.0f, 1.0f / 120.0f);
    q = __fmaf_rn(d, q, 1.0f / 24.0f);
    q = __fmaf_rn(d, q, 1.0f / 6.0f);
    q = __fmaf_rn(d, q, 0.5f);
    return __fmul_rn(__fmul_rn(d, d), q);
  }
  return expm1f(d) - d;
}

struct TokTerms {
  float q;  // policy term minus its constant part: p = -A + q
  float k;  // KL term
  float g;  // g_pol + beta g_kl
};

// p = -min(rA, clip(r)A) = -A - min((r-1)A, (clip(r)-1)A).  The constant -A
// is summed per sequence in double (-A_i L_i): with a full mask the A_i of a
// group cancel exactly there, which an fp32 A rounded per token would break.
// The remainder uses r - 1 = expm1(d), accurate where r is close to 1.
__device__ __forceinline__ TokTerms tok_terms(float lp, float o, float rf, float A,
                                              const LogpsArgs& a) {
  TokTerms t;
  const float em = expm1f(__fsub_rn(lp, o));  // r - 1
  const float r = em + 1.0f;
  const float unc = em * A;
  const float cl = fminf(fmaxf(em, -a.eps_lo), a.eps_hi) * A;
  t.q = -fminf(unc, cl);
  const float d = a.ref ? __fsub_rn(rf, lp) : 0.0f;
  t.k = k3f(d);
  const bool clipped = (A > 0.f && em > a.eps_hi) || (A < 0.f && em < -a.eps_lo);
  const float gpol = clipped ? 0.f : -A * r;
  t.g = gpol + a.beta * (-expm1f(d));
  return t;
}

// dL/dlogp in double, for tokens whose gradient is large enough that the
// fp32 evaluation could be off by more than its rounding allowance.
__device__ __forceinline__ float w_precise(float lp, float o, float rf, double A, double c,
                                           const LogpsArgs& a) {
  const double r = exp((double)lp - (double)o);
  const double lo = 1.0 - (double)a.eps_lo, hi = 1.0 + (double)a.eps_hi;
  const double gpol = ((A > 0.0 && r > hi) || (A < 0.0 && r < lo)) ? 0.0 : -A * r;
  const double d = a.ref ? (double)rf - (double)lp : 0.0;
  return (float)((double)a.grad_scale * c * (gpol + (double)a.beta * -expm1(d)));
}

__device__ __forceinline__ void kahan(float& s, float& c, float x) {
  float y = __fsub_rn(x, c);
  float t = __fadd_rn(s, y);
  c = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}

__device__ __forceinline__ bool vec_ok(const LogpsArgs& a) {
  uintptr_t m = (uintptr_t)a.logps | (uintptr_t)a.old | (uintptr_t)a.ref | (uintptr_t)a.grad;
  return (a.T % 4 == 0) && ((m & 15) == 0) && (((uintptr_t)a.mask & 3) == 0);
}

__global__ void __launch_bounds__(kSeqThreads) logps_seq_kernel(const LogpsArgs a) {
  __shared__ double s_d[64];
  __shared__ int s_i[32];
  const int64_t b = blockIdx.x;
  const float A = (float)a.A[b];
  const int64_t base = b * a.T;
  float sp = 0.f, cp = 0.f, sk = 0.f, ck = 0.f;
  int cnt = 0;
  if (vec_ok(a)) {
    const int64_t nv = a.T / 4;
    for (int64_t q = threadIdx.x; q < nv; q += blockDim.x) {
      const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(a.mask + base) + q);
      if (mw == 0u) continue;  // masked storage is not read
      const float4 lp = __ldg(reinterpret_cast<const float4*>(a.logps + base) + q);
      const float4 od = __ldg(reinterpret_cast<const float4*>(a.old + base) + q);
      float4 rf = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a.ref) rf = __ldg(reinterpret_cast<const float4*>(a.ref + base) + q);
      const float l4[4] = {lp.x, lp.y, lp.z, lp.w}, o4[4] = {od.x, od.y, od.z, od.w};
      const float r4[4] = {rf.x, rf.y, rf.z, rf.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((mw >> (8 * j)) & 0xFFu) {
          TokTerms t = tok_terms(l4[j], o4[j], r4[j], A, a);
          kahan(sp, cp, t.q);
          kahan(sk, ck, t.k);
          ++cnt;
        }
    }
  } else {
    for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x) {
      if (!a.mask[base + t]) continue;
      TokTerms tt = tok_terms(a.logps[base + t], a.old[base + t],
                              a.ref ? a.ref[base + t] : 0.f, A, a);
      kahan(sp, cp, tt.q);
      kahan(sk, ck, tt.k);
      ++cnt;
    }
  }
  double v[2] = {(double)sp - (double)cp, (double)sk - (double)ck};
  block_sum<double, 2>(v, s_d);
  int n[1] = {cnt};
  block_sum<int, 1>(n, s_i);
  if (threadIdx.x == 0) {
    a.seq[b] = v[0] - a.A[b] * (double)n[0];
    a.seq[a.B + b] = v[1];
    a.L[b] = n[0];
  }
}

__global__ void __launch_bounds__(kGradThreads) logps_grad_kernel(const LogpsArgs a) {
  __shared__ double s_d[64];
  __shared__ long long s_l[64];
  long long ns[2] = {0, 0};
  for (int64_t i = threadIdx.x; i < a.B; i += blockDim.x) {
    int L = a.L[i];
    ns[0] += L;
    ns[1] += L > 0;
  }
  block_sum<long long, 2>(ns, s_l);
  const long long N = ns[0], S = ns[1];

  if (blockIdx.x == 0) {  // the scalar, in fixed order
    double v[2] = {0.0, 0.0};
    for (int64_t i = threadIdx.x; i < a.B; i += blockDim.x) {
      const double P = a.seq[i], K = a.seq[a.B + i];
      const int L = a.L[i];
      if (a.reduction == GRPO_TOKEN_MEAN) {
        v[0] += P;
        v[1] += K;
      } else if (L > 0) {
        v[0] += P / (double)L;
        v[1] += K / (double)L;
      }
      if (a.per_seq) {
        a.per_seq[i] = (float)P;
        a.per_seq[a.B + i] = (float)K;
        a.per_seq[2 * a.B + i] = (float)L;
      }
    }
    block_sum<double, 2>(v, s_d);
    if (threadIdx.x == 0) {
      const double den = a.reduction == GRPO_TOKEN_MEAN ? (double)(N > 0 ? N : 1)
                                                        : (double)(S > 0 ? S : 1);
      const double P = v[0] / den, K = v[1] / den;
      float o0 = (float)(P + (double)a.beta * K), o1 = (float)P, o2 = (float)K;
      if (a.hdr->status != 0u) o0 = o1 = o2 = NAN;
      a.out3[0] = o0;
      a.out3[1] = o1;
      a.out3[2] = o2;
    }
  }
  if (a.grad == nullptr) return;

  const double c_tok = 1.0 / (double)(N > 0 ? N : 1);
  const double inv_S = 1.0 / (double)(S > 0 ? S : 1);
  const int64_t BT = a.B * a.T;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  auto weight = [&](int64_t b) -> double {
    return a.reduction == GRPO_TOKEN_MEAN ? c_tok : inv_S / (double)a.L[b];
  };
  if (vec_ok(a)) {
    const int64_t nv = BT / 4;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nv; q += stride) {
      const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(a.mask) + q);
      float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mw != 0u) {
        const int64_t b = (4 * q) / a.T;
        const double c = weight(b);
        const double Ad = a.A[b];
        const float A = (float)Ad;
        const float gc = (float)((double)a.grad_scale * c);
        const float4 lp = __ldg(reinterpret_cast<const float4*>(a.logps) + q);
        const float4 od = __ldg(reinterpret_cast<const float4*>(a.old) + q);
        float4 rf = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.ref) rf = __ldg(reinterpret_cast<const float4*>(a.ref) + q);
        const float l4[4] = {lp.x, lp.y, lp.z, lp.w}, o4[4] = {od.x, od.y, od.z, od.w};
        const float r4[4] = {rf.x, rf.y, rf.z, rf.w};
        float w4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          w4[j] = 0.f;
          if ((mw >> (8 * j)) & 0xFFu) {
            float w = gc * tok_terms(l4[j], o4[j], r4[j], A, a).g;
            if (fabsf(w) > kWPrecise) w = w_precise(l4[j], o4[j], r4[j], Ad, c, a);
            w4[j] = w;
          }
        }
        out = make_float4(w4[0], w4[1], w4[2], w4[3]);
      }
      reinterpret_cast<float4*>(a.grad)[q] = out;
    }
  } else {
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < BT; j += stride) {
      float w = 0.f;
      if (a.mask[j]) {
        const int64_t b = j / a.T;
        const double c = weight(b);
        const double Ad = a.A[b];
        const float rf = a.ref ? a.ref[j] : 0.f;
        w = (float)((double)a.grad_scale * c) * tok_terms(a.logps[j], a.old[j], rf, (float)Ad, a).g;
        if (fabsf(w) > kWPrecise) w = w_precise(a.logps[j], a.old[j], rf, Ad, c, a);
      }
      a.grad[j] = w;
    }
  }
}

cudaError_t launch_logps(const LogpsArgs& a, cudaStream_t s) {
  if (a.B > 0) {
    logps_seq_kernel<<<(unsigned)a.B, kSeqThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int64_t grid = 1;
  if (a.grad) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t work = (a.B * a.T + 4 * kGradThreads - 1) / (4 * kGradThreads);
    grid = (int64_t)sms * 8;
    if (grid > work) grid = work;
    if (grid < 1) grid = 1;
  }
  logps_grad_kernel<<<(unsigned)grid, kGradThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
