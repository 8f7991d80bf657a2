// grpo_rows.cu -- the fused forward + backward over vocabulary rows.
//
// One persistent CTA (512 threads, two per SM) takes token rows from a
// device counter.  For an active row (completion_mask != 0):
//   sweep 1   one streaming read of the policy row and of the reference row,
//             each reduced to (max, sum exp) by a per-thread online
//             normaliser and a fixed-order block combine
//             (RL-Kernel "GRPO Loss" intro: logits -> ratio / KL via online
//             softmax; grpo.cpp README "CUDA": carry the row maximum and
//             normaliser together);
//   finish    warp 0, in double: logp, ref_logp, ratio, clipped surrogate,
//             k3 KL, token weight and w = dL/dlogp (RL-Kernel "Accuracy";
//             dockyard_rl "One loss, many algorithms", "Reference-KL
//             penalty"); the few transcendentals run on separate lanes;
//   sweep 2   a second read of the policy row (kept in L2 by an evict_last
//             policy on the first read) writes dL/dx_v = w (1[v=a] - softmax_v)
//             into the gradient buffer (grpo.cpp README "CUDA": the fused
//             kernel writes the full logits gradient, in place if asked).
// A masked row is never read: its gradient row is written as zeros (or left
// alone under GRPO_SKIP_MASKED_GRAD_ROWS).
//
// Precision.  The fast normaliser (MUFU 2^x, fp32 Kahan sums, compensated
// warp sums, double across warps) has a relative error below 2^-19.  When the
// gradient is stored in fp32 and a row's gradient is large enough that this
// error could exceed 2^-31 on an element, the row is refined: both
// normalisers are recomputed with a float-float exponential and float-float
// sums, and gradient elements above 2^-12 are evaluated in double.  bf16 /
// f16 gradients never need it.
//
// Per-token policy and KL terms go to [B,T] double slots; the fixed-order
// reduction over them is in grpo_reduce.cu.
#include "grpo_internal.cuh"

namespace grpo {

static constexpr int kRowThreads = 512;
static constexpr int kUnroll = 4;
static constexpr double kZErrBound = 0x1p-19;
static constexpr double kTau = 0x1p-31;
static constexpr float kElemPrecise = 0x1p-12f;

struct RowScalars {
  double lse_p, w;
  double p, k, logp;
  float LL;    // fl32(lse_p * log2e): base-2 shift of the gradient exponent
  float wneg;  // -w as float
  float ga;    // gradient at the action element
  int precise;
};

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

// ---------------------------------------------------------------- sweep 1
template <typename T>
__device__ __forceinline__ void lse_fast(const T* row, int64_t V, OnlineLse& st, uint64_t pol) {
  constexpr int VEC = Storage<T>::kVec;
  const Geom<T> gm(row, V);
  if ((int)threadIdx.x < gm.head || (int)threadIdx.x < gm.tail) {
    float x[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) x[j] = -INFINITY;
    if ((int)threadIdx.x < gm.head) x[0] = Storage<T>::load1(row + threadIdx.x);
    if ((int)threadIdx.x < gm.tail) x[1] = Storage<T>::load1(row + gm.t0 + threadIdx.x);
    st.update<VEC>(x);
  }
  const uint4* vp = reinterpret_cast<const uint4*>(row + gm.head);
  const int64_t stride = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (kUnroll - 1) * stride < gm.nvec; k += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_hint(vp + k + u * stride, pol);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float x[VEC];
      Storage<T>::unpack(v[u], x);
      st.update<VEC>(x);
    }
  }
  for (; k < gm.nvec; k += stride) {
    float x[VEC];
    Storage<T>::unpack(ld_hint(vp + k, pol), x);
    st.update<VEC>(x);
  }
}

// Block combine of the per-thread normalisers of the policy (a) and
// reference (b) rows.  Every thread gets the row maxima; warp 0 gets the two
// sums Z = sum_v 2^(x_v log2e - ML) in double (ML = fl(M log2e)).
__device__ __forceinline__ void combine_lse(const OnlineLse& a, const OnlineLse& b,
                                            float* fs, double* ds, float& Ma, float& Mb,
                                            double& Za, double& Zb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  float ma = warp_max(a.m), mb = warp_max(b.m);
  __syncthreads();
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
  if (lane == 0) {
    ds[warp] = (double)wa.hi + (double)wa.lo;
    ds[32 + warp] = (double)wb.hi + (double)wb.lo;
  }
  __syncthreads();
  if (warp == 0) {
    Za = warp_sum(lane < nw ? ds[lane] : 0.0);
    Zb = warp_sum(lane < nw ? ds[32 + lane] : 0.0);
  }
}

// ------------------------------------------------- precise normaliser sweep
// sum_v exp(x_v - M) with x_v - M exact as a float pair, float-float
// exponentials and float-float per-thread sums; warp 0 gets the total.
template <typename T>
__device__ double sum_exp_precise(const T* row, int64_t V, float M, const float* thi,
                                  const float* tlo, const ExpTable& tb, double* ds) {
  FF acc = {0.f, 0.f};
  for (int64_t v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = Storage<T>::load1(row + v);
    const FF t = two_sum(x, -M);
    const FF e = exp_ff(t.hi, t.lo, thi, tlo, tb);
    const FF s = two_sum(acc.hi, e.hi);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, e.lo));
  }
  double z[1] = {(double)acc.hi + (double)acc.lo};
  block_sum<double, 1>(z, ds);
  return z[0];
}

// ------------------------------------------------------------- row finish
// Run by all 32 lanes of warp 0; the result is valid in lane 0.  lse_* are
// the logsumexp of the two rows as (base, log argument): lse = base + log(z).
__device__ RowScalars finish_row(const RowArgs& a, double base_p, double z_p, double base_r,
                                 double z_r, float xa, float ya, float o, double A, double c,
                                 bool want_grad) {
  const int lane = threadIdx.x & 31;
  xa = __shfl_sync(0xFFFFFFFFu, xa, 0);
  ya = __shfl_sync(0xFFFFFFFFu, ya, 0);
  o = __shfl_sync(0xFFFFFFFFu, o, 0);
  // level 1: the two logs on lanes 0 / 1
  const double lz = log(lane == 1 ? z_r : z_p);
  const double lse_p = base_p + __shfl_sync(0xFFFFFFFFu, lz, 0);
  const double lse_r = base_r + __shfl_sync(0xFFFFFFFFu, lz, 1);
  const double lp = (double)xa - lse_p;
  const double lr = (double)ya - lse_r;
  const double d = lr - lp;
  // level 2: expm1 of (logp - old, d, logp) on lanes 0 / 1 / 2
  const double arg = lane == 0 ? lp - (double)o : (lane == 1 ? d : lp);
  const double em = expm1(arg);
  const double rm1 = __shfl_sync(0xFFFFFFFFu, em, 0);
  const double emd = __shfl_sync(0xFFFFFFFFu, em, 1);
  const double emlp = __shfl_sync(0xFFFFFFFFu, em, 2);
  RowScalars r;
  const double ratio = 1.0 + rm1;
  const double lo_b = 1.0 - (double)a.eps_lo, hi_b = 1.0 + (double)a.eps_hi;
  const double unc = ratio * A;
  const double rc = ratio < lo_b ? lo_b : (ratio > hi_b ? hi_b : ratio);
  const double cl = rc * A;
  const double gpol = ((A > 0.0 && ratio > hi_b) || (A < 0.0 && ratio < lo_b)) ? 0.0 : -A * ratio;
  const double beta = (double)a.beta, gs = (double)a.grad_scale;
  const double w = gs * c * (gpol - beta * emd);
  r.lse_p = lse_p;
  r.p = -(unc < cl ? unc : cl);
  r.k = emd - d;
  r.logp = lp;
  r.w = w;
  r.wneg = (float)(-w);
  r.LL = (float)(lse_p * (double)kLog2e);
  r.ga = (float)(-w * emlp);
  r.precise = 0;
  if (want_grad && a.precise_ok) {
    const double sens = fabs(w) + fabs(gs * c) * (fabs(A) * ratio + 2.0 * beta * (1.0 + emd));
    r.precise = sens * kZErrBound > kTau;
  }
  return r;
}

// ---------------------------------------------------------------- sweep 2
__device__ __forceinline__ float grad_elem(float x, int64_t v, const RowScalars& rs, int64_t act) {
  const float p = ex2_fast(__fmaf_rn(x, kLog2e, -rs.LL));
  float g = __fmul_rn(rs.wneg, p);
  if (rs.precise && fabsf(g) > kElemPrecise) g = (float)(-rs.w * exp((double)x - rs.lse_p));
  if (v == act) g = rs.ga;
  return g;
}

template <typename T>
__device__ void grad_sweep(const T* x, T* g, int64_t V, int64_t act, const RowScalars& rs,
                           uint64_t pol_in, uint64_t pol_out) {
  constexpr int VEC = Storage<T>::kVec;
  const bool same_phase = (((uintptr_t)x ^ (uintptr_t)g) & 15) == 0;
  if (!same_phase) {  // differently aligned buffers: element by element
    for (int64_t v = threadIdx.x; v < V; v += blockDim.x)
      Storage<T>::store1(g + v, grad_elem(Storage<T>::load1(x + v), v, rs, act));
    return;
  }
  const Geom<T> gm(x, V);
  if ((int)threadIdx.x < gm.head) {
    const int64_t v = threadIdx.x;
    Storage<T>::store1(g + v, grad_elem(Storage<T>::load1(x + v), v, rs, act));
  }
  if ((int)threadIdx.x < gm.tail) {
    const int64_t v = gm.t0 + threadIdx.x;
    Storage<T>::store1(g + v, grad_elem(Storage<T>::load1(x + v), v, rs, act));
  }
  const uint4* xv = reinterpret_cast<const uint4*>(x + gm.head);
  uint4* gv = reinterpret_cast<uint4*>(g + gm.head);
  const int64_t stride = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (kUnroll - 1) * stride < gm.nvec; k += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_hint(xv + k + u * stride, pol_in);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[VEC];
      Storage<T>::unpack(v[u], f);
      const int64_t base = gm.head + (k + u * stride) * VEC;
#pragma unroll
      for (int j = 0; j < VEC; ++j) f[j] = grad_elem(f[j], base + j, rs, act);
      st_hint(gv + k + u * stride, Storage<T>::pack(f), pol_out);
    }
  }
  for (; k < gm.nvec; k += stride) {
    float f[VEC];
    Storage<T>::unpack(ld_hint(xv + k, pol_in), f);
    const int64_t base = gm.head + k * VEC;
#pragma unroll
    for (int j = 0; j < VEC; ++j) f[j] = grad_elem(f[j], base + j, rs, act);
    st_hint(gv + k, Storage<T>::pack(f), pol_out);
  }
}

template <typename T>
__device__ void zero_row(T* g, int64_t V, uint64_t pol) {
  const Geom<T> gm(g, V);
  if ((int)threadIdx.x < gm.head) Storage<T>::store1(g + threadIdx.x, 0.f);
  if ((int)threadIdx.x < gm.tail) Storage<T>::store1(g + gm.t0 + threadIdx.x, 0.f);
  uint4* gv = reinterpret_cast<uint4*>(g + gm.head);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = threadIdx.x; k < gm.nvec; k += blockDim.x) st_hint(gv + k, z, pol);
}

// ------------------------------------------------------------------ kernel
template <typename T>
__global__ void __launch_bounds__(kRowThreads, 2) rows_kernel(const RowArgs a) {
  __shared__ float s_f[64];
  __shared__ double s_d[64];
  __shared__ float s_thi[64], s_tlo[64];
  __shared__ long long s_row;
  __shared__ RowScalars s_rs;
  __shared__ long long s_NS[2];

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x < 64) {
    s_thi[threadIdx.x] = a.tab.hi[threadIdx.x];
    s_tlo[threadIdx.x] = a.tab.lo[threadIdx.x];
  }
  // N = active tokens, S = live sequences (every CTA, fixed order)
  {
    long long ns[2] = {0, 0};
    for (int64_t i = threadIdx.x; i < a.B; i += blockDim.x) {
      const int L = a.L[i];
      ns[0] += L;
      ns[1] += L > 0;
    }
    block_sum<long long, 2>(ns, reinterpret_cast<long long*>(s_d));
    if (threadIdx.x == 0) { s_NS[0] = ns[0]; s_NS[1] = ns[1]; }
  }
  __syncthreads();
  const long long N = s_NS[0], S = s_NS[1];
  // token weight: 1/max(N,1) (token mean) or 1/(max(S,1) L_i) (sequence mean)
  const double c_tok = 1.0 / (double)(N > 0 ? N : 1);
  const double inv_S = 1.0 / (double)(S > 0 ? S : 1);
  const int64_t BT = a.B * a.T;
  const bool want_grad = a.grad != nullptr;
  const bool zero_masked = want_grad && !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS);
  const uint64_t keep = l2_evict_last(), stream_out = l2_evict_first();

  for (;;) {
    if (threadIdx.x == 0) s_row = (long long)atomicAdd(&a.hdr->row_counter, 1ull);
    __syncthreads();
    const int64_t row = s_row;
    __syncthreads();
    if (row >= BT) break;
    T* grow = want_grad ? reinterpret_cast<T*>(a.grad) + row * a.V : nullptr;

    if (!a.mask[row]) {
      if (threadIdx.x == 0 && a.logps_out) a.logps_out[row] = 0.f;
      if (zero_masked) zero_row<T>(grow, a.V, stream_out);
      continue;
    }
    const int64_t act = a.actions[row];
    if (act < 0 || act >= a.V) {
      if (threadIdx.x == 0) {
        atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_ACTION_RANGE);
        a.slot_p[row] = NAN;
        a.slot_k[row] = NAN;
        if (a.logps_out) a.logps_out[row] = NAN;
      }
      if (zero_masked) zero_row<T>(grow, a.V, stream_out);
      continue;
    }
    const T* x = reinterpret_cast<const T*>(a.policy) + row * a.V;
    const T* y = reinterpret_cast<const T*>(a.ref) + row * a.V;
    const int64_t b = row / a.T;
    float xa = 0.f, ya = 0.f, o = 0.f;
    double Ab = 0.0, c = 0.0;
    if (threadIdx.x == 0) {
      xa = Storage<T>::load1(x + act);
      ya = Storage<T>::load1(y + act);
      o = __ldg(a.old + row);
      Ab = a.A[b];
      c = a.reduction == GRPO_TOKEN_MEAN ? c_tok : inv_S / (double)a.L[b];
    }

    // sweep 1: identical code for both rows, so equal rows give equal results
    OnlineLse sp, sr;
    sp.init();
    sr.init();
    lse_fast<T>(x, a.V, sp, want_grad ? keep : stream_out);
    lse_fast<T>(y, a.V, sr, stream_out);
    float Mp, Mr;
    double Zp = 0.0, Zr = 0.0;
    combine_lse(sp, sr, s_f, s_d, Mp, Mr, Zp, Zr);
    if (warp == 0) {
      const double bp = (double)__fmul_rn(Mp, kLog2e) * kLn2;
      const double br = (double)__fmul_rn(Mr, kLog2e) * kLn2;
      Ab = __shfl_sync(0xFFFFFFFFu, Ab, 0);
      c = __shfl_sync(0xFFFFFFFFu, c, 0);
      RowScalars rs = finish_row(a, bp, Zp, br, Zr, xa, ya, o, Ab, c, want_grad);
      if (threadIdx.x == 0) s_rs = rs;
    }
    __syncthreads();

    if (s_rs.precise) {  // block-uniform
      const double zp = sum_exp_precise<T>(x, a.V, Mp, s_thi, s_tlo, a.tab, s_d);
      const double zr = sum_exp_precise<T>(y, a.V, Mr, s_thi, s_tlo, a.tab, s_d);
      if (warp == 0) {
        Ab = __shfl_sync(0xFFFFFFFFu, Ab, 0);
        c = __shfl_sync(0xFFFFFFFFu, c, 0);
        RowScalars rs = finish_row(a, (double)Mp, zp, (double)Mr, zr, xa, ya, o, Ab, c, want_grad);
        rs.precise = 1;
        if (threadIdx.x == 0) s_rs = rs;
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      a.slot_p[row] = s_rs.p;
      a.slot_k[row] = s_rs.k;
      if (a.logps_out) a.logps_out[row] = (float)s_rs.logp;
    }
    if (want_grad) {
      const RowScalars rs = s_rs;
      grad_sweep<T>(x, grow, a.V, act, rs, stream_out, stream_out);
    }
    __syncthreads();  // s_rs is rewritten by the next row
  }
}

cudaError_t launch_rows(const RowArgs& a, grpo_dtype_t dt, const grpo_profile_t* prof,
                        cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  const void* fn = dt == GRPO_F32 ? (const void*)rows_kernel<float>
                   : dt == GRPO_BF16 ? (const void*)rows_kernel<__nv_bfloat16>
                                     : (const void*)rows_kernel<__half>;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRowThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)sms * per_sm;
  const int64_t rows = a.B * a.T;
  if (grid > rows) grid = rows;
  if (grid < 1) return cudaSuccess;
  if (prof && prof->start) cudaEventRecord((cudaEvent_t)prof->start, s);
  switch (dt) {
    case GRPO_F32: rows_kernel<float><<<(unsigned)grid, kRowThreads, 0, s>>>(a); break;
    case GRPO_BF16: rows_kernel<__nv_bfloat16><<<(unsigned)grid, kRowThreads, 0, s>>>(a); break;
    default: rows_kernel<__half><<<(unsigned)grid, kRowThreads, 0, s>>>(a); break;
  }
  e = cudaGetLastError();
  if (prof && prof->stop) cudaEventRecord((cudaEvent_t)prof->stop, s);
  return e;
}

}  // namespace grpo
