// grpo_rows.cu -- the fused forward + backward over vocabulary rows.
//
// Persistent CTAs (kRowThreads threads, kRowBlocksPerSM per SM) claim token
// rows from a device counter, one row per CTA at a time (the next row is
// claimed while the current one is processed), in row-major or, where that
// measured faster, token-major order (see the launcher).  For an active row
// (completion_mask != 0):
//   sweep 1   one streaming read of the policy and reference rows, both in
//             flight together, each reduced to (max, sum exp) by a per-thread
//             online normaliser and a fixed-order block combine in float-float
//             arithmetic (RL-Kernel "GRPO Loss" intro: the ratio and KL come
//             from logits through an online softmax; grpo.cpp README "CUDA":
//             carry the row maximum and normaliser together);
//   finish    one thread, fp32 / float-float: logp, ref_logp, ratio, clipped
//             surrogate, k3 KL, token weight and w = dL/dlogp (RL-Kernel
//             "Accuracy"; dockyard_rl "One loss, many algorithms",
//             "Reference-KL penalty");
//   sweep 2   the policy row is read again, back to front (the lines sweep 1
//             read last are the likeliest L2 hits), and
//             dL/dx_v = w (1[v=a] - softmax_v) is written into the gradient
//             buffer (grpo.cpp README "CUDA": the fused kernel writes the full
//             logits gradient, in place if asked).
// A masked row is never read: its gradient is written as zeros (or left alone
// under GRPO_SKIP_MASKED_GRAD_ROWS).
//
// Precision.  The fast normaliser (MUFU 2^x, fp32 Kahan sums, compensated
// warp and block sums) has a relative error below 2^-19.  When the gradient
// is stored in fp32 and a row's gradient is sensitive enough that this error
// could break the one-ulp bar (see kFastErrBound / kTau), the row is refined:
// the normaliser of the policy and/or reference row is recomputed with a
// float-float exponential and float-float sums, the row is finished in
// double, and gradient elements above 2^-12 are evaluated in double.  bf16 /
// f16 gradients never need it.
//
// Per-token policy and KL terms go to [B,T] double slots; the fixed-order
// reduction over them is in grpo_reduce.cu.
#include "grpo_rows_common.cuh"

namespace grpo {

// Online normaliser over the elements [e0, e1), element by element.
template <typename T>
__device__ __forceinline__ void lse_elements(const T* row, int64_t e0, int64_t e1, OnlineLse& st) {
  constexpr int VEC = Storage<T>::kVec;
  for (int64_t v = e0 + threadIdx.x; v < e1; v += blockDim.x) {
    float f[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) f[j] = -INFINITY;
    f[0] = Storage<T>::load1(row + v);
    st.update<VEC>(f);
  }
}

// Online normaliser of one row over its 16-byte vectors (kUnroll in flight
// per thread) plus its unaligned head / tail scalars.
template <typename T>
__device__ __forceinline__ void lse_row(const T* row, int64_t V, OnlineLse& st, uint64_t pol,
                                        uint4* keep) {
  constexpr int VEC = Storage<T>::kVec;
  const Geom<T> g(row, V);
  const int64_t nsm = keep ? (g.nvec < kPolicySmemVecs ? g.nvec : kPolicySmemVecs) : 0;
  lse_elements<T>(row, 0, g.head, st);
  lse_elements<T>(row, g.t0, V, st);
  const uint4* vb = reinterpret_cast<const uint4*>(row + g.head);
  const int64_t stride = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (kUnroll - 1) * stride < g.nvec; k += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_hint(vb + k + u * stride, pol);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (k + u * stride < nsm) keep[k + u * stride] = v[u];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[VEC];
      Storage<T>::unpack(v[u], f);
      st.update<VEC>(f);
    }
  }
  for (; k < g.nvec; k += stride) {
    float f[VEC];
    const uint4 v = ld_hint(vb + k, pol);
    if (k < nsm) keep[k] = v;
    Storage<T>::unpack(v, f);
    st.update<VEC>(f);
  }
}

// ---------------------------------------------------------------- sweep 1
// Normalisers of the policy row x and the reference row y.  When both rows
// have the same 16-byte phase their vectors stream in one loop (both in
// flight together), and each thread visits the same positions of both rows in
// the same order: equal rows give bit-identical normalisers, so KL is exactly
// 0 when ref == policy.  Rows of different phases are swept one after the
// other.
//
// With `keep`, the first kPolicySmemVecs policy vectors go to shared memory
// and, when tmem_vecs > 0 and the row is long enough for every thread to
// reach them in the unrolled loop, the next tmem_vecs per thread to tensor
// memory at `tb` (this thread's lane and column base).  Returns the vectors
// per thread kept in tensor memory (0 or tmem_vecs; block-uniform).
template <typename T>
__device__ __forceinline__ int lse_pair(const T* x, const T* y, int64_t V, OnlineLse& sx,
                                        OnlineLse& sy, uint64_t pol_x, uint64_t pol_y,
                                        uint4* keep, uint32_t tb, int tmem_vecs) {
  constexpr int VEC = Storage<T>::kVec;
  const Geom<T> gx(x, V), gy(y, V);
  if (gy.head != gx.head) {
    lse_row<T>(x, V, sx, pol_x, keep);
    lse_row<T>(y, V, sy, pol_y, nullptr);
    return 0;
  }
  const int64_t nsm = keep ? (gx.nvec < kPolicySmemVecs ? gx.nvec : kPolicySmemVecs) : 0;
  constexpr int U = kPairUnroll;
  const int tmv =
      (keep && tmem_vecs > 0 && gx.nvec >= (int64_t)kRowThreads * (kSmemJ + tmem_vecs + U))
          ? tmem_vecs
          : 0;
  // with the tensor-memory slice, the kept vectors are read evict-first: only
  // the rest of the row is wanted in L2 for sweep 2 (on shorter rows, whose
  // whole policy slice stays in L2 anyway, the plain policy measured faster)
  const int64_t nkept = tmv ? nsm + (int64_t)kRowThreads * tmv : 0;
  // head / tail scalars, as one padded vector per thread
  const bool h = (int)threadIdx.x < gx.head;
  const bool t = (int)threadIdx.x < gx.tail;
  if (h || t) {
    float fx[VEC], fy[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) fx[j] = fy[j] = -INFINITY;
    if (h) {
      fx[0] = Storage<T>::load1(x + threadIdx.x);
      fy[0] = Storage<T>::load1(y + threadIdx.x);
    }
    if (t) {
      fx[1] = Storage<T>::load1(x + gx.t0 + threadIdx.x);
      fy[1] = Storage<T>::load1(y + gx.t0 + threadIdx.x);
    }
    sx.update<VEC>(fx);
    sy.update<VEC>(fy);
  }
  const uint4* xv = reinterpret_cast<const uint4*>(x + gx.head);
  const uint4* yv = reinterpret_cast<const uint4*>(y + gx.head);
  const int64_t stride = blockDim.x;
  int64_t k = threadIdx.x;
  // every thread runs the unrolled loop at least kSmemJ + tmv + 1 steps of
  // `stride` deep (the length test above), so the tensor-memory stores, whose
  // condition depends on the step only, are taken by whole warps
  for (; k + (U - 1) * stride < gx.nvec; k += U * stride) {
    uint4 vx[U], vy[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      vx[u] = ld_hint(xv + k + u * stride, k + u * stride < nkept ? pol_y : pol_x);
      vy[u] = ld_hint(yv + k + u * stride, pol_y);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t q = k + u * stride;
      if (q < nsm)
        keep[q] = vx[u];
      else if (q < nkept)
        tmem_st4(tb + 4u * (uint32_t)((q - nsm) / kRowThreads), vx[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float f[VEC];
      Storage<T>::unpack(vx[u], f);
      sx.update<VEC>(f);
      Storage<T>::unpack(vy[u], f);
      sy.update<VEC>(f);
    }
  }
  for (; k < gx.nvec; k += stride) {
    float f[VEC];
    const uint4 v = ld_hint(xv + k, pol_x);
    if (k < nsm) keep[k] = v;
    Storage<T>::unpack(v, f);
    sx.update<VEC>(f);
    Storage<T>::unpack(ld_hint(yv + k, pol_y), f);
    sy.update<VEC>(f);
  }
  if (tmv) tmem_wait_st();  // this thread's stores land before its sweep-2 loads
  return tmv;
}

// ------------------------------------------------- precise normaliser sweep
// sum_v exp(x_v - M) with x_v - M exact as a float pair, float-float
// exponentials (exp_ff) and float-float per-thread sums; every thread gets
// the block total (double).
__device__ __forceinline__ void ff_accumulate(FF& acc, float x, float M, const float* thi,
                                              const float* tlo, const ExpTable& tb) {
  const FF t = two_sum(x, -M);
  const FF e = exp_ff(t.hi, t.lo, thi, tlo, tb);
  const FF s = two_sum(acc.hi, e.hi);
  acc.hi = s.hi;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, e.lo));
}

template <typename T>
__device__ double sum_exp_precise(const T* row, int64_t V, float M, const float* thi,
                                  const float* tlo, const ExpTable& tb, double* ds) {
  constexpr int VEC = Storage<T>::kVec;
  const Geom<T> g(row, V);
  FF acc = {0.f, 0.f};
  for (int64_t v = threadIdx.x; v < g.head; v += blockDim.x)
    ff_accumulate(acc, Storage<T>::load1(row + v), M, thi, tlo, tb);
  for (int64_t v = g.t0 + threadIdx.x; v < V; v += blockDim.x)
    ff_accumulate(acc, Storage<T>::load1(row + v), M, thi, tlo, tb);
  const uint4* vb = reinterpret_cast<const uint4*>(row + g.head);
  const int64_t stride = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (kUnroll - 1) * stride < g.nvec; k += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(vb + k + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[VEC];
      Storage<T>::unpack(v[u], f);
#pragma unroll
      for (int j = 0; j < VEC; ++j) ff_accumulate(acc, f[j], M, thi, tlo, tb);
    }
  }
  for (; k < g.nvec; k += stride) {
    float f[VEC];
    Storage<T>::unpack(__ldg(vb + k), f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) ff_accumulate(acc, f[j], M, thi, tlo, tb);
  }
  double z[1] = {(double)acc.hi + (double)acc.lo};
  block_sum<double, 1>(z, ds);
  return z[0];
}

// ---------------------------------------------------------------- sweep 2
// dL/dx = w (onehot - softmax) over a row, vectors visited back to front when
// kReverseSweep2: the lines sweep 1 read last are read first.  The action
// element is patched once per vector, outside the element loop.
template <typename T, bool kPrecise>
__device__ void grad_row(const T* x, T* g, int64_t V, int64_t act, const RowScalars& rs,
                         uint64_t pol_in, uint64_t pol_out, const uint4* kept, uint32_t tb = 0,
                         int tmv = 0) {
  constexpr int VEC = Storage<T>::kVec;
  const bool same_phase = (((uintptr_t)x ^ (uintptr_t)g) & 15) == 0;
  if (!same_phase) {  // differently aligned buffers: element by element
    for (int64_t v = threadIdx.x; v < V; v += blockDim.x)
      Storage<T>::store1(g + v, grad_at<kPrecise>(Storage<T>::load1(x + v), v, rs, act));
    return;
  }
  const Geom<T> gm(x, V);
  if ((int)threadIdx.x < gm.head) {
    const int64_t v = threadIdx.x;
    Storage<T>::store1(g + v, grad_at<kPrecise>(Storage<T>::load1(x + v), v, rs, act));
  }
  if ((int)threadIdx.x < gm.tail) {
    const int64_t v = gm.t0 + threadIdx.x;
    Storage<T>::store1(g + v, grad_at<kPrecise>(Storage<T>::load1(x + v), v, rs, act));
  }
  const uint4* xv = reinterpret_cast<const uint4*>(x + gm.head);
  uint4* gv = reinterpret_cast<uint4*>(g + gm.head);
  const int64_t stride = blockDim.x;
  const int64_t n = gm.nvec;
  // the vector holding the action element, and its lane (or none)
  const int64_t arel = act - gm.head;
  const int64_t aq = (arel >= 0 && arel < n * VEC) ? arel / VEC : -1;
  const int alane = (int)(arel - aq * VEC);
  auto emit = [&](const uint4& in, int64_t q) {
    float f[VEC];
    Storage<T>::unpack(in, f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) f[j] = grad_elem<kPrecise>(f[j], rs);
    if (q == aq) {
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (j == alane) f[j] = rs.ga;
    }
    st_hint(gv + q, Storage<T>::pack(f), pol_out);
  };
  // vectors [0, nsm) were kept in shared memory by sweep 1, the next tmv per
  // thread in tensor memory; the rest, in the sweep order, come from global
  // memory (mostly L2)
  const int64_t nsm = kept ? (n < kPolicySmemVecs ? n : kPolicySmemVecs) : 0;
  const int64_t ntm = (int64_t)kRowThreads * tmv;
  const int64_t ng = n - nsm - ntm;
  auto atg = [&](int64_t k) -> int64_t { return kReverseSweep2 ? n - 1 - k : nsm + ntm + k; };
  constexpr int U = kGradUnroll;
  int64_t k = threadIdx.x;
  for (; k + (U - 1) * stride < ng; k += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_hint(xv + atg(k + u * stride), pol_in);
#pragma unroll
    for (int u = 0; u < U; ++u) emit(v[u], atg(k + u * stride));
  }
  for (; k < ng; k += stride) emit(ld_hint(xv + atg(k), pol_in), atg(k));
  if (tmv) {
    __syncwarp();  // the tensor-memory loads are warp-collective
    for (int j = 0; j < tmv; j += 2) {
      uint4 v[2];
      tmem_ld8(tb + 4u * (uint32_t)j, v);
#pragma unroll
      for (int i = 0; i < 2; ++i) emit(v[i], nsm + threadIdx.x + (int64_t)kRowThreads * (j + i));
    }
  }
  for (int64_t q = threadIdx.x; q < nsm; q += stride) emit(kept[q], q);
}

// zeros over a gradient row
template <typename T>
__device__ void zero_row(T* g, int64_t V, uint64_t pol) {
  const Geom<T> gm(g, V);
  if ((int)threadIdx.x < gm.head) Storage<T>::store1(g + threadIdx.x, 0.f);
  if ((int)threadIdx.x < gm.tail) Storage<T>::store1(g + gm.t0 + threadIdx.x, 0.f);
  uint4* gv = reinterpret_cast<uint4*>(g + gm.head);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = threadIdx.x; k < gm.nvec; k += blockDim.x) st_hint(gv + k, z, pol);
}

// rows_kernel's claim order, a bit of the kernel's own copy of the flags
// (set by its launcher; callers' flags never hold it): token-major claims,
// slot t of every sequence before slot t + 1.
static constexpr unsigned kClaimTokenMajor = 0x20000000u;

// The row a claim stands for: the claimed index itself, or, token-major,
// slot claimed / B of sequence claimed % B; -1 past the last row.
__device__ __forceinline__ long long claimed_row(const RowArgs& a, long long claimed) {
  const long long BT = a.B * a.T;
  if (claimed >= BT) return -1;
  return (a.flags & kClaimTokenMajor) ? (claimed % a.B) * a.T + claimed / a.B : claimed;
}

// ------------------------------------------------------------------ kernel
// kTmem: the instantiation that may keep the tensor-memory slice.  16-bit
// rows too short to reach it take the other one, which holds no
// tensor-memory code at all (a kernel that may allocate tensor memory
// measured 1.3 % slower on the 64 KB rows of the fused workload, where the
// slice is never used).
template <typename T, bool kTmem>
__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) rows_kernel(const RowArgs a) {
  extern __shared__ __align__(16) uint4 s_keep[];  // kPolicySmemVecs vectors
  __shared__ float s_f[64];
  __shared__ FF s_zs[64];
  __shared__ double s_d[64];
  __shared__ float s_thi[64], s_tlo[64];
  __shared__ RowScalars s_rs;
  __shared__ float s_M[2];
  __shared__ long long s_NS[2];
  __shared__ long long s_next;
  __shared__ uint32_t s_tmem, s_tb_cols;
  __shared__ double s_c[2];
  __shared__ unsigned s_clip[3];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 64) {
    s_thi[threadIdx.x] = a.tab.hi[threadIdx.x];
    s_tlo[threadIdx.x] = a.tab.lo[threadIdx.x];
  }
  // tensor memory for the second kept slice (block-uniform; released below,
  // after the last row, on every path)
  const int tcols = kTmem && a.grad != nullptr ? a.tmem_cols : 0;
  if (kTmem && warp == 0) {
    if (tcols) tmem_alloc(&s_tmem, (uint32_t)tcols);
    tmem_relinquish();
  }
  if (tcols) tmem_fence_before_sync();
  // N = active tokens, S = live sequences of the whole batch (counted by prep,
  // or given by a shard call), read here once
  if (threadIdx.x == 0) {
    s_NS[0] = a.NS[0];
    s_NS[1] = a.NS[1];
    s_next = claimed_row(a, (long long)atomicAdd(&a.hdr->row_counter, 1ull));
    s_tb_cols = (uint32_t)(tcols / 2);
  }
  __syncthreads();
  if (tcols) tmem_fence_after_sync();
  // thread 0's per-CTA values live in shared memory: every thread holds the
  // kernel's registers, and the sweeps need them all
  if (threadIdx.x == 0) {
    const long long N = s_NS[0], S = s_NS[1];
    // token weight: 1/max(N,1) (token mean), 1/(max(S,1) L_i) (sequence
    // mean) or 1/C (fixed constant)
    s_c[0] = a.reduction == GRPO_FIXED_CONSTANT ? 1.0 / (double)a.norm_c
                                                : 1.0 / (double)(N > 0 ? N : 1);
    s_c[1] = 1.0 / (double)(S > 0 ? S : 1);
    s_clip[0] = s_clip[1] = s_clip[2] = 0u;  // this CTA's clipped rows
  }
  const bool want_grad = a.grad != nullptr;
  const bool zero_masked = want_grad && !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS);

  int64_t row = s_next;
  while (row >= 0) {
    // L2 policies, made per row (one instruction each) rather than held
    const uint64_t keep = l2_evict_last(), stream = l2_evict_first();
    long long claim = 0;  // the next row, claimed while this one is processed
    if (threadIdx.x == 0) claim = (long long)atomicAdd(&a.hdr->row_counter, 1ull);
    const T* x = reinterpret_cast<const T*>(a.policy) + row * a.V;
    const T* y = reinterpret_cast<const T*>(a.ref) + row * a.V;
    T* grow = want_grad ? reinterpret_cast<T*>(a.grad) + row * a.V : nullptr;
    const bool active = a.mask[row] != 0;
    const int64_t act = active ? a.actions[row] : 0;  // masked storage is not read
    if (!active) {
      if (threadIdx.x == 0 && a.logps_out) a.logps_out[row] = 0.f;
      if (zero_masked) zero_row<T>(grow, a.V, stream);
    } else if (act < 0 || act >= a.V) {
      if (threadIdx.x == 0) {
        atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_ACTION_RANGE);
        a.slot_p[row] = NAN;
        a.slot_k[row] = NAN;
        if (a.logps_out) a.logps_out[row] = NAN;
      }
      if (zero_masked) zero_row<T>(grow, a.V, stream);
    } else {
      const int64_t b = row / a.T;
      float xa = 0.f, ya = 0.f, o = 0.f;
      double Ab = 0.0, c = 0.0;
      if (threadIdx.x == 0) {
        xa = Storage<T>::load1(x + act);
        ya = Storage<T>::load1(y + act);
        o = __ldg(a.old + row);
        Ab = a.A[b];
        c = a.reduction == GRPO_SEQUENCE_MEAN ? s_c[1] / (double)a.L[b] : s_c[0];
      }

      // sweep 1, the block combine, the fast finish
      OnlineLse sp, sr;
      sp.init();
      sr.init();
      const uint32_t tb = tmem_thread_base(s_tmem, s_tb_cols);
      const int tmv = lse_pair<T>(x, y, a.V, sp, sr, want_grad ? keep : stream, stream,
                                  want_grad ? s_keep : nullptr, tb,
                                  kTmem ? (int)s_tb_cols / 4 : 0);
      float Mp, Mr;
      FF Zp = {0.f, 0.f}, Zr = {0.f, 0.f};
      combine_ff(sp, sr, s_f, s_zs, Mp, Mr, Zp, Zr);
      if (threadIdx.x == 0) {
        s_rs = finish_fast(a, __fmul_rn(Mp, kLog2e), Zp, __fmul_rn(Mr, kLog2e), Zr, xa, ya, o,
                           (float)Ab, (float)c, want_grad);
        s_M[0] = Mp;
        s_M[1] = Mr;
      }
      __syncthreads();

      if (s_rs.precise) {  // block-uniform
        const int which = s_rs.precise;
        const float RMp = s_M[0], RMr = s_M[1];
        double zp = 0.0, zr = 0.0;
        if (which & 1) zp = sum_exp_precise<T>(x, a.V, RMp, s_thi, s_tlo, a.tab, s_d);
        if (which & 2) zr = sum_exp_precise<T>(y, a.V, RMr, s_thi, s_tlo, a.tab, s_d);
        if (warp == 0) {
          // a row that is not refined keeps its fast sum, taken to base M:
          // sum_v exp(x_v - M) = 2^(fl(M log2e) - M log2e) Z
          if (!(which & 1))
            zp = ((double)__shfl_sync(0xFFFFFFFFu, Zp.hi, 0) +
                  (double)__shfl_sync(0xFFFFFFFFu, Zp.lo, 0)) *
                 exp2((double)__fmul_rn(RMp, kLog2e) - (double)RMp * 1.4426950408889634);
          if (!(which & 2))
            zr = ((double)__shfl_sync(0xFFFFFFFFu, Zr.hi, 0) +
                  (double)__shfl_sync(0xFFFFFFFFu, Zr.lo, 0)) *
                 exp2((double)__fmul_rn(RMr, kLog2e) - (double)RMr * 1.4426950408889634);
          Ab = __shfl_sync(0xFFFFFFFFu, Ab, 0);
          c = __shfl_sync(0xFFFFFFFFu, c, 0);
          const RowScalars rs =
              finish_precise(a, (double)RMp, zp, (double)RMr, zr, xa, ya, o, Ab, c);
          if (lane == 0) s_rs = rs;
        }
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        a.slot_p[row] = s_rs.q;
        a.slot_k[row] = s_rs.k;
        if (a.logps_out) a.logps_out[row] = (float)s_rs.logp;
        if (s_rs.clip) ++s_clip[s_rs.clip - 1];
      }
      if (want_grad) {
        const RowScalars rs = s_rs;
        const uint32_t tb = tmem_thread_base(s_tmem, s_tb_cols);
        if (rs.precise)
          grad_row<T, true>(x, grow, a.V, act, rs, stream, stream, s_keep, tb, tmv);
        else
          grad_row<T, false>(x, grow, a.V, act, rs, stream, stream, s_keep, tb, tmv);
      }
    }
    __syncthreads();  // everyone is done with s_rs / s_next of this row
    if (threadIdx.x == 0) s_next = claimed_row(a, claim);
    __syncthreads();
    row = s_next;
  }
  if (threadIdx.x == 0) {
    const unsigned n_clip[3] = {s_clip[0], s_clip[1], s_clip[2]};
    add_clip_counts(a.hdr, n_clip);
  }
  if (kTmem && s_tb_cols) {  // every thread's tensor-memory loads were waited for
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(s_tmem, 2u * s_tb_cols);
  }
}

// ------------------------------------------------------------------ GSPO
// Sequence-level ratios need every token's log-prob of a sequence before any
// gradient of it, so the fused row pass splits in two around the
// per-sequence step in grpo_reduce.cu:
//   gspo_sweep1_kernel  sweep 1 and the finish of every active row: logp and
//                       d = ref_logp - logp into the two token slots (both
//                       rows refined to double when the gradient is fp32);
//   (reduce)            rho_i, the per-token terms and w into the slots;
//   gspo_sweep2_kernel  sweep 2 of every row from (logp, w): the gradient,
//                       zeros on masked rows.
// Rows are claimed from two device counters, as in rows_kernel: sweep 1 from
// the first row on, reading the policy rows evict-last, sweep 2 from the last
// claim back (token-major on long 16-bit rows: see the launcher), so that its
// first rows include the ones L2 still holds from sweep 1 (the second read of
// the policy is the method's own: rho_i needs every token of the sequence
// before any gradient of it).
template <typename T>
__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) gspo_sweep1_kernel(const RowArgs a) {
  __shared__ float s_f[64];
  __shared__ FF s_zs[64];
  __shared__ double s_d[64];
  __shared__ float s_thi[64], s_tlo[64];
  __shared__ RowScalars s_rs;
  __shared__ float s_M[2];
  __shared__ long long s_next;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 64) {
    s_thi[threadIdx.x] = a.tab.hi[threadIdx.x];
    s_tlo[threadIdx.x] = a.tab.lo[threadIdx.x];
  }
  if (threadIdx.x == 0) s_next = (long long)atomicAdd(&a.hdr->row_counter, 1ull);
  __syncthreads();
  const int64_t BT = a.B * a.T;
  const bool refine = a.precise_ok && a.grad != nullptr;
  const uint64_t stream = l2_evict_first(), keep = l2_evict_last();
  int64_t row = s_next;
  while (row < BT) {
    long long claim = 0;
    if (threadIdx.x == 0) claim = (long long)atomicAdd(&a.hdr->row_counter, 1ull);
    const T* x = reinterpret_cast<const T*>(a.policy) + row * a.V;
    const T* y = reinterpret_cast<const T*>(a.ref) + row * a.V;
    const bool active = a.mask[row] != 0;
    const int64_t act = active ? a.actions[row] : 0;
    if (!active) {
      if (threadIdx.x == 0 && a.logps_out) a.logps_out[row] = 0.f;
    } else if (act < 0 || act >= a.V) {
      if (threadIdx.x == 0) {
        atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_ACTION_RANGE);
        a.slot_p[row] = NAN;
        a.slot_k[row] = NAN;
        if (a.logps_out) a.logps_out[row] = NAN;
      }
    } else {
      float xa = 0.f, ya = 0.f, o = 0.f;
      if (threadIdx.x == 0) {
        xa = Storage<T>::load1(x + act);
        ya = Storage<T>::load1(y + act);
        o = __ldg(a.old + row);
      }
      OnlineLse sp, sr;
      sp.init();
      sr.init();
      lse_pair<T>(x, y, a.V, sp, sr, keep, stream, nullptr, 0u, 0);
      float Mp, Mr;
      FF Zp = {0.f, 0.f}, Zr = {0.f, 0.f};
      combine_ff(sp, sr, s_f, s_zs, Mp, Mr, Zp, Zr);
      if (threadIdx.x == 0) {
        s_rs = finish_fast(a, __fmul_rn(Mp, kLog2e), Zp, __fmul_rn(Mr, kLog2e), Zr, xa, ya, o,
                           0.f, 0.f, false);
        s_M[0] = Mp;
        s_M[1] = Mr;
      }
      __syncthreads();
      if (refine) {  // block-uniform: both rows in double (the ratio is a sequence mean)
        const float RMp = s_M[0], RMr = s_M[1];
        const double zp = sum_exp_precise<T>(x, a.V, RMp, s_thi, s_tlo, a.tab, s_d);
        const double zr = sum_exp_precise<T>(y, a.V, RMr, s_thi, s_tlo, a.tab, s_d);
        if (warp == 0) {
          const RowScalars rs = finish_precise(a, (double)RMp, zp, (double)RMr, zr, xa, ya, o,
                                               0.0, 0.0);
          if (lane == 0) s_rs = rs;
        }
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        a.slot_p[row] = s_rs.logp;
        a.slot_k[row] = s_rs.dlr;
        if (a.logps_out) a.logps_out[row] = (float)s_rs.logp;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) s_next = claim;
    __syncthreads();
    row = s_next;
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) gspo_sweep2_kernel(const RowArgs a) {
  __shared__ RowScalars s_rs;
  __shared__ long long s_next;
  if (threadIdx.x == 0) s_next = (long long)atomicAdd(&a.hdr->row_counter2, 1ull);
  __syncthreads();
  const int64_t BT = a.B * a.T;
  const bool zero_masked = !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS);
  const uint64_t stream = l2_evict_first();
  int64_t k = s_next;  // claims count from the last claim back
  while (k < BT) {
    const int64_t row = claimed_row(a, BT - 1 - k);
    long long claim = 0;
    if (threadIdx.x == 0) claim = (long long)atomicAdd(&a.hdr->row_counter2, 1ull);
    const T* x = reinterpret_cast<const T*>(a.policy) + row * a.V;
    T* grow = reinterpret_cast<T*>(a.grad) + row * a.V;
    const bool active = a.mask[row] != 0;
    const int64_t act = active ? a.actions[row] : 0;
    if (!active || act < 0 || act >= a.V) {
      if (zero_masked) zero_row<T>(grow, a.V, stream);
    } else {
      if (threadIdx.x == 0) {  // the row's scalars from logp and w
        const double lp = a.slot_p[row], w = a.slot_k[row];
        RowScalars rs;
        rs.lse_p = (double)Storage<T>::load1(x + act) - lp;
        rs.w = w;
        rs.wneg = (float)(-w);
        rs.LL = (float)(rs.lse_p * (double)kLog2e);
        rs.ga = (float)(-w * expm1(lp));
        rs.q = rs.k = 0.0;
        rs.logp = lp;
        rs.dlr = 0.0;
        rs.precise = a.precise_ok;
        rs.clip = 0;
        s_rs = rs;
      }
      __syncthreads();
      const RowScalars rs = s_rs;
      if (rs.precise)
        grad_row<T, true>(x, grow, a.V, act, rs, stream, stream, nullptr);
      else
        grad_row<T, false>(x, grow, a.V, act, rs, stream, stream, nullptr);
    }
    __syncthreads();
    if (threadIdx.x == 0) s_next = claim;
    __syncthreads();
    k = s_next;
  }
}

template <typename T>
static cudaError_t launch_gspo_t(const RowArgs& a, int phase, const grpo_profile_t* prof,
                                 cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int64_t grid = (int64_t)sms * kRowBlocksPerSM;
  const int64_t rows = a.B * a.T;
  if (grid > rows) grid = rows;
  if (grid < 1) return cudaSuccess;
  if (phase == 1) {
    if (prof && prof->start) cudaEventRecord((cudaEvent_t)prof->start, s);
    gspo_sweep1_kernel<T><<<(unsigned)grid, kRowThreads, 0, s>>>(a);
  } else {
    // sweep 2 claims token-major on long 16-bit rows whose masked rows are
    // zero-filled, as rows_kernel does (large-vocabulary rows: the three
    // GSPO kernels 3.205 against 3.245 ms; token-major in sweep 1 as well,
    // 3.226 ms); sweep 1 claims row-major
    RowArgs ka = a;
    const bool long_rows = a.V * (int64_t)sizeof(T) >=
                           (int64_t)16 * kRowThreads * (kSmemJ + kTmemVecs + kPairUnroll);
    if (sizeof(T) == 2 && long_rows && !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS))
      ka.flags |= kClaimTokenMajor;
    gspo_sweep2_kernel<T><<<(unsigned)grid, kRowThreads, 0, s>>>(ka);
  }
  e = cudaGetLastError();
  if (phase == 2 && prof && prof->stop) cudaEventRecord((cudaEvent_t)prof->stop, s);
  return e;
}

cudaError_t launch_gspo_rows(const RowArgs& a, grpo_dtype_t dt, int phase,
                             const grpo_profile_t* prof, cudaStream_t s) {
  switch (dt) {
    case GRPO_F32: return launch_gspo_t<float>(a, phase, prof, s);
    case GRPO_BF16: return launch_gspo_t<__nv_bfloat16>(a, phase, prof, s);
    default: return launch_gspo_t<__half>(a, phase, prof, s);
  }
}

// ------------------------------------------------------- vocab-parallel
// The gradient of a rank's vocabulary slice [v_begin, v_begin + V) of every
// row (RowArgs.V is the slice width; policy / grad are [rows, V]) from the
// row's logsumexp and w = dL/dlogp (lse_w[row], lse_w[rows + row]):
// dL/dx_v = w (1[v = a] - exp(x_v - lse)); zeros on masked rows.
template <typename T>
__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) vocab_grad_kernel(
    const RowArgs a, int64_t v_begin, const double* lse_w) {
  __shared__ RowScalars s_rs;
  const int64_t BT = a.B * a.T;
  const bool zero_masked = !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS);
  const uint64_t stream = l2_evict_first();
  for (int64_t row = blockIdx.x; row < BT; row += gridDim.x) {
    const T* x = reinterpret_cast<const T*>(a.policy) + row * a.V;
    T* grow = reinterpret_cast<T*>(a.grad) + row * a.V;
    const bool active = a.mask[row] != 0;
    const int64_t act = active ? a.actions[row] - v_begin : -1;  // relative to the slice
    const double lse = active ? lse_w[row] : 0.0;
    if (!active || !(lse == lse)) {  // masked, or a row the merge rejected
      if (zero_masked) zero_row<T>(grow, a.V, stream);
      continue;
    }
    if (threadIdx.x == 0) {
      const double w = lse_w[BT + row];
      RowScalars rs;
      rs.lse_p = lse;
      rs.w = w;
      rs.wneg = (float)(-w);
      rs.LL = (float)(lse * (double)kLog2e);
      rs.ga = (act >= 0 && act < a.V)
                  ? (float)(-w * expm1((double)Storage<T>::load1(x + act) - lse))
                  : 0.f;
      rs.q = rs.k = rs.logp = rs.dlr = 0.0;
      rs.precise = a.precise_ok;
      rs.clip = 0;
      s_rs = rs;
    }
    __syncthreads();
    const RowScalars rs = s_rs;
    if (rs.precise)
      grad_row<T, true>(x, grow, a.V, act, rs, stream, stream, nullptr);
    else
      grad_row<T, false>(x, grow, a.V, act, rs, stream, stream, nullptr);
    __syncthreads();
  }
}

template <typename T>
static cudaError_t launch_vocab_grad_t(const RowArgs& a, int64_t v_begin, const double* lse_w,
                                       cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int64_t grid = (int64_t)sms * kRowBlocksPerSM;
  if (grid > a.B * a.T) grid = a.B * a.T;
  if (grid < 1) return cudaSuccess;
  vocab_grad_kernel<T><<<(unsigned)grid, kRowThreads, 0, s>>>(a, v_begin, lse_w);
  return cudaGetLastError();
}

cudaError_t launch_vocab_grad(const RowArgs& a, grpo_dtype_t dt, int64_t v_begin,
                              const double* lse_w, cudaStream_t s) {
  switch (dt) {
    case GRPO_F32: return launch_vocab_grad_t<float>(a, v_begin, lse_w, s);
    case GRPO_BF16: return launch_vocab_grad_t<__nv_bfloat16>(a, v_begin, lse_w, s);
    default: return launch_vocab_grad_t<__half>(a, v_begin, lse_w, s);
  }
}

// CTAs of `kernel` resident per SM, from its registers, shared memory and
// threads, and the shared-memory carveout (percent) they need.  The occupancy
// calculator counts a kernel that allocates tensor memory as one CTA per SM;
// the hardware co-schedules such CTAs up to the other limits (their
// allocations then have to fit together, which the launcher checks), so the
// count is taken from the kernel's attributes.
static cudaError_t resident_ctas(const void* kernel, int threads, int dyn_smem, int dev,
                                 int* out, int* carveout) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  int regs_sm = 0, smem_sm = 0, thr_sm = 0, blk_sm = 0, smem_res = 0;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) ||
      (e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) ||
      (e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) ||
      (e = cudaDeviceGetAttribute(&blk_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev)) ||
      (e = cudaDeviceGetAttribute(&smem_res, cudaDevAttrReservedSharedMemoryPerBlock, dev)))
    return e;
  const int warps = (threads + 31) / 32;
  const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in 256s
  int n = regs_sm / (regs_warp * warps > 0 ? regs_warp * warps : 1);
  const int smem = (int)fa.sharedSizeBytes + dyn_smem + smem_res;
  if (smem_sm / smem < n) n = smem_sm / smem;
  if (thr_sm / threads < n) n = thr_sm / threads;
  if (blk_sm < n) n = blk_sm;
  *out = n > 0 ? n : 1;
  const int64_t need = (int64_t)(*out) * smem;
  int pct = (int)((need * 100 + smem_sm - 1) / smem_sm);
  *carveout = pct < 100 ? pct : 100;
  return cudaSuccess;
}

template <typename T, bool kTmem>
static cudaError_t launch_rows_kernel(const RowArgs& a, int tmem_cols, const grpo_profile_t* prof,
                                      cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  e = cudaFuncSetAttribute(rows_kernel<T, kTmem>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kPolicySmemBytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0, carveout = 0;
  e = resident_ctas((const void*)rows_kernel<T, kTmem>, kRowThreads, kPolicySmemBytes, dev,
                    &per_sm, &carveout);
  if (e != cudaSuccess) return e;
  // the shared-memory share of the SM's L1 that those CTAs need, and no more
  // (the largest carveout measured about 9 % slower on the row kernel)
  e = cudaFuncSetAttribute(rows_kernel<T, kTmem>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           carveout);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sms * per_sm;
  const int64_t rows = a.B * a.T;
  if (grid > rows) grid = rows;
  // the resident CTAs of an SM must fit its 512 tensor-memory columns
  // together, or an allocation would wait for another CTA to exit
  RowArgs ka = a;
  ka.tmem_cols = (kTmem && per_sm * tmem_cols <= 512) ? tmem_cols : 0;
  // Claim order.  Prefix masks put a sequence's active rows together, so
  // row-major claims alternate between stretches of active rows (both rows
  // read, the gradient written) and stretches of masked rows (zero fills
  // only); token-major claims (slot t of every sequence, then t + 1) change
  // that mix gradually over the launch.  Measured per launch, token-major
  // against row-major: the large-vocabulary rows (16-bit, tensor-memory
  // slice, masked rows zero-filled) 2.827 against 2.861 ms, with the same
  // DRAM traffic; the 64 KB fused rows 1.393 against 1.384 ms, the 513 KB
  // fp32 rows 5.605 against 5.584 ms, and the masked-row mode (no zero
  // fills) 2.024 against 1.995 ms.  So only the first kind claims
  // token-major.
  if (kTmem && sizeof(T) == 2 && ka.tmem_cols && a.grad &&
      !(a.flags & GRPO_SKIP_MASKED_GRAD_ROWS))
    ka.flags |= kClaimTokenMajor;
  if (prof && prof->start) cudaEventRecord((cudaEvent_t)prof->start, s);
  rows_kernel<T, kTmem><<<(unsigned)grid, kRowThreads, kPolicySmemBytes, s>>>(ka);
  e = cudaGetLastError();
  if (prof && prof->stop) cudaEventRecord((cudaEvent_t)prof->stop, s);
  return e;
}

template <typename T>
static cudaError_t launch_t(const RowArgs& a, const grpo_profile_t* prof, cudaStream_t s) {
  // only rows long enough to reach the tensor-memory slice (and only calls
  // that write a gradient) take the instantiation that allocates it
  const bool long_rows =
      a.V * (int64_t)sizeof(T) >= (int64_t)16 * kRowThreads * (kSmemJ + kTmemVecs + kPairUnroll);
  const bool slice = long_rows && a.grad != nullptr;
  if constexpr (sizeof(T) == 4) {
    // fp32 rows keep one instantiation (the plain one spilled registers)
    return launch_rows_kernel<T, true>(a, slice ? kTmemCols : 0, prof, s);
  } else {
    if (slice) return launch_rows_kernel<T, true>(a, kTmemCols, prof, s);
    return launch_rows_kernel<T, false>(a, 0, prof, s);
  }
}

cudaError_t launch_rows(const RowArgs& a, grpo_dtype_t dt, const grpo_profile_t* prof,
                        cudaStream_t s) {
  switch (dt) {
    case GRPO_F32: return launch_t<float>(a, prof, s);
    case GRPO_BF16: return launch_t<__nv_bfloat16>(a, prof, s);
    default: return launch_t<__half>(a, prof, s);
  }
}

}  // namespace grpo
