// grpo_vocab.cu -- vocabulary-parallel log-probs (tensor parallelism over V).
//
// RL-Kernel "GRPO Loss" page, "Tensor and Data Parallel", step 1: the
// selected log-probs come from a vocab-parallel logprob, so that ratio and KL
// are bit-identical at every tensor-parallel degree.  Here a rank holding the
// vocabulary slice [v_begin, v_begin + Vk) of every row reduces the slice
// chunk by chunk -- fixed chunks of kVChunk vocabulary entries, numbered over
// the whole vocabulary -- to partial normalisers (M_c, Z_c); the ranks'
// partials, concatenated in rank order, are merged in chunk order.  A chunk's
// partial is computed the same way whichever rank holds it (its elements go
// to warp lanes by their index in the chunk, not by their address), so any
// split at chunk boundaries gives the same bits.
//
//   vocab_partials_kernel  one warp per (row, chunk): the chunk's max and
//                          sum of exp(x - max) (fp32 logits: two passes with
//                          a float-float exponential; 16-bit logits: one pass
//                          of online normalisers with MUFU 2^x);
//                          the action logit where the rank owns it
//   vocab_merge_kernel     one thread per row: the chunks folded in order,
//                          logsumexp in double, logp and d = ref_logp - logp
//                          into the token slots for the per-token step
#include "grpo_rows_common.cuh"

namespace grpo {

static constexpr int kVocabWarps = 4;  // measured: 8 warps per CTA 4 % slower
static constexpr int kMergeThreads = 256;

// The elements of run j (16 bytes of storage) of a chunk, -inf beyond n.
template <typename T>
__device__ __forceinline__ void load_run(const T* x, int64_t j, int64_t n, bool vec,
                                         float (&f)[Storage<T>::kVec]) {
  constexpr int R = Storage<T>::kVec;
  const int64_t e0 = j * R;
  if (vec && e0 + R <= n) {
    Storage<T>::unpack(__ldg(reinterpret_cast<const uint4*>(x) + j), f);
    return;
  }
#pragma unroll
  for (int e = 0; e < R; ++e) f[e] = e0 + e < n ? Storage<T>::load1(x + e0 + e) : -INFINITY;
}

// A chunk's partial normaliser, by one warp: runs of 16 bytes of storage go
// to lane (run index mod 32), each lane takes its runs in order; a fixed xor
// tree combines the lanes.  Every lane gets (M, Z), Z = sum exp(x - M).
//
// MUFU path (16-bit logits): one pass, each lane an online normaliser in
// base 2 (its running max m, mL = fl(m log2e), a Kahan sum of
// 2^(x log2e - mL)); the lanes' sums rescaled to the chunk's ML = fl(M log2e)
// and added as float pairs; finally Z = Z_2 2^(ML - M log2e), the residual
// exponent taken exactly with an FMA.
// The lanes' online normalisers of one chunk reduced to the chunk's (M, Z).
__device__ __forceinline__ void finish_partial(const OnlineLse& st, float& M, FF& Z) {
  const float m = warp_max(st.m);
  if (m == -INFINITY) {  // an empty chunk contributes nothing
    M = -INFINITY;
    Z = FF{0.f, 0.f};
    return;
  }
  const float ML = __fmul_rn(m, kLog2e);
  const float z = st.m == -INFINITY ? 0.f : __fmul_rn(__fsub_rn(st.s, st.c),
                                                      ex2_fast(__fsub_rn(st.mL, ML)));
  const FF s = warp_sum_ff(z);
  const FF z2 = FF{__shfl_sync(0xFFFFFFFFu, s.hi, 0), __shfl_sync(0xFFFFFFFFu, s.lo, 0)};
  const float resid = -__fmaf_rn(m, kLog2e, -ML);  // ML - m log2e, exactly
  Z = ff_scale(z2, ex2_fast(resid));
  M = m;
}

// The MUFU path over the same chunk of the policy (x) and reference (y)
// rows at once, kRunsAhead runs of each in flight per lane: the loads run
// ahead of the updates, and each row's normaliser still takes its runs in
// index order, so (M, Z) are the bits one row alone would give.
static constexpr int kRunsAhead = 4;
template <typename T>
__device__ void chunk_pair_fast(const T* x, const T* y, int64_t n, float& Mx, FF& Zx, float& My,
                                FF& Zy) {
  constexpr int R = Storage<T>::kVec;
  const int lane = threadIdx.x & 31;
  const bool vec = (((uintptr_t)x | (uintptr_t)y) & 15) == 0;
  const int64_t nruns = (n + R - 1) / R;
  const int64_t nfull = vec ? n / R : 0;  // runs read as whole vectors
  OnlineLse sx, sy;
  sx.init();
  sy.init();
  int64_t j = lane;
  for (; j + 32 * (kRunsAhead - 1) < nfull; j += 32 * kRunsAhead) {
    uint4 vx[kRunsAhead], vy[kRunsAhead];
#pragma unroll
    for (int u = 0; u < kRunsAhead; ++u) {
      vx[u] = __ldg(reinterpret_cast<const uint4*>(x) + j + 32 * u);
      vy[u] = __ldg(reinterpret_cast<const uint4*>(y) + j + 32 * u);
    }
#pragma unroll
    for (int u = 0; u < kRunsAhead; ++u) {
      float f[R];
      Storage<T>::unpack(vx[u], f);
      sx.update<R>(f);
      Storage<T>::unpack(vy[u], f);
      sy.update<R>(f);
    }
  }
  for (; j < nruns; j += 32) {
    float f[R];
    load_run<T>(x, j, n, vec, f);
    sx.update<R>(f);
    load_run<T>(y, j, n, vec, f);
    sy.update<R>(f);
  }
  finish_partial(sx, Mx, Zx);
  finish_partial(sy, My, Zy);
}

// Float-float path (fp32 logits): the chunk's max first, then
// sum exp(x - M) with the float-float exponential and float-pair sums.
template <typename T>
__device__ void chunk_partial(const T* x, int64_t n, const float* thi, const float* tlo,
                              const ExpTable& tab, float& M, FF& Z) {
  constexpr int R = Storage<T>::kVec;
  const int lane = threadIdx.x & 31;
  const bool vec = ((uintptr_t)x & 15) == 0;
  const int64_t nruns = (n + R - 1) / R;
  float m = -INFINITY;
  bool nan = false;
  for (int64_t j = lane; j < nruns; j += 32) {
    float f[R];
    load_run<T>(x, j, n, vec, f);
#pragma unroll
    for (int e = 0; e < R; ++e) {
      nan |= f[e] != f[e];
      m = fmaxf(m, f[e]);
    }
  }
  m = warp_max(m);
  nan = __any_sync(0xFFFFFFFFu, nan);
  FF s = {0.f, 0.f};
  if (m != -INFINITY && !nan) {
    for (int64_t j = lane; j < nruns; j += 32) {
      float f[R];
      load_run<T>(x, j, n, vec, f);
#pragma unroll
      for (int e = 0; e < R; ++e) {
        if (f[e] == -INFINITY) continue;
        const FF d = two_sum(f[e], -m);
        s = ff_add(s, exp_ff(d.hi, d.lo, thi, tlo, tab));
      }
    }
  }
  s = warp_sum_ff2(s);
  Z = FF{__shfl_sync(0xFFFFFFFFu, s.hi, 0), __shfl_sync(0xFFFFFFFFu, s.lo, 0)};
  M = nan ? NAN : m;
}

// At most 72 registers, 7 CTAs per SM (measured: 3.61 against 3.67 ms per
// two-slice step on the large-vocabulary rows at the 80 registers it takes
// unbounded).
template <typename T, bool kPrecise>
__global__ void __launch_bounds__(32 * kVocabWarps, 7) vocab_partials_kernel(const VocabArgs a) {
  __shared__ float s_thi[64], s_tlo[64];
  if (threadIdx.x < 64) {
    s_thi[threadIdx.x] = a.tab.hi[threadIdx.x];
    s_tlo[threadIdx.x] = a.tab.lo[threadIdx.x];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t rows = a.rows;
  const int64_t items = rows * a.nck;
  const int64_t wstride = (int64_t)gridDim.x * kVocabWarps;
  for (int64_t it = (int64_t)blockIdx.x * kVocabWarps + (threadIdx.x >> 5); it < items;
       it += wstride) {
    const int64_t c = it / rows, row = it - c * rows;  // chunk-major: rows of a chunk together
    if (!a.mask[row]) continue;
    const int64_t e0 = c * kVChunk;
    const int64_t n = (a.Vk - e0) < kVChunk ? (a.Vk - e0) : kVChunk;
    const T* xp = reinterpret_cast<const T*>(a.policy) + row * a.Vk + e0;
    const T* xr = reinterpret_cast<const T*>(a.ref) + row * a.Vk + e0;
    float Mp, Mr;
    FF Zp, Zr;
    if (kPrecise) {
      chunk_partial<T>(xp, n, s_thi, s_tlo, a.tab, Mp, Zp);
      chunk_partial<T>(xr, n, s_thi, s_tlo, a.tab, Mr, Zr);
    } else {
      chunk_pair_fast<T>(xp, xr, n, Mp, Zp, Mr, Zr);
    }
    if (lane == 0) {
      a.part_p[c * rows + row] = make_float4(Mp, Zp.hi, Zp.lo, 0.f);
      a.part_r[c * rows + row] = make_float4(Mr, Zr.hi, Zr.lo, 0.f);
    }
    if (c == 0 && lane == 0) {  // the action logit, where this slice holds it
      const int64_t act = a.actions[row] - a.v_begin;
      const bool own = act >= 0 && act < a.Vk;
      a.act_logits[row] = own ? Storage<T>::load1(reinterpret_cast<const T*>(a.policy) +
                                                  row * a.Vk + act)
                              : 0.f;
      a.act_logits[rows + row] = own ? Storage<T>::load1(reinterpret_cast<const T*>(a.ref) +
                                                         row * a.Vk + act)
                                     : 0.f;
    }
  }
}

// The row's logsumexp from its chunk partials, folded in chunk order:
// M = max M_c, Z = sum_c Z_c e^(M_c - M) in float pairs (a float-float
// exponential), then M + log Z in double.
__device__ __forceinline__ double fold_chunks(const float4* part, int64_t rows, int64_t row,
                                              int64_t nck, const float* thi, const float* tlo,
                                              const ExpTable& tab) {
  float M = -INFINITY;
  bool nan = false;
  for (int64_t c = 0; c < nck; ++c) {
    const float m = part[c * rows + row].x;
    nan |= m != m;
    M = fmaxf(M, m);
  }
  if (nan) return NAN;
  if (M == -INFINITY) return -INFINITY;
  FF Z = {0.f, 0.f};
  for (int64_t c = 0; c < nck; ++c) {
    const float4 r = part[c * rows + row];
    if (r.x == -INFINITY) continue;
    const FF d = two_sum(r.x, -M);
    const FF e = exp_ff(d.hi, d.lo, thi, tlo, tab);
    // (Z_c.hi + Z_c.lo) * e as a float pair
    const float ph = __fmul_rn(r.y, e.hi);
    const float pl = __fmaf_rn(r.y, e.hi, -ph);
    const float lo = __fadd_rn(pl, __fadd_rn(__fmul_rn(r.y, e.lo), __fmul_rn(r.z, e.hi)));
    Z = ff_add(Z, fast_two_sum(ph, lo));
  }
  return (double)M + log((double)Z.hi + (double)Z.lo);
}

__global__ void __launch_bounds__(kMergeThreads) vocab_merge_kernel(const VocabArgs a) {
  __shared__ float s_thi[64], s_tlo[64];
  if (threadIdx.x < 64) {
    s_thi[threadIdx.x] = a.tab.hi[threadIdx.x];
    s_tlo[threadIdx.x] = a.tab.lo[threadIdx.x];
  }
  __syncthreads();
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= a.rows) return;
  if (!a.mask[row]) {  // a masked row has no logsumexp and no gradient weight
    a.lse_w[row] = 0.0;
    a.lse_w[a.rows + row] = 0.0;
    if (a.logps_out) a.logps_out[row] = 0.f;
    return;
  }
  const int64_t act = a.actions[row];
  if (act < 0 || act >= a.V) {  // no slice holds this action
    atomicOr(&a.hdr->status, (unsigned)GRPO_ERR_ACTION_RANGE);
    a.slot_p[row] = NAN;
    a.slot_k[row] = NAN;
    a.lse_w[row] = NAN;
    if (a.logps_out) a.logps_out[row] = NAN;
    return;
  }
  const double lse_p = fold_chunks(a.part_p, a.rows, row, a.nck, s_thi, s_tlo, a.tab);
  const double lse_r = fold_chunks(a.part_r, a.rows, row, a.nck, s_thi, s_tlo, a.tab);
  const double lp = (double)a.act_logits[row] - lse_p;
  const double lr = (double)a.act_logits[a.rows + row] - lse_r;
  a.slot_p[row] = lp;
  a.slot_k[row] = lr - lp;
  a.lse_w[row] = lse_p;
  if (a.logps_out) a.logps_out[row] = (float)lp;
}

template <typename T>
static cudaError_t launch_partials_t(const VocabArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // one wave of resident CTAs, each warp striding over the items
  const void* kern = a.precise ? (const void*)vocab_partials_kernel<T, true>
                               : (const void*)vocab_partials_kernel<T, false>;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kVocabWarps, 0);
  if (e != cudaSuccess) return e;
  const int64_t items = a.rows * a.nck;
  int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  const int64_t need = (items + kVocabWarps - 1) / kVocabWarps;
  if (grid > need) grid = need;
  if (grid < 1) return cudaSuccess;
  if (a.precise)
    vocab_partials_kernel<T, true><<<(unsigned)grid, 32 * kVocabWarps, 0, s>>>(a);
  else
    vocab_partials_kernel<T, false><<<(unsigned)grid, 32 * kVocabWarps, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_vocab_partials(const VocabArgs& a, grpo_dtype_t dt, cudaStream_t s) {
  switch (dt) {
    case GRPO_F32: return launch_partials_t<float>(a, s);
    case GRPO_BF16: return launch_partials_t<__nv_bfloat16>(a, s);
    default: return launch_partials_t<__half>(a, s);
  }
}

cudaError_t launch_vocab_merge(const VocabArgs& a, cudaStream_t s) {
  const int64_t grid = (a.rows + kMergeThreads - 1) / kMergeThreads;
  if (grid < 1) return cudaSuccess;
  vocab_merge_kernel<<<(unsigned)grid, kMergeThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
