// grpo_api.cu -- the C ABI of libgrpo_gb300.so (declared in include/grpo.h):
// argument validation, workspace carving and the launch sequence.
//
// Every host-checkable error is found before the first CUDA call, so a
// rejected call launches nothing.  A call enqueues, in stream order:
//   memset of the workspace header (status word, counters)
//   prep     group advantages (+ active-token counts)   grpo_prep.cu
//   rows     fused sweep over vocabulary rows            grpo_rows.cu
//   reduce   fixed-order reduction to the scalars        grpo_reduce.cu
// or, for the logps-only boundary, prep + the kernel of grpo_logps.cu.
// A shard call (grpo_shard_t) runs the same kernels on its sequences, with
// the whole batch's groups and counts, and leaves the scalar to
// grpo_loss_finalize.
#include <math.h>
#include <string.h>

#include "grpo_internal.cuh"

using namespace grpo;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t elem_size(grpo_dtype_t dt) { return dt == GRPO_F32 ? 4 : 2; }

grpo_status_t check_params(const grpo_params_t* p) {
  if (!p) return GRPO_ERR_NULL;
  if (!(isfinite(p->clip_eps_lo) && isfinite(p->clip_eps_hi) && isfinite(p->beta) &&
        isfinite(p->adv_eps) && isfinite(p->grad_scale)))
    return GRPO_ERR_PARAM;
  if (!(p->clip_eps_lo >= 0.f && p->clip_eps_lo < 1.f)) return GRPO_ERR_PARAM;
  if (!(p->clip_eps_hi >= 0.f)) return GRPO_ERR_PARAM;
  if (!(p->beta >= 0.f)) return GRPO_ERR_PARAM;
  if (!(p->adv_eps > 0.f)) return GRPO_ERR_PARAM;
  if (p->reduction != GRPO_TOKEN_MEAN && p->reduction != GRPO_SEQUENCE_MEAN &&
      p->reduction != GRPO_FIXED_CONSTANT)
    return GRPO_ERR_PARAM;
  if (p->reduction == GRPO_FIXED_CONSTANT && !(isfinite(p->norm_constant) && p->norm_constant > 0.f))
    return GRPO_ERR_PARAM;
  if (p->flags & ~(GRPO_ADV_EPS_ADD | GRPO_SKIP_MASKED_GRAD_ROWS | GRPO_FLAG_SEPARATE_PREP |
                   GRPO_FLAG_WORKSPACE_CLEAN | GRPO_FLAG_OVERLAP_LAUNCH | GRPO_FLAG_TEST_STALLED_COPY |
                   GRPO_FLAG_TEST_STALLED_BARRIER))
    return GRPO_ERR_PARAM;
  if (p->kl_type != GRPO_KL_K3 && p->kl_type != GRPO_KL_K1 && p->kl_type != GRPO_KL_K2)
    return GRPO_ERR_PARAM;
  if (p->surrogate != GRPO_SURROGATE_CLIP && p->surrogate != GRPO_SURROGATE_CISPO)
    return GRPO_ERR_PARAM;
  if (p->dual_clip_c != 0.f) {  // off, or c > 1 with the clipped surrogate
    if (!(isfinite(p->dual_clip_c) && p->dual_clip_c > 1.f)) return GRPO_ERR_PARAM;
    if (p->surrogate != GRPO_SURROGATE_CLIP) return GRPO_ERR_PARAM;
  }
  if (p->ratio_level != 0 && p->ratio_level != 1) return GRPO_ERR_PARAM;
  if (p->ratio_level == 1 &&
      (p->reduction != GRPO_SEQUENCE_MEAN || p->surrogate != GRPO_SURROGATE_CLIP))
    return GRPO_ERR_PARAM;  // GSPO is sequence-level only
  if (p->clip_counts && ((uintptr_t)p->clip_counts & 7)) return GRPO_ERR_ALIGN;
  return GRPO_OK;
}

Variant variant_of(const grpo_params_t* p) {
  Variant v;
  v.eps_lo = p->clip_eps_lo;
  v.eps_hi = p->clip_eps_hi;
  v.beta = p->beta;
  v.dual_c = p->dual_clip_c;
  v.kl_type = p->kl_type;
  v.surrogate = p->surrogate;
  v.seq_ratio = p->ratio_level;
  return v;
}

// Resolves the group spec to (spp, boundaries, G).
grpo_status_t check_groups(const grpo_groups_t* g, int64_t B, int32_t* spp,
                           const int64_t** bounds, int64_t* G) {
  if (!g) return GRPO_ERR_NULL;
  if (g->num_seqs != B) return GRPO_ERR_SHAPE;
  const bool has_spp = g->samples_per_prompt != 0;
  const bool has_csr = g->group_boundaries != nullptr;
  if (has_spp == has_csr || g->samples_per_prompt < 0) return GRPO_ERR_GROUP_SPEC;
  if (has_spp) {
    if (B % g->samples_per_prompt != 0) return GRPO_ERR_SHAPE;
    *spp = g->samples_per_prompt;
    *bounds = nullptr;
    *G = B / g->samples_per_prompt;
  } else {
    if (g->num_groups < 0 || g->num_groups > B || (B > 0 && g->num_groups < 1))
      return GRPO_ERR_SHAPE;
    if (!aligned(g->group_boundaries, 8)) return GRPO_ERR_ALIGN;
    *spp = 0;
    *bounds = g->group_boundaries;
    *G = g->num_groups;
  }
  return GRPO_OK;
}

// Slots per sequence: positions and counts within a sequence are 32-bit.
static constexpr int64_t kMaxT = (int64_t)1 << 30;

grpo_status_t check_ws(const void* ws, size_t ws_bytes, int64_t B, int64_t T) {
  if (!ws) return GRPO_ERR_NULL;
  if (!aligned(ws, 256)) return GRPO_ERR_ALIGN;
  if (ws_bytes < WsLayout(B, T).total) return GRPO_ERR_WORKSPACE;
  return GRPO_OK;
}

// 2^(j/64) as float pairs and the three-part split of ln2/64 used by the
// precise exponential (Tang's method); built once from libm's double exp2.
const ExpTable& exp_table() {
  static const ExpTable tab = [] {
    ExpTable t;
    for (int j = 0; j < 64; ++j) {
      double v = exp2((double)j / 64.0);
      t.hi[j] = (float)v;
      t.lo[j] = (float)(v - (double)t.hi[j]);
    }
    const double L = 0.69314718055994530942 / 64.0;
    const double c1 = floor(L * 131072.0 + 0.5) / 131072.0;  // 11 significant bits
    t.c1 = (float)c1;
    t.c2 = (float)(L - c1);
    t.c3 = (float)(L - c1 - (double)t.c2);
    t.inv = (float)(64.0 / 0.69314718055994530942);
    return t;
  }();
  return tab;
}

grpo_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA; }

// A call's place in the batch: the whole batch, or a shard (grpo_shard_t)
// whose groups and rewards span Bg sequences while its token arguments cover
// B of them from seq_begin on.
struct Placement {
  int64_t Bg = 0, seq_begin = 0;
  const unsigned long long* NS = nullptr;  // the batch counts, when given
  SeqTotal* totals = nullptr;              // the shard's records, when sharded
  bool shard = false;
};
grpo_status_t placement_of(const grpo_params_t* p, const grpo_groups_t* g, int64_t B,
                           Placement* pl) {
  if (!p->shard) {
    pl->Bg = B;
    return GRPO_OK;
  }
  const grpo_shard_t* sh = p->shard;
  pl->shard = true;
  pl->Bg = g->num_seqs;
  pl->seq_begin = sh->seq_begin;
  if (pl->seq_begin < 0 || pl->Bg < 0 || pl->seq_begin > pl->Bg || B > pl->Bg - pl->seq_begin)
    return GRPO_ERR_SHAPE;
  if (!sh->global_counts || (B > 0 && !sh->totals_out)) return GRPO_ERR_NULL;
  if (!aligned(sh->global_counts, 8) || !aligned(sh->totals_out, 16)) return GRPO_ERR_ALIGN;
  pl->NS = sh->global_counts;
  pl->totals = reinterpret_cast<SeqTotal*>(sh->totals_out);
  return GRPO_OK;
}

}  // namespace

extern "C" size_t grpo_workspace_size(int64_t B, int64_t T, int64_t num_groups) {
  if (B < 0 || T < 0 || num_groups < 0) return 0;
  return WsLayout(B, T).total;
}

extern "C" grpo_status_t grpo_group_adv(const float* rewards, const grpo_groups_t* groups,
                                        float adv_eps, uint32_t flags, float* adv_out,
                                        void* ws, size_t ws_bytes, void* stream) {
  if (!groups || !adv_out) return GRPO_ERR_NULL;
  const int64_t B = groups->num_seqs;
  if (B < 0) return GRPO_ERR_SHAPE;
  if (B > 0 && !rewards) return GRPO_ERR_NULL;
  int32_t spp;
  const int64_t* bounds;
  int64_t G;
  grpo_status_t st = check_groups(groups, B, &spp, &bounds, &G);
  if (st != GRPO_OK) return st;
  if (!(isfinite(adv_eps) && adv_eps > 0.f)) return GRPO_ERR_PARAM;
  if (flags & ~GRPO_ADV_EPS_ADD) return GRPO_ERR_PARAM;
  if (!aligned(rewards, 4) || !aligned(adv_out, 4)) return GRPO_ERR_ALIGN;
  if ((st = check_ws(ws, ws_bytes, B, 0)) != GRPO_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const WsLayout lay(B, 0);
  WsHeader* hdr = (WsHeader*)w;
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return GRPO_ERR_CUDA;
  PrepArgs pa{rewards, bounds, B, 0, G, B, 0, &hdr->N, spp, adv_eps,
              (int)(flags & GRPO_ADV_EPS_ADD), nullptr, 0, (double*)(w + lay.off_A), nullptr,
              adv_out, nullptr, nullptr, hdr};
  return cuda_status(launch_prep(pa, s));
}

extern "C" grpo_status_t grpo_loss_fwd_bwd(
    const void* policy_logits, const void* ref_logits, grpo_dtype_t dt, int64_t B, int64_t T,
    int64_t V, const int64_t* action_ids, const float* old_logps,
    const uint8_t* completion_mask, const float* rewards, const grpo_groups_t* groups,
    const grpo_params_t* params, void* grad_logits, float* out3, float* per_seq,
    float* logps_out, float* adv_out, void* ws, size_t ws_bytes, void* stream) {
  if (dt != GRPO_F32 && dt != GRPO_BF16 && dt != GRPO_F16) return GRPO_ERR_DTYPE;
  if (B < 0 || T < 0 || T > kMaxT || V < 1) return GRPO_ERR_SHAPE;
  if (!params || !groups) return GRPO_ERR_NULL;
  const bool any_rows = B > 0 && T > 0;
  if (any_rows && (!policy_logits || !ref_logits || !action_ids || !old_logps ||
                   !completion_mask))
    return GRPO_ERR_NULL;
  grpo_status_t st = check_params(params);
  if (st != GRPO_OK) return st;
  Placement pl;
  if ((st = placement_of(params, groups, B, &pl)) != GRPO_OK) return st;
  if (!out3 && !pl.shard) return GRPO_ERR_NULL;
  if (pl.Bg > 0 && !rewards) return GRPO_ERR_NULL;
  int32_t spp;
  const int64_t* bounds;
  int64_t G;
  if ((st = check_groups(groups, pl.Bg, &spp, &bounds, &G)) != GRPO_OK) return st;
  const size_t es = elem_size(dt);
  if (!aligned(policy_logits, es) || !aligned(ref_logits, es) || !aligned(grad_logits, es) ||
      !aligned(action_ids, 8) || !aligned(old_logps, 4) || !aligned(rewards, 4) ||
      !aligned(out3, 4) || !aligned(per_seq, 4) || !aligned(logps_out, 4) ||
      !aligned(adv_out, 4))
    return GRPO_ERR_ALIGN;
  if ((st = check_ws(ws, ws_bytes, pl.Bg, T)) != GRPO_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const WsLayout lay(pl.Bg, T);
  WsHeader* hdr = (WsHeader*)w;
  int32_t* L = (int32_t*)(w + lay.off_L);
  double* A = (double*)(w + lay.off_A);  // [Bg]: every group's advantages
  double* slot_p = (double*)(w + lay.off_slots);
  double* slot_k = slot_p + B * T;
  const unsigned long long* NS = pl.NS ? pl.NS : &hdr->N;
  SeqTotal* totals = pl.shard ? pl.totals : (SeqTotal*)(w + lay.off_seq);

  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return GRPO_ERR_CUDA;
  PrepArgs pa{rewards, bounds, B, T, G, pl.Bg, pl.seq_begin, &hdr->N, spp, params->adv_eps,
              (int)(params->flags & GRPO_ADV_EPS_ADD), completion_mask, 1, A, nullptr, adv_out, L,
              nullptr, hdr};
  cudaError_t e = launch_prep(pa, s);
  if (e != cudaSuccess) return GRPO_ERR_CUDA;

  const Variant var = variant_of(params);
  if (any_rows) {
    RowArgs ra;
    ra.policy = policy_logits;
    ra.ref = ref_logits;
    ra.grad = grad_logits;
    ra.actions = action_ids;
    ra.old = old_logps;
    ra.mask = completion_mask;
    ra.L = L;
    ra.A = A + pl.seq_begin;
    ra.slot_p = slot_p;
    ra.slot_k = slot_k;
    ra.logps_out = logps_out;
    ra.hdr = hdr;
    ra.NS = NS;
    ra.B = B;
    ra.T = T;
    ra.V = V;
    ra.eps_lo = params->clip_eps_lo;
    ra.eps_hi = params->clip_eps_hi;
    ra.beta = params->beta;
    ra.grad_scale = params->grad_scale;
    ra.reduction = params->reduction;
    ra.flags = params->flags;
    ra.precise_ok = dt == GRPO_F32;
    ra.tab = exp_table();
    ra.var = var;
    ra.norm_c = params->norm_constant;
    if (var.seq_ratio) {  // GSPO: sweep 1, the per-sequence step, sweep 2
      if (launch_gspo_rows(ra, dt, 1, params->profile, s) != cudaSuccess) return GRPO_ERR_CUDA;
      ReduceArgs rd{completion_mask, L, A + pl.seq_begin, totals, slot_p, slot_k, B, T,
                    params->beta, params->reduction, hdr, NS, out3, per_seq, 1,
                    params->norm_constant, params->clip_counts, pl.shard ? 1 : 0, var, old_logps,
                    params->grad_scale, 1, nullptr};
      if (launch_reduce(rd, s) != cudaSuccess) return GRPO_ERR_CUDA;
      if (grad_logits && launch_gspo_rows(ra, dt, 2, params->profile, s) != cudaSuccess)
        return GRPO_ERR_CUDA;
      if (!grad_logits && params->profile && params->profile->stop)
        cudaEventRecord((cudaEvent_t)params->profile->stop, s);
      return GRPO_OK;
    }
    e = launch_rows(ra, dt, params->profile, s);
    if (e != cudaSuccess) return GRPO_ERR_CUDA;
  }
  Variant rv = var;
  rv.seq_ratio = 0;  // no rows: nothing for the GSPO step to do
  ReduceArgs rd{completion_mask, L, A + pl.seq_begin, totals, slot_p, slot_k, B, T,
                params->beta, params->reduction, hdr, NS, out3, per_seq,
                var.splits_A() ? 1 : 0, params->norm_constant,
                params->clip_counts, pl.shard ? 1 : 0, rv, old_logps, params->grad_scale, 0,
                nullptr};
  return cuda_status(launch_reduce(rd, s));
}

extern "C" grpo_status_t grpo_loss_from_logps(const float* logps, const float* old_logps,
                                              const float* ref_logps,
                                              const uint8_t* completion_mask, int64_t B,
                                              int64_t T, const float* rewards,
                                              const grpo_groups_t* groups,
                                              const grpo_params_t* params, float* grad_logps,
                                              float* out3, float* per_seq, float* adv_out,
                                              void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || T < 0 || T > kMaxT) return GRPO_ERR_SHAPE;
  if (!params || !groups) return GRPO_ERR_NULL;
  grpo_status_t st = check_params(params);
  if (st != GRPO_OK) return st;
  const bool any_rows = B > 0 && T > 0;
  if (any_rows && (!logps || !old_logps || !completion_mask)) return GRPO_ERR_NULL;
  if (any_rows && !ref_logps && params->beta != 0.f) return GRPO_ERR_NULL;
  Placement pl;
  if ((st = placement_of(params, groups, B, &pl)) != GRPO_OK) return st;
  if (!out3 && !pl.shard) return GRPO_ERR_NULL;
  if (pl.Bg > 0 && !rewards) return GRPO_ERR_NULL;
  int32_t spp;
  const int64_t* bounds;
  int64_t G;
  if ((st = check_groups(groups, pl.Bg, &spp, &bounds, &G)) != GRPO_OK) return st;
  if (!aligned(logps, 4) || !aligned(old_logps, 4) || !aligned(ref_logps, 4) ||
      !aligned(rewards, 4) || !aligned(grad_logps, 4) || !aligned(out3, 4) ||
      !aligned(per_seq, 4) || !aligned(adv_out, 4))
    return GRPO_ERR_ALIGN;
  if ((st = check_ws(ws, ws_bytes, pl.Bg, T)) != GRPO_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const WsLayout lay(pl.Bg, T);
  WsHeader* hdr = (WsHeader*)w;
  int32_t* L = (int32_t*)(w + lay.off_L);
  double* A = (double*)(w + lay.off_A);     // [Bg]: every group's advantages
  float2* Aff = (float2*)(w + lay.off_Aff);  // [Bg]
  int2* rng = (int2*)(w + lay.off_rng);
  const unsigned long long* NS = pl.NS ? pl.NS : &hdr->N;
  SeqTotal* totals = pl.shard ? pl.totals : (SeqTotal*)(w + lay.off_seq);
  // one cooperative launch when the batch's CTAs fit the GPU at once, else
  // the separate advantage / count pass first
  bool fused = false;
  if (!(params->flags & GRPO_FLAG_SEPARATE_PREP) && B > 0 && T > 0) {
    int64_t cap = 0;
    if (logps_fused_capacity(&cap) != cudaSuccess) return GRPO_ERR_CUDA;
    fused = B <= cap;
  }
  // the logps kernel's last CTA leaves the header clean; the caller may
  // state that it still is (GRPO_FLAG_WORKSPACE_CLEAN)
  if (!(params->flags & GRPO_FLAG_WORKSPACE_CLEAN) &&
      cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess)
    return GRPO_ERR_CUDA;
  PrepArgs pa{rewards, bounds, B, T, G, pl.Bg, pl.seq_begin, &hdr->N, spp, params->adv_eps,
              (int)(params->flags & GRPO_ADV_EPS_ADD), completion_mask, 1, A, Aff, adv_out, L,
              rng, hdr};
  if (!fused && launch_prep(pa, s) != cudaSuccess) return GRPO_ERR_CUDA;
  LogpsArgs la{logps, old_logps, ref_logps, completion_mask, A + pl.seq_begin,
               Aff + pl.seq_begin, rng, L, totals, grad_logps, out3,
               per_seq, hdr, B, T, params->clip_eps_lo, params->clip_eps_hi, params->beta,
               params->grad_scale, params->reduction, variant_of(params),
               params->norm_constant, params->clip_counts, NS, pl.shard ? 1 : 0, params->flags,
               fused ? 1 : 0, rewards, bounds, G, pl.Bg, pl.seq_begin, spp, params->adv_eps,
               (int)(params->flags & GRPO_ADV_EPS_ADD), adv_out,
               (uint32_t*)(w + lay.off_slots)};
  cudaError_t e = launch_logps(la, params->profile, s);
  if (fused && e == cudaErrorCooperativeLaunchTooLarge) {
    // fewer SMs than the device has (a partitioned device, say): the two
    // launches instead, which give the same bits
    (void)cudaGetLastError();
    if (launch_prep(pa, s) != cudaSuccess) return GRPO_ERR_CUDA;
    la.fused = 0;
    e = launch_logps(la, params->profile, s);
  }
  return cuda_status(e);
}

extern "C" grpo_status_t grpo_count_active(const uint8_t* completion_mask, int64_t B, int64_t T,
                                           unsigned long long* counts_out, void* stream) {
  if (B < 0 || T < 0 || T > kMaxT) return GRPO_ERR_SHAPE;
  if (!counts_out || (B > 0 && T > 0 && !completion_mask)) return GRPO_ERR_NULL;
  if (!aligned(counts_out, 8)) return GRPO_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(counts_out, 0, 2 * sizeof(unsigned long long), s) != cudaSuccess)
    return GRPO_ERR_CUDA;
  PrepArgs pa{nullptr, nullptr, B, T, 0, B, 0, counts_out, 0, 1.f, 0, completion_mask, 1,
              nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return cuda_status(launch_prep(pa, s));
}

extern "C" grpo_status_t grpo_loss_finalize(const grpo_seq_total_t* totals, int64_t B,
                                            const unsigned long long* global_counts,
                                            const grpo_params_t* params, float* out3,
                                            void* stream) {
  if (B < 0) return GRPO_ERR_SHAPE;
  if (!params || !out3 || !global_counts || (B > 0 && !totals)) return GRPO_ERR_NULL;
  grpo_status_t st = check_params(params);
  if (st != GRPO_OK) return st;
  if (!aligned(totals, 16) || !aligned(global_counts, 8) || !aligned(out3, 4))
    return GRPO_ERR_ALIGN;
  return cuda_status(launch_finalize(reinterpret_cast<const SeqTotal*>(totals), B, global_counts,
                                     params->reduction, params->norm_constant, params->beta,
                                     out3, (cudaStream_t)stream));
}

extern "C" size_t grpo_vocab_chunk(void) { return (size_t)kVChunk; }

extern "C" grpo_status_t grpo_vocab_partials(const void* policy_slice, const void* ref_slice,
                                             grpo_dtype_t dt, int64_t B, int64_t T, int64_t Vk,
                                             int64_t v_begin, const int64_t* action_ids,
                                             const uint8_t* completion_mask, void* partials_p,
                                             void* partials_r, float* action_logits,
                                             void* stream) {
  if (dt != GRPO_F32 && dt != GRPO_BF16 && dt != GRPO_F16) return GRPO_ERR_DTYPE;
  if (B < 0 || T < 0 || T > kMaxT || Vk < 1 || v_begin < 0 || v_begin % kVChunk != 0)
    return GRPO_ERR_SHAPE;
  const int64_t rows = B * T;
  if (rows > 0 && (!policy_slice || !ref_slice || !action_ids || !completion_mask ||
                   !partials_p || !partials_r || !action_logits))
    return GRPO_ERR_NULL;
  const size_t es = elem_size(dt);
  if (!aligned(policy_slice, es) || !aligned(ref_slice, es) || !aligned(action_ids, 8) ||
      !aligned(partials_p, 16) || !aligned(partials_r, 16) || !aligned(action_logits, 4))
    return GRPO_ERR_ALIGN;
  VocabArgs va{};
  va.policy = policy_slice;
  va.ref = ref_slice;
  va.actions = action_ids;
  va.mask = completion_mask;
  va.rows = rows;
  va.Vk = Vk;
  va.v_begin = v_begin;
  va.nck = (Vk + kVChunk - 1) / kVChunk;
  va.part_p = (float4*)partials_p;
  va.part_r = (float4*)partials_r;
  va.act_logits = action_logits;
  va.precise = dt == GRPO_F32;
  va.tab = exp_table();
  return cuda_status(launch_vocab_partials(va, dt, (cudaStream_t)stream));
}

extern "C" grpo_status_t grpo_vocab_loss(const void* partials_p, const void* partials_r,
                                         int64_t num_chunks, const float* action_logits,
                                         int64_t V, const int64_t* action_ids,
                                         const float* old_logps, const uint8_t* completion_mask,
                                         int64_t B, int64_t T, const float* rewards,
                                         const grpo_groups_t* groups, const grpo_params_t* params,
                                         double* lse_w, float* out3, float* per_seq,
                                         float* logps_out, float* adv_out, void* ws,
                                         size_t ws_bytes, void* stream) {
  if (B < 0 || T < 0 || T > kMaxT || V < 1) return GRPO_ERR_SHAPE;
  if (num_chunks != (V + kVChunk - 1) / kVChunk) return GRPO_ERR_SHAPE;
  if (!params || !groups) return GRPO_ERR_NULL;
  const int64_t rows = B * T;
  if (rows > 0 && (!partials_p || !partials_r || !action_logits || !action_ids || !old_logps ||
                   !completion_mask || !lse_w))
    return GRPO_ERR_NULL;
  grpo_status_t st = check_params(params);
  if (st != GRPO_OK) return st;
  Placement pl;
  if ((st = placement_of(params, groups, B, &pl)) != GRPO_OK) return st;
  if (!out3 && !pl.shard) return GRPO_ERR_NULL;
  if (pl.Bg > 0 && !rewards) return GRPO_ERR_NULL;
  int32_t spp;
  const int64_t* bounds;
  int64_t G;
  if ((st = check_groups(groups, pl.Bg, &spp, &bounds, &G)) != GRPO_OK) return st;
  if (!aligned(partials_p, 16) || !aligned(partials_r, 16) || !aligned(action_logits, 4) ||
      !aligned(action_ids, 8) || !aligned(old_logps, 4) || !aligned(rewards, 4) ||
      !aligned(lse_w, 8) || !aligned(out3, 4) || !aligned(per_seq, 4) || !aligned(logps_out, 4) ||
      !aligned(adv_out, 4))
    return GRPO_ERR_ALIGN;
  if ((st = check_ws(ws, ws_bytes, pl.Bg, T)) != GRPO_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)ws;
  const WsLayout lay(pl.Bg, T);
  WsHeader* hdr = (WsHeader*)w;
  int32_t* L = (int32_t*)(w + lay.off_L);
  double* A = (double*)(w + lay.off_A);
  double* slot_p = (double*)(w + lay.off_slots);
  double* slot_k = slot_p + rows;
  const unsigned long long* NS = pl.NS ? pl.NS : &hdr->N;
  SeqTotal* totals = pl.shard ? pl.totals : (SeqTotal*)(w + lay.off_seq);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return GRPO_ERR_CUDA;
  PrepArgs pa{rewards, bounds, B, T, G, pl.Bg, pl.seq_begin, &hdr->N, spp, params->adv_eps,
              (int)(params->flags & GRPO_ADV_EPS_ADD), completion_mask, 1, A, nullptr, adv_out, L,
              nullptr, hdr};
  if (launch_prep(pa, s) != cudaSuccess) return GRPO_ERR_CUDA;
  if (rows > 0) {
    VocabArgs va{};
    va.actions = action_ids;
    va.mask = completion_mask;
    va.rows = rows;
    va.nck = num_chunks;
    va.V = V;
    va.part_p = (float4*)partials_p;
    va.part_r = (float4*)partials_r;
    va.act_logits = (float*)action_logits;
    va.tab = exp_table();
    va.slot_p = slot_p;
    va.slot_k = slot_k;
    va.lse_w = lse_w;
    va.logps_out = logps_out;
    va.hdr = hdr;
    if (launch_vocab_merge(va, s) != cudaSuccess) return GRPO_ERR_CUDA;
  }
  const Variant var = variant_of(params);
  ReduceArgs rd{completion_mask, L, A + pl.seq_begin, totals, slot_p, slot_k, B, T,
                params->beta, params->reduction, hdr, NS, out3, per_seq,
                var.splits_A() ? 1 : 0, params->norm_constant, params->clip_counts,
                pl.shard ? 1 : 0, var, old_logps, params->grad_scale, rows > 0 ? 1 : 0,
                rows > 0 ? lse_w + rows : nullptr};
  return cuda_status(launch_reduce(rd, s));
}

extern "C" grpo_status_t grpo_vocab_grad(const void* policy_slice, grpo_dtype_t dt, int64_t B,
                                         int64_t T, int64_t Vk, int64_t v_begin,
                                         const int64_t* action_ids,
                                         const uint8_t* completion_mask, const double* lse_w,
                                         void* grad_slice, uint32_t flags, void* stream) {
  if (dt != GRPO_F32 && dt != GRPO_BF16 && dt != GRPO_F16) return GRPO_ERR_DTYPE;
  if (B < 0 || T < 0 || T > kMaxT || Vk < 1 || v_begin < 0) return GRPO_ERR_SHAPE;
  if (flags & ~GRPO_SKIP_MASKED_GRAD_ROWS) return GRPO_ERR_PARAM;
  if (B * T > 0 && (!policy_slice || !action_ids || !completion_mask || !lse_w || !grad_slice))
    return GRPO_ERR_NULL;
  const size_t es = elem_size(dt);
  if (!aligned(policy_slice, es) || !aligned(grad_slice, es) || !aligned(action_ids, 8) ||
      !aligned(lse_w, 8))
    return GRPO_ERR_ALIGN;
  RowArgs ra{};
  ra.policy = policy_slice;
  ra.grad = grad_slice;
  ra.actions = action_ids;
  ra.mask = completion_mask;
  ra.B = B;
  ra.T = T;
  ra.V = Vk;
  ra.flags = flags;
  ra.precise_ok = dt == GRPO_F32;
  return cuda_status(launch_vocab_grad(ra, dt, v_begin, lse_w, (cudaStream_t)stream));
}

extern "C" grpo_status_t grpo_read_device_status(const void* ws, void* stream) {
  if (!ws) return GRPO_ERR_NULL;
  WsHeader h;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GRPO_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GRPO_ERR_CUDA;
  return (grpo_status_t)(h.status | h.last_status);
}

extern "C" const char* grpo_status_string(grpo_status_t status) {
  switch ((int)status) {
    case GRPO_OK: return "ok";
    case GRPO_ERR_NULL: return "a required pointer is NULL";
    case GRPO_ERR_SHAPE: return "invalid shape";
    case GRPO_ERR_DTYPE: return "unsupported dtype";
    case GRPO_ERR_ALIGN: return "misaligned pointer";
    case GRPO_ERR_GROUP_SPEC: return "give exactly one of samples_per_prompt and group_boundaries";
    case GRPO_ERR_PARAM: return "invalid loss parameter";
    case GRPO_ERR_WORKSPACE: return "workspace too small";
    case GRPO_ERR_CUDA: return "CUDA error";
    case GRPO_ERR_ACTION_RANGE: return "action id outside [0, V) on an active token";
    case GRPO_ERR_CSR: return "group_boundaries is not 0 = g0 < g1 < ... < gG = B";
    case GRPO_ERR_NONFINITE_REWARD: return "non-finite reward";
    case GRPO_ERR_TIMEOUT: return "an asynchronous copy did not complete in time";
    default: return "several device-detected errors (OR of status bits)";
  }
}
