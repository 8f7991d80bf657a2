/*
 * grpo.h -- C ABI of the GB300 (sm_103a) fused GRPO loss library
 *           (libgrpo_gb300.so).
 *
 * What is computed (RL-Kernel "GRPO Loss" operator page, sections "Entry
 * Point", "Tensor Contract", "Group specification", "Accuracy" and
 * "Normalizer semantics"; dockyard_rl "GRPO and the clipped policy-gradient
 * loss", sections "One loss, many algorithms" and "Reference-KL penalty";
 * grpo.cpp README, section "CUDA"):
 *
 *   A_i      = (R_i - mean_g R) / max(std_g R, adv_eps)     population std;
 *              A_i = 0 when every reward of the group is equal
 *   logp     = x_a - logsumexp(x)      x = policy row, a = action id
 *   ref_logp = y_a - logsumexp(y)      y = reference row
 *   r        = exp(logp - old_logp)
 *   p        = -min(r A, clip(r, 1 - eps_lo, 1 + eps_hi) A)
 *   d        = ref_logp - logp,  k = e^d - d - 1                (k3 KL)
 *   c        = 1 / max(N,1)                 token mean (N active tokens), or
 *              1 / (max(S,1) L_i)           sequence mean (S live sequences)
 *   policy_loss = sum c p,  kl = sum c k,  loss = policy_loss + beta kl
 *   dL/dlogp    = w = grad_scale c (g_pol + beta (1 - e^d)),
 *                 g_pol = 0 if (A>0, r>1+eps_hi) or (A<0, r<1-eps_lo), else -A r
 *   dL/dx_v     = w (1[v = a] - softmax(x)_v)
 *
 * That is the default loss; grpo_params_t selects the variants documented
 * with it (KL estimators k1 / k2, CISPO, the dual clip, the fixed-constant
 * normaliser, GSPO sequence-level ratios) and the clip counters.  Sequence
 * sharding (grpo_shard_t) and vocabulary parallelism (grpo_vocab_*) compute
 * the same loss, bit-identically at every degree.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers to row-major contiguous
 *     arrays owned by the caller; the library allocates nothing, keeps no
 *     state between calls and is safe to call concurrently on different
 *     streams with different workspaces.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronising.  Outputs are device values.
 *   - completion_mask is one byte per token, nonzero = active.  Masked
 *     tokens' logits, action ids and old_logps are never read: any value,
 *     NaN included, is allowed there.
 *   - Host-checkable errors (null pointers, shapes, parameters, alignment,
 *     workspace size) are returned at once and nothing is launched.
 *     Data-dependent errors found on the device (an action id outside
 *     [0, V) on an active token, malformed CSR offsets, a non-finite reward)
 *     set a bit in the workspace status word and make the three loss outputs
 *     NaN; read them with grpo_read_device_status().  No kernel ever traps.
 *   - Results are bitwise reproducible run to run: no reduction depends on
 *     CTA scheduling.
 */
#ifndef GRPO_GB300_H
#define GRPO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GRPO_OK = 0,
  GRPO_ERR_NULL = 1,       /* a required pointer is NULL */
  GRPO_ERR_SHAPE = 2,      /* negative sizes, T > 2^30, V < 1, B not a multiple of spp, ... */
  GRPO_ERR_DTYPE = 3,      /* unknown grpo_dtype_t */
  GRPO_ERR_ALIGN = 4,      /* a pointer is not aligned to its element size, or
                              the workspace is not 256-byte aligned */
  GRPO_ERR_GROUP_SPEC = 5, /* not exactly one of samples_per_prompt / boundaries */
  GRPO_ERR_PARAM = 6,      /* eps / beta / adv_eps / grad_scale / reduction / variant invalid,
                              or a flag bit this header does not define */
  GRPO_ERR_WORKSPACE = 7,  /* ws_bytes < grpo_workspace_size(...) */
  GRPO_ERR_CUDA = 8,       /* a CUDA launch failed */
  /* device-detected; bits of the status word (grpo_read_device_status) */
  GRPO_ERR_ACTION_RANGE = 16,    /* active token with action id outside [0, V) */
  GRPO_ERR_CSR = 32,             /* boundaries not 0 = g_0 < g_1 < ... < g_G = B */
  GRPO_ERR_NONFINITE_REWARD = 64, /* a reward is NaN or infinite */
  GRPO_ERR_TIMEOUT = 128          /* a bounded wait (an asynchronous copy, the grid
                                     barrier of the one-launch logps kernel) ran out */
} grpo_status_t;

typedef enum { GRPO_F32 = 0, GRPO_BF16 = 1, GRPO_F16 = 2 } grpo_dtype_t;

/* Normaliser ("Normalizer semantics"): the global active-token count, the
 * per-sequence count then the mean over live sequences, or a declared
 * constant (the Dr.GRPO form: the divisor does not depend on the mask). */
typedef enum {
  GRPO_TOKEN_MEAN = 0,
  GRPO_SEQUENCE_MEAN = 1,
  GRPO_FIXED_CONSTANT = 2 /* c = 1 / grpo_params_t.norm_constant for every active token */
} grpo_reduction_t;

/* Reference-KL estimator (dockyard_rl "Reference-KL penalty"; Relax
 * "REINFORCE++" and "REINFORCE++-baseline"), d = ref_logp - logp; the
 * gradient is the pathwise derivative of each formula. */
typedef enum {
  GRPO_KL_K3 = 0, /* e^d - d - 1 (low-variance, unbiased)     d/dlogp: 1 - e^d */
  GRPO_KL_K1 = 1, /* logp - ref_logp (the log ratio)          d/dlogp: 1 */
  GRPO_KL_K2 = 2  /* (logp - ref_logp)^2 / 2                  d/dlogp: logp - ref_logp */
} grpo_kl_t;

/* Policy surrogate (dockyard_rl "One loss, many algorithms", "CISPO"). */
typedef enum {
  GRPO_SURROGATE_CLIP = 0, /* -min(r A, clip(r) A), optionally dual-clipped */
  GRPO_SURROGATE_CISPO = 1 /* -A sg(clip(r)) logp: every token keeps a gradient
                              -A clip(r) through logp */
} grpo_surrogate_t;

/* Flags (grpo_params_t.flags and grpo_group_adv's flags). */
#define GRPO_ADV_EPS_ADD 1u          /* divide by std + adv_eps instead of max(std, adv_eps) */
#define GRPO_SKIP_MASKED_GRAD_ROWS 2u /* leave gradient rows of masked tokens untouched
                                         (caller pre-zeroed them) instead of writing 0 */
/* grpo_loss_from_logps: run the advantage / active-count pass as its own
 * launch before the per-sequence kernel.  By default, when every sequence's
 * CTA fits on the GPU at once (B up to 7 per SM: 1,064 on GB300), the pass is
 * folded into that kernel, launched cooperatively: each CTA scans its own
 * mask row and forms its own advantage, and the CTAs meet at a grid barrier
 * (bounded like every wait: GRPO_ERR_TIMEOUT) before the counts N and S are
 * read.  Both forms give the same bits.  Ignored by the other entry points. */
#define GRPO_FLAG_SEPARATE_PREP 4u
/* grpo_loss_from_logps: the caller states that the workspace header is clean
 * -- the previous call that used this workspace was a grpo_loss_from_logps
 * call that returned GRPO_OK (each such call leaves the header clean when
 * its kernels end, whatever status its data produced), or the caller zeroed
 * the workspace -- so the call skips its reset of the header (one memset
 * launch, about 1.3 us on GB300).  For loops that compute the loss from
 * log-probs step after step on one workspace.  Ignored by the other entry
 * points, which always reset the header (and leave it in use). */
#define GRPO_FLAG_WORKSPACE_CLEAN 8u
/* grpo_loss_from_logps' one-launch form: launch the kernel as a programmatic
 * dependent of the kernel before it on the stream, so that its CTAs are
 * dispatched while that kernel's last CTAs still run (they wait for it to
 * complete before touching memory), instead of as a cooperative launch, which
 * would rule that out (about 2 us per call on GB300).  The kernel's grid
 * barrier still needs every CTA of the batch resident at once, which only the
 * cooperative launch guarantees: with this flag the caller states that no
 * other kernel holds SMs for long while the call runs (nothing running on
 * other streams, say).  If that does not hold, the barrier's bounded wait runs
 * out (0.2 s) and the call reports GRPO_ERR_TIMEOUT with NaN loss outputs.
 * Ignored by the other entry points and by the two-launch form. */
#define GRPO_FLAG_OVERLAP_LAUNCH 16u
/* Test hook, for the failure-detection tests only: in grpo_loss_from_logps'
 * staged path (T % 16 == 0, 16-byte aligned arrays) the first asynchronous
 * copy of sequence 0 is made to under-deliver, so its bounded wait runs out
 * (after 0.2 s): the call then sets GRPO_ERR_TIMEOUT, the loss outputs are
 * NaN, the sequence's gradient is not written, and the context stays usable.
 * Ignored by the other entry points. */
#define GRPO_FLAG_TEST_STALLED_COPY 0x80000000u
/* Test hook, for the failure-detection tests only: in grpo_loss_from_logps'
 * one-launch form, the CTA of sequence 0 waits at the grid barrier for one
 * CTA more than there are, so its bounded wait runs out (after 0.2 s): the
 * call sets GRPO_ERR_TIMEOUT and the loss outputs are NaN; the context stays
 * usable.  Ignored elsewhere (and with GRPO_FLAG_SEPARATE_PREP). */
#define GRPO_FLAG_TEST_STALLED_BARRIER 0x40000000u

/* Group specification (RL-Kernel "GRPO Loss", "Group specification"): give
 * either samples_per_prompt > 0 or CSR group_boundaries of length
 * num_groups + 1 with boundaries[0] = 0, boundaries[num_groups] = num_seqs
 * and strictly increasing entries, e.g. {0, 8, 16, 24}; not both. */
typedef struct {
  int64_t num_seqs;                /* B */
  int32_t samples_per_prompt;      /* > 0: uniform groups of this size, B % spp == 0 */
  int32_t _reserved;
  const int64_t *group_boundaries; /* device pointer or NULL */
  int64_t num_groups;              /* used with group_boundaries (>= 1 when B > 0) */
} grpo_groups_t;

/* Optional timing hook: when non-NULL, `start` / `stop` (cudaEvent_t handles)
 * are recorded on the stream immediately before and after the main kernel
 * of a call -- the fused row kernel of grpo_loss_fwd_bwd, the per-token
 * kernel of grpo_loss_from_logps -- so a caller can time it alone. */
typedef struct {
  void *start;
  void *stop;
} grpo_profile_t;

/* One sequence's totals in the exact form the final reduction consumes
 * (policy and KL totals and the active count; opaque).  A data-parallel
 * shard writes one record per sequence it owns; concatenated in shard
 * order they are the whole batch's, and grpo_loss_finalize turns them into
 * the three loss outputs. */
typedef struct {
  unsigned char opaque[32];
} grpo_seq_total_t;

/* A data-parallel shard of the batch (RL-Kernel "Tensor and Data Parallel"):
 * a rank owns a contiguous range of whole sequences.  With a shard, a call's
 * rewards and group specification describe the WHOLE batch (advantages are
 * replicated: every rank normalises every group over the same rewards and
 * keeps its own slice), while the token arguments (logits or log-probs,
 * action_ids, old_logps, completion_mask, gradients, per_seq, adv_out)
 * cover only the shard's B sequences, starting at sequence seq_begin of the
 * batch.  The token weights use the whole batch's counts; besides the
 * counts, the per-sequence totals are all that ranks exchange.  Whatever the
 * partition, every gradient,
 * per-sequence total and loss output is bit-identical to the unsharded
 * call's. */
typedef struct {
  int64_t seq_begin;                        /* the shard's first sequence in the batch */
  const unsigned long long *global_counts;  /* device [2]: N (active tokens) and S (live
                                               sequences) of the whole batch, e.g. the sum
                                               over shards of grpo_count_active */
  grpo_seq_total_t *totals_out;             /* device [B]: the shard's per-sequence totals */
} grpo_shard_t;

/* Call parameters.  Zero-initialising the variant fields (kl_type,
 * surrogate, dual_clip_c, norm_constant, clip_counts) gives the GRPO loss
 * of the operator page: the clipped surrogate with k3 and no dual clip. */
typedef struct {
  float clip_eps_lo;  /* eps_lo, 0 <= eps_lo < 1   (clip_eps on the pages) */
  float clip_eps_hi;  /* eps_hi >= 0                (DAPO clip-higher when > eps_lo) */
  float beta;         /* KL coefficient >= 0 */
  float adv_eps;      /* > 0, 1e-6 on the pages */
  float grad_scale;   /* finite; multiplies every gradient (1 = dL/dlogits) */
  int32_t reduction;  /* grpo_reduction_t */
  uint32_t flags;     /* GRPO_ADV_EPS_ADD | GRPO_SKIP_MASKED_GRAD_ROWS | GRPO_FLAG_SEPARATE_PREP */
  int32_t kl_type;    /* grpo_kl_t */
  int32_t surrogate;  /* grpo_surrogate_t */
  float dual_clip_c;  /* 0: off.  > 1: dual clip ("ratio_clip_c", a lower bound
                         on negative-advantage terms): for A < 0 the objective is
                         max(min(r A, clip(r) A), c A), whose policy gradient is 0
                         where r > c.  Only with GRPO_SURROGATE_CLIP. */
  float norm_constant; /* GRPO_FIXED_CONSTANT: the declared constant, finite and
                          > 0; ignored by the other reductions */
  int32_t ratio_level; /* 0: token ratios r_t.  1: GSPO, one ratio per sequence,
                          rho_i = exp(mean over its active tokens of logp - old),
                          used by every token of the sequence in the clipped
                          surrogate (Relax "REINFORCE++ / REINFORCE++-baseline",
                          GSPO row; dockyard_rl sequence_level_importance_ratios).
                          Needs GRPO_SEQUENCE_MEAN and GRPO_SURROGATE_CLIP. */
  const grpo_profile_t *profile; /* host pointer or NULL */
  const grpo_shard_t *shard;     /* host pointer or NULL (the whole batch) */
  unsigned long long *clip_counts; /* device [3] or NULL: overwritten with the
                          number of active tokens clipped at the upper bound,
                          at the lower bound, and by the dual clip.  Clipped
                          surrogate: (A > 0, r > 1 + eps_hi), (A < 0,
                          r < 1 - eps_lo), (A < 0, r > c) -- the tokens whose
                          policy gradient a clip removes.  CISPO: r > 1 + eps_hi,
                          r < 1 - eps_lo (the weight clip(r) differs from r),
                          whatever the sign of A; the third is 0. */
} grpo_params_t;

/* Bytes of workspace the entry points below need for B sequences of T
 * token slots in num_groups groups (any of the three entry points; a
 * workspace of this size serves all of them).  A shard call (grpo_shard_t)
 * needs grpo_workspace_size(total sequences of the batch, T, 0).  The workspace is caller-owned
 * device memory, 256-byte aligned, needs no initialisation, and must not be
 * shared by calls that may run concurrently.  Returns 0 for invalid sizes. */
size_t grpo_workspace_size(int64_t B, int64_t T, int64_t num_groups);

/* Group-normalised advantages only ("Accuracy": advantages; "Group
 * specification").  rewards [B] f32 device; adv_out [B] f32 device.
 * flags: GRPO_ADV_EPS_ADD.  Writes the status word of `ws`. */
grpo_status_t grpo_group_adv(const float *rewards, const grpo_groups_t *groups,
                             float adv_eps, uint32_t flags, float *adv_out,
                             void *ws, size_t ws_bytes, void *stream);

/* The fused forward + backward from logits ("Entry Point": grpo_loss(...)
 * then loss.backward(); "Tensor Contract").
 *   policy_logits, ref_logits : [B,T,V] of dtype `dt`, contiguous.  ref may
 *                               equal policy.
 *   action_ids                : [B,T] int64.
 *   old_logps                 : [B,T] f32.
 *   completion_mask           : [B,T] uint8 / bool.
 *   rewards                   : [B] f32.
 *   grad_logits (nullable)    : [B,T,V] of dtype `dt`; receives dL/dlogits
 *                               (overwritten, not accumulated; may equal
 *                               policy_logits for an in-place gradient).
 *                               NULL = forward only.
 *   out3                      : [3] f32: loss, policy_loss, kl (not written,
 *                               and may be NULL, in a shard call).
 *   per_seq (nullable)        : [3,B] f32: per-sequence policy totals
 *                               sum_t p, KL totals sum_t k, active counts L_i.
 *   logps_out (nullable)      : [B,T] f32: logp of active tokens, 0 elsewhere.
 *   adv_out (nullable)        : [B] f32: the advantages used.
 * Pointers must be aligned to their element size; rows need not be 16-byte
 * aligned.  B, T >= 0, V >= 1. */
grpo_status_t grpo_loss_fwd_bwd(const void *policy_logits, const void *ref_logits,
                                grpo_dtype_t dt, int64_t B, int64_t T, int64_t V,
                                const int64_t *action_ids, const float *old_logps,
                                const uint8_t *completion_mask, const float *rewards,
                                const grpo_groups_t *groups, const grpo_params_t *params,
                                void *grad_logits, float *out3, float *per_seq,
                                float *logps_out, float *adv_out, void *ws,
                                size_t ws_bytes, void *stream);

/* The same loss when the per-token log-probs are already known (grpo.cpp
 * README "CUDA": the selected-token GRPO loss; RL-Kernel "Tensor and Data
 * Parallel": the objective only ever receives log-probs, the vocabulary
 * already reduced away).
 *   logps, old_logps : [B,T] f32.   ref_logps : [B,T] f32, NULL iff beta == 0.
 *   completion_mask  : [B,T] uint8.  rewards : [B] f32.
 *   grad_logps (nullable) : [B,T] f32, receives dL/dlogp (0 on masked tokens).
 *   out3, per_seq, adv_out : as for grpo_loss_fwd_bwd. */
grpo_status_t grpo_loss_from_logps(const float *logps, const float *old_logps,
                                   const float *ref_logps, const uint8_t *completion_mask,
                                   int64_t B, int64_t T, const float *rewards,
                                   const grpo_groups_t *groups, const grpo_params_t *params,
                                   float *grad_logps, float *out3, float *per_seq,
                                   float *adv_out, void *ws, size_t ws_bytes, void *stream);

/* grpo_loss_fwd_bwd for callers that cannot allocate device memory where
 * they need the loss -- code running while a stream is captured into a CUDA
 * graph, hosts whose device memory belongs to another allocator, loops that
 * cannot afford a cudaMalloc / cudaFree.  The operator pages have no
 * counterpart: this is a deployment variant of the same computation.
 * Arguments and results are those of grpo_loss_fwd_bwd without `ws` /
 * `ws_bytes`: the scratch memory is a fixed 4.5 MiB array in the library's
 * device image, present on every GPU that loads the library until the
 * process exits.  Sizes whose grpo_workspace_size(B, T, 0) exceeds 4.5 MiB
 * are rejected with GRPO_ERR_WORKSPACE (any B <= 8192 with B*T <= 262144
 * fits); in a shard call (grpo_params_t.shard) the limit applies to the
 * whole batch, grpo_workspace_size(groups->num_seqs, T, 0).  No device
 * memory is allocated.
 * The first call in a device's context looks the array's device address up
 * (with that device current) and keeps it for that context; make that first
 * call before any stream capture, and again after anything that replaces
 * the context (cudaDeviceReset).  All calls share the array: calls whose GPU
 * work may overlap (other streams or threads without ordering between them)
 * race on it and must be serialised by the caller. */
grpo_status_t grpo_loss_fwd_bwd_static(const void *policy_logits, const void *ref_logits,
                                       grpo_dtype_t dt, int64_t B, int64_t T, int64_t V,
                                       const int64_t *action_ids, const float *old_logps,
                                       const uint8_t *completion_mask, const float *rewards,
                                       const grpo_groups_t *groups, const grpo_params_t *params,
                                       void *grad_logits, float *out3, float *per_seq,
                                       float *logps_out, float *adv_out, void *stream);

/* Sequence sharding ("Tensor and Data Parallel", steps 2-6).  A rank that
 * owns B sequences of T slots counts them: counts_out (device [2]) receives
 * N = sum of active tokens and S = sequences with at least one, as exact
 * integers; the whole batch's counts are the sums over ranks.  (The page's
 * normaliser uses the batch-wide active-token count, exchanged as integers,
 * which makes it the same at any number of ranks.) */
grpo_status_t grpo_count_active(const uint8_t *completion_mask, int64_t B, int64_t T,
                                unsigned long long *counts_out, void *stream);

/* The loss outputs from the whole batch's per-sequence totals: the records
 * of every shard concatenated in shard order (B records, all from the same
 * entry point: grpo_loss_fwd_bwd or grpo_loss_from_logps), the batch counts
 * (device [2], as in grpo_shard_t) and the same params (reduction,
 * norm_constant, beta).  out3 = {loss, policy_loss, kl}, computed by the
 * same code, in the same order, as an unsharded call; so the result is
 * bit-identical to it (the page rules out an all-reduce for this sum: it
 * runs over the sequences in their declared order). */
grpo_status_t grpo_loss_finalize(const grpo_seq_total_t *totals, int64_t B,
                                 const unsigned long long *global_counts,
                                 const grpo_params_t *params, float *out3, void *stream);

/* Vocabulary parallelism (tensor parallelism over V; RL-Kernel "Tensor and
 * Data Parallel", step 1: the selected log-probs come from a vocab-parallel
 * log-prob, so the ratio and KL are bitwise the same at every tensor-parallel
 * degree).  A rank holds the
 * slice [v_begin, v_begin + Vk) of every policy and reference row, v_begin a
 * multiple of grpo_vocab_chunk() (every slice but the last spans whole
 * chunks).  The loss is formed by three calls around one exchange:
 *   1. grpo_vocab_partials on every rank: one partial normaliser per row and
 *      per chunk of its slice (the max M_c and sum_v exp(x_v - M_c) as a
 *      float pair), chunk-major [chunks][B*T] records of 16 bytes, and the
 *      action's policy / reference logit where the slice holds it (0
 *      elsewhere).  A chunk's record depends only on the chunk's logits, not
 *      on the rank or its memory alignment.
 *   2. the exchange (the caller's collective): every rank's records
 *      concatenated in rank order (= chunk order), and the action logits
 *      summed over ranks (exact: one rank holds each);
 *   3. grpo_vocab_loss on every rank (identical inputs, identical results):
 *      the chunks folded in order to each row's logsumexp, logp and
 *      ref_logp, then the loss as grpo_loss_fwd_bwd would form it from them
 *      (every variant, groups, sharding over sequences); lse_w receives
 *      [2][B*T] doubles: the policy logsumexp and w = dL/dlogp per row;
 *   4. grpo_vocab_grad on every rank: its slice of dL/dlogits from lse_w.
 * Any split at chunk boundaries -- one rank included -- gives the same bits
 * everywhere.  The fused grpo_loss_fwd_bwd is the faster single-rank path;
 * the two agree within the stated tolerances, not bit for bit. */
size_t grpo_vocab_chunk(void);

grpo_status_t grpo_vocab_partials(const void *policy_slice, const void *ref_slice,
                                  grpo_dtype_t dt, int64_t B, int64_t T, int64_t Vk,
                                  int64_t v_begin, const int64_t *action_ids,
                                  const uint8_t *completion_mask, void *partials_p,
                                  void *partials_r, float *action_logits, void *stream);

/* partials_p / partials_r: [num_chunks][B*T] records of all slices
 * (num_chunks = ceil(V / grpo_vocab_chunk())); action_logits: [2][B*T]
 * summed over slices; V: the whole vocabulary (action ids outside [0, V)
 * set GRPO_ERR_ACTION_RANGE).  Other arguments as for grpo_loss_fwd_bwd. */
grpo_status_t grpo_vocab_loss(const void *partials_p, const void *partials_r,
                              int64_t num_chunks, const float *action_logits, int64_t V,
                              const int64_t *action_ids, const float *old_logps,
                              const uint8_t *completion_mask, int64_t B, int64_t T,
                              const float *rewards, const grpo_groups_t *groups,
                              const grpo_params_t *params, double *lse_w, float *out3,
                              float *per_seq, float *logps_out, float *adv_out, void *ws,
                              size_t ws_bytes, void *stream);

/* grad_slice [B,T,Vk] (dtype dt, overwritten): dL/dx_v = w (1[v = a] -
 * exp(x_v - lse)) over the slice; zeros on masked rows unless flags has
 * GRPO_SKIP_MASKED_GRAD_ROWS. */
grpo_status_t grpo_vocab_grad(const void *policy_slice, grpo_dtype_t dt, int64_t B, int64_t T,
                              int64_t Vk, int64_t v_begin, const int64_t *action_ids,
                              const uint8_t *completion_mask, const double *lse_w,
                              void *grad_slice, uint32_t flags, void *stream);

/* Synchronises `stream` and returns the device status the last call on this
 * workspace left (GRPO_OK or an OR of the device-detected bits), or
 * GRPO_ERR_CUDA.  (grpo_loss_from_logps moves its status bits into a second
 * header word when its kernels end, leaving the header clean for the next
 * call; both words are read.)  The only entry point that blocks. */
grpo_status_t grpo_read_device_status(const void *ws, void *stream);

/* Static description of a status code. */
const char *grpo_status_string(grpo_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_GB300_H */
