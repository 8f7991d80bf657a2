/*
 * oracle.c -- TEST INFRASTRUCTURE.  A plain, slow, double-precision CPU
 * statement of the GRPO loss forward + backward, written from the operator
 * descriptions; it exists only to check the CUDA library against.  Only the
 * test-suite, the smoke check and the CPU-baseline leg of the benchmark load
 * it.  It shares no code with the CUDA library.
 *
 * Sources (page title, section):
 *   [RK]  RL-Kernel "GRPO Loss" operator page: "Accuracy" (reference
 *         semantics of NativeGRPOLossOp), "Tensor Contract", "Group
 *         specification", "Normalizer semantics", "Tensor and Data Parallel".
 *   [DY]  dockyard_rl "GRPO and the clipped policy-gradient loss": "One loss,
 *         many algorithms" (asymmetric clip eps_lo / eps_hi), "Advantage
 *         estimation" (degenerate group -> zero advantage), "Reference-KL
 *         penalty" (k3 estimator).
 *   [RX]  Relax "REINFORCE++ / REINFORCE++-baseline": "Notation and mask
 *         contract" (boolean mask selection), "PPO and KL reduction"
 *         (response mean).
 *   [GC]  grpo.cpp README, "The length-normalization detail" (token mean vs
 *         sequence mean weights) and "CUDA" (fused logits boundary:
 *         dL/dlogits = w (onehot - softmax)).
 *
 * Readings where the pages leave a step open (all stated in the design
 * notes): population std floored at adv_eps (or std + adv_eps on request);
 * a group whose rewards are all equal gets advantage exactly 0; k3 is
 * e^d - d - 1 with d = ref_logp - logp, and its gradient is the pathwise
 * derivative of that formula; empty denominators are clamped to 1; the
 * sequence mean averages over sequences with at least one active token; at
 * r exactly on a clip bound the unclipped branch's gradient is taken.
 *
 * Everything is double.  Inputs are the exact stored values (f32, bf16 or
 * f16 bits are widened exactly; dtype 3 is double, used by the
 * finite-difference checks).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_F64 = 3 };

/* ---------------------------------------------------------------- storage */
static double or_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exp = (h >> 10) & 0x1F;
  int man = h & 0x3FF;
  double v;
  if (exp == 0)
    v = ldexp((double)man, -24); /* subnormal: man * 2^-24 */
  else if (exp == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexp((double)(man | 0x400), exp - 25);
  return sign ? -v : v;
}

static double or_load(const void *p, int dtype, int64_t i) {
  switch (dtype) {
  case OR_F32:
    return (double)((const float *)p)[i];
  case OR_BF16: {
    uint32_t u = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  case OR_F16:
    return or_half_to_double(((const uint16_t *)p)[i]);
  default:
    return ((const double *)p)[i];
  }
}

/* Round a double to a binary format with `prec` significant bits, smallest
 * normal exponent `emin` (value 2^emin) and largest finite `maxv`, to
 * nearest, ties to even.  nearbyint() rounds to nearest-even in the default
 * rounding mode. */
static double or_round_fmt(double x, int prec, int emin, double maxv) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(fabs(x), &e); /* |x| in [2^(e-1), 2^e) */
  int ex = e - 1;
  if (ex < emin) ex = emin; /* subnormal range: fixed quantum */
  double q = ldexp(1.0, ex - (prec - 1));
  double r = nearbyint(x / q) * q;
  if (fabs(r) > maxv) r = copysign(INFINITY, x);
  return r;
}

static void or_store(void *p, int dtype, int64_t i, double x) {
  switch (dtype) {
  case OR_F32:
    ((float *)p)[i] = (float)x;
    break;
  case OR_BF16: {
    float f = (float)or_round_fmt(x, 8, -126, 3.3895313892515355e38);
    uint32_t u;
    memcpy(&u, &f, 4);
    ((uint16_t *)p)[i] = (uint16_t)(u >> 16); /* exact: f has 8 significant bits */
    break;
  }
  case OR_F16: {
    double r = or_round_fmt(x, 11, -14, 65504.0);
    uint16_t s = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    uint16_t h;
    if (isinf(a))
      h = 0x7C00;
    else if (isnan(a))
      h = 0x7E00;
    else if (a < ldexp(1.0, -14))
      h = (uint16_t)(a / ldexp(1.0, -24)); /* subnormal: exact multiple */
    else {
      int e;
      double m = frexp(a, &e); /* a = m 2^e, m in [0.5,1) */
      h = (uint16_t)(((e - 1 + 15) << 10) | ((uint16_t)(m * 2048.0) & 0x3FF));
    }
    ((uint16_t *)p)[i] = s | h;
    break;
  }
  default:
    ((double *)p)[i] = x;
  }
}

/* ------------------------------------------------------ group advantages
 * [RK] "Accuracy": adv = (r - mean_g) / std_g(unbiased=False).clamp_min(eps),
 * over the groups of [RK] "Group specification" (uniform samples_per_prompt
 * or CSR group_boundaries [0, ..., B]).  [DY] "Advantage estimation": a
 * degenerate group (all rewards equal) has zero advantage -- taken literally
 * as A = 0 exactly.  eps_add != 0 gives the std + eps variant.
 * Returns 0, 1 (bad boundaries) or 2 (non-finite reward). */
int oracle_group_advantages(const float *rewards, int64_t B, const int64_t *bounds,
                            int64_t G, double adv_eps, int eps_add, double *A) {
  if (G < 0 || (B > 0 && G < 1)) return 1;
  if (G >= 1 && (bounds[0] != 0 || bounds[G] != B)) return 1;
  for (int64_t g = 0; g < G; ++g)
    if (bounds[g + 1] <= bounds[g]) return 1;
  for (int64_t i = 0; i < B; ++i)
    if (!isfinite((double)rewards[i])) return 2;
  for (int64_t g = 0; g < G; ++g) {
    int64_t lo = bounds[g], hi = bounds[g + 1];
    double n = (double)(hi - lo);
    double sum = 0.0, mx = -INFINITY, mn = INFINITY;
    for (int64_t i = lo; i < hi; ++i) {
      double r = (double)rewards[i];
      sum += r;
      if (r > mx) mx = r;
      if (r < mn) mn = r;
    }
    double mean = sum / n;
    double ss = 0.0;
    for (int64_t i = lo; i < hi; ++i) {
      double d = (double)rewards[i] - mean;
      ss += d * d;
    }
    double sd = sqrt(ss / n); /* population std */
    double den = eps_add ? sd + adv_eps : (sd > adv_eps ? sd : adv_eps);
    for (int64_t i = lo; i < hi; ++i)
      A[i] = (mx == mn) ? 0.0 : ((double)rewards[i] - mean) / den;
  }
  return 0;
}

/* -------------------------------------------------------- log-softmax row
 * log pi(a) = x_a - logsumexp(x) with logsumexp = M + log(sum_v exp(x_v - M)),
 * M = max_v x_v; the sum is Neumaier-compensated.  ([RK] intro: per-token
 * ratio / KL come from the log-softmax of the vocabulary row; [GC] "CUDA":
 * the row maximum and normaliser.)  lse[r] for every row; logp[r] =
 * x[r, actions[r]] - lse[r] when actions is given. */
void oracle_log_softmax_rows(const void *rows, int dtype, int64_t nrows, int64_t V,
                             const int64_t *actions, double *lse, double *logp) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t base = r * V;
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
      double x = or_load(rows, dtype, base + v);
      if (x > M || isnan(x)) M = x;
    }
    double s = 0.0, c = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      double t = exp(or_load(rows, dtype, base + v) - M);
      double u = s + t;
      if (fabs(s) >= fabs(t))
        c += (s - u) + t;
      else
        c += (t - u) + s;
      s = u;
    }
    double L = M + log(s + c);
    lse[r] = L;
    if (actions) logp[r] = or_load(rows, dtype, base + actions[r]) - L;
  }
}

/* ------------------------------------------------ vocabulary-parallel rows
 * RL-Kernel "GRPO Loss", "Tensor and Data Parallel" step 1 (the
 * vocab-parallel logprob): a rank holding the vocabulary slice [v0, v1)
 * reduces its part of a row to a partial normaliser (M_k, Z_k), M_k the
 * slice maximum and Z_k = sum_{v in slice} exp(x_v - M_k); the row's
 * logsumexp is M + log(sum_k Z_k exp(M_k - M)) with M = max_k M_k (an empty
 * slice has M_k = -inf and contributes nothing).  Partials are computed per
 * row for the slice; merge folds K partials per row in slice order. */
void oracle_lse_partial(const void *rows, int dtype, int64_t nrows, int64_t V, int64_t v0,
                        int64_t v1, double *M_out, double *Z_out) {
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t base = r * V;
    double M = -INFINITY;
    for (int64_t v = v0; v < v1; ++v) {
      double x = or_load(rows, dtype, base + v);
      if (x > M || isnan(x)) M = x;
    }
    double s = 0.0, c = 0.0;
    if (M != -INFINITY)
      for (int64_t v = v0; v < v1; ++v) {
        double t = exp(or_load(rows, dtype, base + v) - M);
        double u = s + t;
        if (fabs(s) >= fabs(t))
          c += (s - u) + t;
        else
          c += (t - u) + s;
        s = u;
      }
    M_out[r] = M;
    Z_out[r] = s + c;
  }
}

void oracle_lse_merge(int64_t nrows, int64_t K, const double *M, const double *Z,
                      double *lse) {
  for (int64_t r = 0; r < nrows; ++r) {
    double Mx = -INFINITY;
    for (int64_t k = 0; k < K; ++k)
      if (M[k * nrows + r] > Mx) Mx = M[k * nrows + r];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
      if (M[k * nrows + r] != -INFINITY) s += Z[k * nrows + r] * exp(M[k * nrows + r] - Mx);
    lse[r] = Mx + log(s);
  }
}

/* ------------------------------------------------------------ token loss
 * Per active token (mask != 0; masked tokens are never read, [RX] "Notation
 * and mask contract"):
 *   ratio  r = exp(logp - old)                          [RK] "Accuracy"
 *   policy p = -min(r A, clip(r, 1 - eps_lo, 1 + eps_hi) A)   [RK], [DY]
 *   k3     k = e^d - d - 1 = expm1(d) - d, d = ref - logp     [DY] KL penalty
 * Weights c_it ([RK] "Normalizer semantics"; [GC] length-normalization table):
 *   token mean (0):     1 / max(N, 1),          N = number of active tokens
 *   sequence mean (1):  1 / (max(S, 1) * L_i),  S = sequences with L_i > 0
 *   fixed constant (2): 1 / C for a declared C > 0 (the Dr.GRPO form, [RK]
 *                       "Normalizer semantics", fixed_constant mode)
 *   policy_loss = sum c p, kl = sum c k, loss = policy_loss + beta kl.
 * Reduction as two nested sums ([RK] "Tensor and Data Parallel", step 3):
 * token slots -> per-sequence totals (P_i, K_i) -> the scalar.
 * Gradient w.r.t. logp (the logps-only boundary's output):
 *   w = grad_scale * c * (g_pol + beta g_kl),
 *   g_pol = 0 if (A > 0 and r > 1 + eps_hi) or (A < 0 and r < 1 - eps_lo),
 *           else -A r;
 *   g_kl  = d k / d logp = 1 - e^d = -expm1(d).
 *
 * Variants ([DY] "One loss, many algorithms", "CISPO", "Reference-KL
 * penalty"; [RX] "REINFORCE++" and "REINFORCE++-baseline"):
 *   kl_type 1, k1 (the log ratio):  k = logp - ref = -d,  g_kl = 1
 *   kl_type 2, k2:                  k = (logp - ref)^2 / 2 = d^2 / 2,
 *                                   g_kl = logp - ref = -d
 *   dual clip c > 1 (A < 0 only: a floor under the objective of tokens
 *     with negative advantage):  p = -max(min(r A, clip(r) A), c A), which for A < 0 is
 *     -A min(max(r, 1 - eps_lo), c); g_pol is also 0 where r > c.
 *   surrogate 1, CISPO:  p = -A sg(clip(r)) logp, so g_pol = -A clip(r)
 *     (the clipped weight sits behind a stop-gradient; every token keeps a
 *     gradient through logp).  Not combined with the dual clip.
 *   sequence-level ratio (seq_ratio 1, GSPO; Relax "REINFORCE++ /
 *     REINFORCE++-baseline" algorithm table, and dockyard_rl
 *     "sequence_level_importance_ratios"): every active token of sequence i
 *     uses rho_i = exp((1/L_i) sum_t (logp - old)) in place of its own r,
 *     then the clipped surrogate; the policy gradient of token t is
 *     d/dlogp_it of the sequence-mean loss, c_it (-A rho_i) (0 when rho_i is
 *     clipped), because each of the L_i equal terms carries rho_i / L_i.
 *     Sequence mean only (the page rejects the global-token reduction).
 * Clip counters (counts, nullable, [3]): tokens clipped at the upper bound,
 * at the lower bound, and by the dual clip.  For the clipped surrogate the
 * first two are (A > 0 and r > 1 + eps_hi) and (A < 0 and r < 1 - eps_lo) --
 * the tokens whose policy gradient the clip removes; for CISPO they are the
 * tokens whose weight clip(r) differs from r (r > 1 + eps_hi, r < 1 - eps_lo).
 *
 * ref_logp may be NULL: the KL term is then 0.
 * out3 = {loss, policy_loss, kl}; per_seq = [P (B) | K (B) | L (B)];
 * w, ratio (nullable) are [B,T] with 0 on masked tokens. */
void oracle_loss_from_logps(int64_t B, int64_t T, const double *logp,
                            const double *ref_logp, const double *old,
                            const uint8_t *mask, const double *A, double eps_lo,
                            double eps_hi, double beta, double grad_scale,
                            int reduction, int kl_type, int surrogate, double dual_c,
                            double norm_const, int seq_ratio, double *out3, double *per_seq,
                            double *w, double *ratio, int64_t *counts) {
  double *P = per_seq, *K = per_seq + B, *Ls = per_seq + 2 * B;
  int64_t N = 0, S = 0;
  int64_t n_hi = 0, n_lo = 0, n_dual = 0;
  for (int64_t i = 0; i < B; ++i) {
    int64_t L = 0;
    for (int64_t t = 0; t < T; ++t)
      if (mask[i * T + t]) ++L;
    Ls[i] = (double)L;
    N += L;
    if (L > 0) ++S;
  }
  for (int64_t i = 0; i < B; ++i) {
    double Pi = 0.0, Ki = 0.0;
    double c;
    if (reduction == 0)
      c = 1.0 / (double)(N > 0 ? N : 1);
    else if (reduction == 1)
      c = Ls[i] > 0 ? 1.0 / ((double)(S > 0 ? S : 1) * Ls[i]) : 0.0;
    else
      c = 1.0 / norm_const;
    double rho = 1.0; /* GSPO: the sequence's ratio */
    if (seq_ratio && Ls[i] > 0) {
      double s = 0.0;
      for (int64_t t = 0; t < T; ++t)
        if (mask[i * T + t]) s += logp[i * T + t] - old[i * T + t];
      rho = exp(s / Ls[i]);
    }
    for (int64_t t = 0; t < T; ++t) {
      int64_t j = i * T + t;
      if (!mask[j]) {
        if (w) w[j] = 0.0;
        if (ratio) ratio[j] = 0.0;
        continue;
      }
      double r = seq_ratio ? rho : exp(logp[j] - old[j]);
      double a = A[i];
      double rc = r < 1.0 - eps_lo ? 1.0 - eps_lo : (r > 1.0 + eps_hi ? 1.0 + eps_hi : r);
      double p, gpol;
      if (surrogate == 1) { /* CISPO */
        p = -a * rc * logp[j];
        gpol = -a * rc;
        if (r > 1.0 + eps_hi) ++n_hi;
        if (r < 1.0 - eps_lo) ++n_lo;
      } else {
        double unclipped = r * a;
        double clipped = rc * a;
        double obj = unclipped < clipped ? unclipped : clipped;
        int hi = a > 0.0 && r > 1.0 + eps_hi;
        int lo = a < 0.0 && r < 1.0 - eps_lo;
        int dual = dual_c > 0.0 && a < 0.0 && r > dual_c;
        if (dual_c > 0.0 && a < 0.0 && dual_c * a > obj) obj = dual_c * a;
        p = -obj;
        gpol = (hi || lo || dual) ? 0.0 : -a * r;
        n_hi += hi;
        n_lo += lo;
        n_dual += dual;
      }
      double d = ref_logp ? ref_logp[j] - logp[j] : 0.0;
      double k, gkl;
      if (kl_type == 1) {
        k = -d;
        gkl = 1.0;
      } else if (kl_type == 2) {
        k = 0.5 * d * d;
        gkl = -d;
      } else {
        k = expm1(d) - d;
        gkl = -expm1(d);
      }
      if (!ref_logp) {
        k = 0.0;
        gkl = 0.0;
      }
      Pi += p;
      Ki += k;
      if (w) w[j] = grad_scale * c * (gpol + beta * gkl);
      if (ratio) ratio[j] = r;
    }
    P[i] = Pi;
    K[i] = Ki;
  }
  double pol = 0.0, kl = 0.0;
  if (reduction == 0 || reduction == 2) {
    double n = reduction == 0 ? (double)(N > 0 ? N : 1) : norm_const;
    for (int64_t i = 0; i < B; ++i) {
      pol += P[i];
      kl += K[i];
    }
    pol /= n;
    kl /= n;
  } else {
    double s = (double)(S > 0 ? S : 1);
    for (int64_t i = 0; i < B; ++i)
      if (Ls[i] > 0) {
        pol += P[i] / Ls[i];
        kl += K[i] / Ls[i];
      }
    pol /= s;
    kl /= s;
  }
  out3[0] = pol + beta * kl;
  out3[1] = pol;
  out3[2] = kl;
  if (counts) {
    counts[0] = n_hi;
    counts[1] = n_lo;
    counts[2] = n_dual;
  }
}

/* -------------------------------------------------------- gradient rows
 * dL/dx_v = w (1[v = a] - exp(x_v - lse)) for one active row ([GC] "CUDA":
 * the fused kernel writes the full logits gradient; d logp / d x_v =
 * 1[v=a] - softmax_v).  Written rounded to out_dtype (nearest-even) and,
 * when out_f64 is given, unrounded. */
void oracle_grad_rows(const void *rows, int dtype, int64_t nrows, int64_t V,
                      const int64_t *actions, const double *lse, const double *w,
                      int out_dtype, void *out, double *out_f64) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t base = r * V;
    for (int64_t v = 0; v < V; ++v) {
      double sm = exp(or_load(rows, dtype, base + v) - lse[r]);
      double g = w[r] * ((v == actions[r] ? 1.0 : 0.0) - sm);
      if (out) or_store(out, out_dtype, base + v, g);
      if (out_f64) out_f64[base + v] = g;
    }
  }
}

/* Round doubles to a storage dtype (used by tests to build rounded
 * expectations and ulp tables). */
void oracle_round_to(const double *x, int64_t n, int dtype, void *out) {
  for (int64_t i = 0; i < n; ++i) or_store(out, dtype, i, x[i]);
}
