/*
 * CPU ORACLE for speculative-decoding verification by rejection sampling.
 *
 * TEST INFRASTRUCTURE.  This file is the slow, plain, fp64 statement of what
 * the verifier computes.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code with the CUDA library (no
 * header, no helper, no table) and the library never calls it.
 *
 * Sources (web pages, by title):
 *   - Drafts are sampled from the draft distribution and accepted or rejected
 *     against the target distribution, which the protocol preserves:
 *     "Optimizing speculative decoding" and "GLM-5.2: Tuning MTP speculative
 *     decoding to the limit", section "Rejection sampling and a loss that
 *     optimizes acceptance directly", first bullet.
 *   - The per-token acceptance probability of lossless speculative sampling is
 *     sum_x min(p(x), q(x)): "Optimizing speculative decoding", section
 *     "Kimi K3".
 *   - Total variation is half the sum of absolute probability differences:
 *     "Optimizing speculative decoding", same section as the first item,
 *     second bullet.
 *   - The target verifies the whole k-token chain in one forward pass, i.e.
 *     it provides k+1 target distributions: "Optimizing speculative
 *     decoding", section "The draft model moved inside".  Accepted length
 *     tau: "DSpark for GLM-5.2", introduction.
 *   - "DSpark for GLM-5.2" cites Leviathan, Kalman and Matias (ICML 2023) as
 *     the origin of the scheme.  The pages do not print the residual
 *     distribution max(0, p - q) or the bonus draw; they are the only
 *     completion under which the target distribution is preserved and the
 *     acceptance equals sum min(p, q), and are taken in that reading.
 *
 * Readings where the pages are silent:
 *   - temperature: p = softmax(z / T) for the target and q = softmax(z / T) for
 *     the draft, the chain's T for both; T == 0 means greedy: the one-hot
 *     distribution on the lowest-index maximum.
 *   - accept: if log p(x) >= log q(x) accept; otherwise accept iff
 *     u < exp(log p(x) - log q(x)).  If q(x) == 0, accept iff p(x) > 0.
 *   - the final token uses the extra uniform u[k] (never the rejected
 *     position's uniform), by inverse CDF: y = min{ j : u * S < C_j } with
 *     C_j the inclusive running sum of the weights and S their total; if
 *     rounding leaves no such j, the largest j with positive weight.
 *   - a zero residual at a rejection (possible only through rounding) falls
 *     back to sampling from p with the same uniform.
 *   - tie flags: an accept test with |u - min(1, p/q)| < 1e-6 (0 < p/q), and a
 *     final draw with |u*S - C_j| < 1e-6*S at the chosen j or the one before,
 *     are flagged; a residual fallback is flagged too.
 *   - invalid data: a draft token outside [0, V), a temperature that is NaN,
 *     infinite or negative, or a logit row whose maximum is not finite (any
 *     NaN, any +inf, or every entry -inf) makes the chain invalid: tau = -1 and
 *     all tokens -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define SO_FP32 0
#define SO_BF16 1
#define SO_FP64 2
#define SO_TIE_BAND 1e-6

/* Exact conversion of one stored logit to double (bf16 widens exactly).
 * SO_FP64 rows exist for the tests' finite differences only; the batch
 * drivers accept fp32 and bf16. */
static double logit_at(const void* row, int dtype, int64_t j) {
  if (dtype == SO_FP64) return ((const double*)row)[j];
  if (dtype == SO_FP32) return (double)((const float*)row)[j];
  uint32_t bits = (uint32_t)((const uint16_t*)row)[j] << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* Largest logit of the row; NaN if any entry is NaN. */
static double row_max(const void* row, int dtype, int64_t V) {
  double m = -INFINITY;
  for (int64_t j = 0; j < V; ++j) {
    double z = logit_at(row, dtype, j);
    if (isnan(z)) return NAN;
    if (z > m) m = z;
  }
  return m;
}

/* Greedy (T == 0): index of the largest logit, lowest index among ties. */
int64_t so_argmax(const void* row, int dtype, int64_t V) {
  int64_t a = 0;
  double m = logit_at(row, dtype, 0);
  for (int64_t j = 1; j < V; ++j) {
    double z = logit_at(row, dtype, j);
    if (z > m) { m = z; a = j; }
  }
  return a;
}

/* Temperature softmax in log space, T > 0:
 *   l_j = z_j / T,  lse = max_j l_j + log sum_j exp(l_j - max l),
 *   logp_j = l_j - lse.
 * Returns lse, or NaN when the row's maximum is not finite. */
double so_log_softmax(const void* row, int dtype, int64_t V, double T, double* logp) {
  double zmax = row_max(row, dtype, V);
  if (!isfinite(zmax)) return NAN;
  double lmax = zmax / T;
  double s = 0.0;
  for (int64_t j = 0; j < V; ++j) s += exp(logit_at(row, dtype, j) / T - lmax);
  double lse = lmax + log(s);
  if (logp)
    for (int64_t j = 0; j < V; ++j) logp[j] = logit_at(row, dtype, j) / T - lse;
  return lse;
}

/* The distribution of one row at temperature T as probabilities (and log
 * probabilities).  Returns 0, or 1 when the row is invalid. */
static int row_distribution(const void* row, int dtype, int64_t V, double T, double* p, double* logp) {
  if (T == 0.0) {
    if (!isfinite(row_max(row, dtype, V))) return 1;
    int64_t a = so_argmax(row, dtype, V);
    for (int64_t j = 0; j < V; ++j) {
      p[j] = (j == a) ? 1.0 : 0.0;
      logp[j] = (j == a) ? 0.0 : -INFINITY;
    }
    return 0;
  }
  double lse = so_log_softmax(row, dtype, V, T, logp);
  if (isnan(lse)) return 1;
  for (int64_t j = 0; j < V; ++j) p[j] = exp(logp[j]);
  return 0;
}

/* Accept test for one drafted token x with log p(x) = lp, log q(x) = lq and
 * uniform u.  Returns 1 to accept.  *tie is set when u lies within the tie
 * band of the threshold min(1, p/q). */
int so_accept(double lp, double lq, double u, int* tie) {
  int t = 0, acc;
  if (lq == -INFINITY) {
    acc = lp > -INFINITY;
  } else if (lp >= lq) {
    acc = 1;
    t = fabs(u - 1.0) < SO_TIE_BAND;
  } else {
    double theta = exp(lp - lq);
    acc = u < theta;
    t = theta > 0.0 && fabs(u - theta) < SO_TIE_BAND;
  }
  if (tie) *tie = t;
  return acc;
}

/* Inverse-CDF draw from nonnegative weights w[0..V-1] with uniform u:
 * y = min{ j : u*S < C_j }, C_j = w_0 + ... + w_j (sequential running sum),
 * S = C_{V-1}.  If rounding leaves no such j: the largest j with w_j > 0.
 * Returns -1 when S == 0.  *tie flags |u*S - C| < 1e-6*S at the chosen
 * boundary or the one below it. */
int64_t so_sample(const double* w, int64_t V, double u, int* tie, double* total) {
  double S = 0.0;
  for (int64_t j = 0; j < V; ++j) S += w[j];
  if (total) *total = S;
  if (tie) *tie = 0;
  if (!(S > 0.0)) return -1;
  const double t = u * S;
  double C = 0.0, Cprev = 0.0;
  int64_t y = -1;
  for (int64_t j = 0; j < V; ++j) {
    Cprev = C;
    C += w[j];
    if (t < C) { y = j; break; }
  }
  if (y < 0) {
    for (int64_t j = V - 1; j >= 0; --j)
      if (w[j] > 0.0) { y = j; break; }
    if (tie) *tie = 1;
    return y;
  }
  if (tie) *tie = fabs(t - C) < SO_TIE_BAND * S || fabs(t - Cprev) < SO_TIE_BAND * S;
  return y;
}

/* One chain: inputs and outputs (caller-owned arrays). */
typedef struct {
  int64_t V;
  int32_t k;
  int32_t dtype;
  double T;
  const void* target;     /* (k+1) rows of V logits */
  const void* draft;      /* k rows of V logits */
  const int32_t* x;       /* k drafted tokens */
  const float* u;         /* k+1 uniforms: u[0..k-1] accept tests, u[k] final draw */
  int32_t want_tv;
} so_chain_in;

typedef struct {
  int32_t* tokens;        /* k+1: accepted drafts, then the residual/bonus token, then -1 */
  int32_t tau;            /* accepted drafts 0..k, or -1 for an invalid chain */
  double* p_draft;        /* k: p_i(x_i) for every position */
  double* q_draft;        /* k: q_i(x_i) for every position */
  double* tv;             /* k: 0.5 * sum_j |p_i(j) - q_i(j)| for every position (if want_tv) */
  int32_t* accept_tie;    /* k: tie flag of each accept test taken (0 where not taken) */
  int32_t cdf_tie;        /* final draw flagged (boundary band, overrun or residual fallback) */
  int32_t residual_fallback;
  double residual_mass;   /* S of the residual at the rejection (or 1 for the bonus) */
} so_chain_out;

static void invalidate(const so_chain_in* in, so_chain_out* out) {
  out->tau = -1;
  for (int32_t i = 0; i <= in->k; ++i) out->tokens[i] = -1;
}

/* Verification of one chain by rejection sampling.  Returns 0, or 1 when the
 * chain's data is invalid (then tau = -1). */
int so_verify_chain(const so_chain_in* in, so_chain_out* out) {
  const int64_t V = in->V;
  const int32_t k = in->k;
  const size_t rs = (size_t)V * (in->dtype == SO_FP32 ? 4 : 2);
  out->cdf_tie = 0;
  out->residual_fallback = 0;
  out->residual_mass = 0.0;
  for (int32_t i = 0; i < k; ++i) {
    out->accept_tie[i] = 0;
    out->p_draft[i] = NAN;
    out->q_draft[i] = NAN;
    if (out->tv) out->tv[i] = NAN;
  }
  if (!(in->T >= 0.0) || !isfinite(in->T)) { invalidate(in, out); return 1; }
  for (int32_t i = 0; i < k; ++i)
    if (in->x[i] < 0 || (int64_t)in->x[i] >= V) { invalidate(in, out); return 1; }

  double* p = (double*)malloc((size_t)V * sizeof(double));
  double* q = (double*)malloc((size_t)V * sizeof(double));
  double* lp = (double*)malloc((size_t)V * sizeof(double));
  double* lq = (double*)malloc((size_t)V * sizeof(double));
  double* w = (double*)malloc((size_t)V * sizeof(double));
  int bad = 0;
  int32_t tau = -1;          /* -1: no rejection yet */
  int64_t y = -1;

  /* Every position is evaluated so that p_draft, q_draft and tv exist for all
   * k positions; the accept test runs only until the first rejection. */
  for (int32_t i = 0; i < k && !bad; ++i) {
    const void* trow = (const char*)in->target + (size_t)i * rs;
    const void* drow = (const char*)in->draft + (size_t)i * rs;
    if (row_distribution(trow, in->dtype, V, in->T, p, lp) ||
        row_distribution(drow, in->dtype, V, in->T, q, lq)) { bad = 1; break; }
    const int32_t x = in->x[i];
    out->p_draft[i] = p[x];
    out->q_draft[i] = q[x];
    if (in->want_tv && out->tv) {
      double s = 0.0;
      for (int64_t j = 0; j < V; ++j) s += fabs(p[j] - q[j]);
      out->tv[i] = 0.5 * s;
    }
    if (tau < 0) {
      int tie = 0;
      int acc = so_accept(lp[x], lq[x], (double)in->u[i], &tie);
      if (in->T == 0.0) tie = 0;     /* greedy decisions are exact comparisons */
      out->accept_tie[i] = tie;
      if (!acc) {
        tau = i;
        /* residual distribution at the rejected position: max(0, p - q) */
        for (int64_t j = 0; j < V; ++j) w[j] = p[j] > q[j] ? p[j] - q[j] : 0.0;
        int ctie = 0;
        y = so_sample(w, V, (double)in->u[k], &ctie, &out->residual_mass);
        if (y < 0) {
          /* zero residual (rounding only): sample from p with the same uniform */
          y = so_sample(p, V, (double)in->u[k], &ctie, NULL);
          out->residual_fallback = 1;
          ctie = 1;
        }
        if (in->T == 0.0) ctie = 0;
        out->cdf_tie = ctie;
      }
    }
  }
  if (!bad && tau < 0) {
    /* every draft accepted: bonus token from the last target row */
    const void* trow = (const char*)in->target + (size_t)k * rs;
    if (row_distribution(trow, in->dtype, V, in->T, p, lp)) {
      bad = 1;
    } else {
      tau = k;
      int ctie = 0;
      y = so_sample(p, V, (double)in->u[k], &ctie, &out->residual_mass);
      if (in->T == 0.0) ctie = 0;
      out->cdf_tie = ctie;
    }
  } else if (!bad) {
    /* the bonus row must still be a valid distribution */
    const void* trow = (const char*)in->target + (size_t)k * rs;
    if (!isfinite(row_max(trow, in->dtype, V))) bad = 1;
  }
  free(p); free(q); free(lp); free(lq); free(w);
  if (bad || y < 0) { invalidate(in, out); return 1; }
  out->tau = tau;
  for (int32_t i = 0; i < tau; ++i) out->tokens[i] = in->x[i];
  out->tokens[tau] = (int32_t)y;
  for (int32_t i = tau + 1; i <= k; ++i) out->tokens[i] = -1;
  return 0;
}

/* Entropy, in nats, of one row's distribution at temperature T:
 *   H = -sum_j p_j log p_j,  p = softmax(z / T).
 * The pages tie acceptance degradation to fluctuations in the entropy of the
 * model's output, i.e. in how widely its probability mass is spread
 * ("Optimizing speculative decoding" and "GLM-5.2: Tuning MTP speculative
 * decoding to the limit", section "Rejection sampling and a loss that
 * optimizes acceptance directly"); they print no formula, and Shannon entropy of the distribution
 * the verifier uses is the reading.  Entries with p_j = 0 (logit -inf) add
 * nothing (0 log 0 = 0).  T == 0: the greedy one-hot distribution, H = 0.
 * NaN for a temperature that is NaN, infinite or negative, or a row whose
 * maximum is not finite. */
double so_entropy(const void* row, int dtype, int64_t V, double T) {
  if (!(T >= 0.0) || isinf(T)) return NAN;
  if (!isfinite(row_max(row, dtype, V))) return NAN;
  if (T == 0.0) return 0.0;
  double lse = so_log_softmax(row, dtype, V, T, NULL);
  double h = 0.0;
  for (int64_t j = 0; j < V; ++j) {
    double lp = logit_at(row, dtype, j) / T - lse;
    if (lp > -INFINITY) h -= exp(lp) * lp;
  }
  return h;
}

/* Entropies of every target row [B, k+1] and draft row [B, k] of a batch,
 * each row with its chain's temperature (rows split over threads). */
typedef struct {
  int64_t B, V;
  int32_t k, dtype;
  const void* target; const void* draft; const float* T;
  double* ent_t; double* ent_d;
  int64_t first, stride;
} so_entropy_job;

static void* entropy_worker(void* arg) {
  so_entropy_job* J = (so_entropy_job*)arg;
  const size_t rs = (size_t)J->V * (J->dtype == SO_FP32 ? 4 : 2);
  const int64_t rows = J->B * (2 * (int64_t)J->k + 1);
  for (int64_t r = J->first; r < rows; r += J->stride) {
    const int64_t b = r / (2 * J->k + 1), i = r % (2 * J->k + 1);
    const double T = (double)J->T[b];
    if (i <= J->k)
      J->ent_t[b * (J->k + 1) + i] = so_entropy((const char*)J->target + (size_t)(b * (J->k + 1) + i) * rs, J->dtype, J->V, T);
    else
      J->ent_d[b * J->k + (i - J->k - 1)] =
          so_entropy((const char*)J->draft + (size_t)(b * J->k + (i - J->k - 1)) * rs, J->dtype, J->V, T);
  }
  return NULL;
}

int so_entropy_batch(int64_t B, int32_t k, int64_t V, int32_t dtype, const void* target, const void* draft,
                     const float* T, double* ent_t, double* ent_d, int nthreads) {
  if (B < 0 || k < 1 || V < 1 || (dtype != SO_FP32 && dtype != SO_BF16)) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  so_entropy_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) jobs[t] = (so_entropy_job){B, V, k, dtype, target, draft, T, ent_t, ent_d, t, nthreads};
  if (nthreads == 1) { entropy_worker(&jobs[0]); return 0; }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, entropy_worker, &jobs[t]) != 0) break;
    started++;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = started; t < nthreads; ++t) entropy_worker(&jobs[t]);
  return 0;
}

/* Losses on the draft-target overlap, and their gradient with respect to the
 * draft logits (the target is frozen).  For one position with target row zt,
 * draft row zd and temperature T > 0, p = softmax(zt / T), q = softmax(zd / T):
 *   alpha = sum_x min(p(x), q(x)), the probability that the protocol accepts
 *           the drafted token ("Optimizing speculative decoding", section
 *           "Kimi K3"), = 1 - TV;
 *   kind 0, TV loss:       l = TV = 1 - alpha  ("Optimizing speculative
 *           decoding" and "GLM-5.2: Tuning MTP speculative decoding to the
 *           limit", section "Rejection sampling and a loss that optimizes
 *           acceptance directly", second bullet; per position is the reading);
 *   kind 1, overlap loss:  l = -ln alpha  ("Optimizing speculative decoding",
 *           section "Kimi K3": the negative log of the draft-target overlap).
 * With weight w the position contributes w * l to the loss, and
 *   d(w l)/d zd_m = w * dl/dalpha * (q_m / T) * ([q_m < p_m] - beta),
 *   beta = sum_x [q_x < p_x] q_x,
 * since d min(p_x, q_x)/d q_x = [q_x < p_x] (the strict side at a tie) and
 * d q_x / d zd_m = q_x (delta_xm - q_m) / T.  dl/dalpha is -1 (TV) or
 * -1/alpha (overlap).  `tie` returns the draft mass of the entries with
 * |p - q| <= 1e-6 * max(p, q), where that subgradient choice is arbitrary.
 * Returns 0, or 1 (loss NaN, gradient 0) for T <= 0 or not finite, or a row
 * whose maximum is not finite. */
int so_overlap_grad(const void* trow, const void* drow, int dtype, int64_t V, double T, int kind, double w,
                    double* loss, double* alpha_out, double* grad, double* tie) {
  *loss = NAN;
  *alpha_out = NAN;
  *tie = 0.0;
  for (int64_t j = 0; j < V; ++j) grad[j] = 0.0;
  if (!(T > 0.0) || isinf(T)) return 1;
  double* lp = (double*)malloc(sizeof(double) * (size_t)V);
  double* lq = (double*)malloc(sizeof(double) * (size_t)V);
  if (!lp || !lq) { free(lp); free(lq); return 1; }
  int bad = isnan(so_log_softmax(trow, dtype, V, T, lp)) || isnan(so_log_softmax(drow, dtype, V, T, lq));
  if (!bad) {
    double alpha = 0.0, beta = 0.0, tie_mass = 0.0;
    for (int64_t j = 0; j < V; ++j) {
      const double pj = exp(lp[j]), qj = exp(lq[j]);
      alpha += pj < qj ? pj : qj;
      if (qj < pj) beta += qj;
      const double hi = pj > qj ? pj : qj;
      if (hi > 0.0 && fabs(pj - qj) <= SO_TIE_BAND * hi) tie_mass += qj;
    }
    const double dl = kind == 0 ? -1.0 : -1.0 / alpha;
    *alpha_out = alpha;
    *loss = kind == 0 ? 1.0 - alpha : -log(alpha);
    *tie = tie_mass;
    for (int64_t j = 0; j < V; ++j) {
      const double pj = exp(lp[j]), qj = exp(lq[j]);
      grad[j] = w * dl * (qj / T) * ((qj < pj ? 1.0 : 0.0) - beta);
    }
  }
  free(lp);
  free(lq);
  return bad;
}

/* The losses and draft-logit gradients of a batch: position i of chain b uses
 * target row i and draft row i, weights w [B, k] (NULL: all 1).  Outputs
 * loss, alpha, tie [B, k] and grad [B, k, V] (fp64). */
typedef struct {
  int64_t B, V;
  int32_t k, dtype, kind;
  const void* target; const void* draft; const float* T; const float* w;
  double* loss; double* alpha; double* grad; double* tie;
  int64_t first, stride;
} so_grad_job;

static void* grad_worker(void* arg) {
  so_grad_job* J = (so_grad_job*)arg;
  const size_t rs = (size_t)J->V * (J->dtype == SO_FP32 ? 4 : 2);
  for (int64_t r = J->first; r < J->B * J->k; r += J->stride) {
    const int64_t b = r / J->k, i = r % J->k;
    so_overlap_grad((const char*)J->target + (size_t)(b * (J->k + 1) + i) * rs,
                    (const char*)J->draft + (size_t)(b * J->k + i) * rs, J->dtype, J->V, (double)J->T[b], J->kind,
                    J->w ? (double)J->w[r] : 1.0, &J->loss[r], &J->alpha[r], J->grad + (size_t)r * (size_t)J->V,
                    &J->tie[r]);
  }
  return NULL;
}

int so_overlap_grad_batch(int64_t B, int32_t k, int64_t V, int32_t dtype, const void* target, const void* draft,
                          const float* T, int32_t kind, const float* w, double* loss, double* alpha, double* grad,
                          double* tie, int nthreads) {
  if (B < 0 || k < 1 || V < 1 || (dtype != SO_FP32 && dtype != SO_BF16) || (kind != 0 && kind != 1)) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  so_grad_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t)
    jobs[t] = (so_grad_job){B, V, k, dtype, kind, target, draft, T, w, loss, alpha, grad, tie, t, nthreads};
  if (nthreads == 1) { grad_worker(&jobs[0]); return 0; }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, grad_worker, &jobs[t]) != 0) break;
    started++;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = started; t < nthreads; ++t) grad_worker(&jobs[t]);
  return 0;
}

/* ---- batch driver (chains statically partitioned over threads) ------ */
typedef struct {
  int64_t B, V;
  int32_t k, dtype, want_tv;
  const void* target; const void* draft;
  const int32_t* x; const float* T; const float* u;
  int32_t* tokens; int32_t* tau;
  double* p_draft; double* q_draft; double* tv;
  int32_t* accept_tie; int32_t* cdf_tie; int32_t* fallback; double* mass;
  int64_t first, stride;
} so_batch_job;

static void* batch_worker(void* arg) {
  so_batch_job* J = (so_batch_job*)arg;
  const size_t rs = (size_t)J->V * (J->dtype == SO_FP32 ? 4 : 2);
  const int32_t k = J->k;
  for (int64_t b = J->first; b < J->B; b += J->stride) {
    so_chain_in in = {J->V, k, J->dtype, (double)J->T[b],
                      (const char*)J->target + (size_t)b * (size_t)(k + 1) * rs,
                      (const char*)J->draft + (size_t)b * (size_t)k * rs,
                      J->x + b * k, J->u + b * (k + 1), J->want_tv};
    so_chain_out out = {J->tokens + b * (k + 1), 0, J->p_draft + b * k, J->q_draft + b * k,
                        J->tv ? J->tv + b * k : NULL, J->accept_tie + b * k, 0, 0, 0.0};
    so_verify_chain(&in, &out);
    J->tau[b] = out.tau;
    J->cdf_tie[b] = out.cdf_tie;
    J->fallback[b] = out.residual_fallback;
    J->mass[b] = out.residual_mass;
  }
  return NULL;
}

int so_verify_batch(int64_t B, int32_t k, int64_t V, int32_t dtype, const void* target, const void* draft,
                    const int32_t* x, const float* T, const float* u, int32_t want_tv,
                    int32_t* tokens, int32_t* tau, double* p_draft, double* q_draft, double* tv,
                    int32_t* accept_tie, int32_t* cdf_tie, int32_t* fallback, double* mass, int nthreads) {
  if (B < 0 || k < 1 || V < 1 || (dtype != SO_FP32 && dtype != SO_BF16)) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > B) nthreads = (int)(B > 0 ? B : 1);
  so_batch_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t)
    jobs[t] = (so_batch_job){B, V, k, dtype, want_tv, target, draft, x, T, u, tokens, tau, p_draft, q_draft,
                             want_tv ? tv : NULL, accept_tie, cdf_tie, fallback, mass, t, nthreads};
  if (nthreads == 1) { batch_worker(&jobs[0]); return 0; }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, batch_worker, &jobs[t]) != 0) break;
    started++;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = started; t < nthreads; ++t) batch_worker(&jobs[t]);
  return 0;
}
