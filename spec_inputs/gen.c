/*
 * Seeded synthetic inputs for speculative-decoding verification.
 *
 * This file holds only input generation: a counter-based random number
 * generator, normal variates, bf16 rounding and Gumbel-max draft-token
 * sampling.  It contains none of the verification arithmetic (no softmax, no
 * acceptance test, no residual, no total-variation distance), so the CPU oracle
 * and the CUDA library can both consume its output without sharing any of the
 * method's code.
 *
 * Random numbers: Philox4x32-10, from Salmon, Moraes, Dror and Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4 (the Philox
 * S-box: two 32x32->64 multiplications per round, Weyl key schedule).
 * Key = (seed_lo, seed_hi).  A draw is addressed by (stream, row, column):
 * counter = (column / 4, row, stream, 0), and word column % 4 of the output.
 * A uniform is u = (word >> 8) * 2^-24, exactly representable in fp32.
 *
 * Streams: 0 target normals, 1 draft noise (or independent draft normals),
 * 2 Gumbel noise for draft-token sampling, 3 verification uniforms,
 * 4 boosted-token picks, 5 per-chain temperatures.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define SG_FP32 0
#define SG_BF16 1

enum { ST_TARGET = 0, ST_DRAFT = 1, ST_GUMBEL = 2, ST_VERIFY = 3, ST_BOOST = 4, ST_TEMP = 5 };

/* ---- Philox4x32-10 (Salmon et al., SC'11, section 4.1) ---------------- */
static void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)M0 * c0;
    uint64_t p1 = (uint64_t)M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0; k1 += W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

void sg_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  philox4x32_10(ctr, key, out);
}

static void block4(uint64_t seed, uint32_t stream, uint64_t row, uint64_t col4, uint32_t w[4]) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)col4, (uint32_t)row, stream, (uint32_t)(row >> 32)};
  philox4x32_10(ctr, key, w);
}

static uint32_t word_at(uint64_t seed, uint32_t stream, uint64_t row, uint64_t col) {
  uint32_t w[4];
  block4(seed, stream, row, col >> 2, w);
  return w[col & 3];
}

/* u in [0, 1) on the 2^-24 lattice */
float sg_uniform(uint64_t seed, uint32_t stream, uint64_t row, uint64_t col) {
  return (float)(word_at(seed, stream, row, col) >> 8) * (1.0f / 16777216.0f);
}

/* ---- bf16 round-to-nearest-even from fp32 --------------------------- */
static uint16_t f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}
static float bf16_to_f32(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}
uint16_t sg_f32_to_bf16(float f) { return f32_to_bf16(f); }

/* ---- standard normals: Box-Muller on pairs of lattice uniforms ------- */
/* Normal number `col` of (stream, row): counter col/4 gives four words; words
 * (0,1) make normals 0 and 1 of the block, words (2,3) make normals 2 and 3. */
static void normals4(uint64_t seed, uint32_t stream, uint64_t row, uint64_t col4, double n[4]) {
  uint32_t w[4];
  block4(seed, stream, row, col4, w);
  for (int h = 0; h < 2; ++h) {
    double u1 = ((double)(w[2 * h] >> 8) + 0.5) * (1.0 / 16777216.0);   /* (0, 1) */
    double u2 = (double)(w[2 * h + 1] >> 8) * (1.0 / 16777216.0);       /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586 * u2;
    n[2 * h] = r * cos(a);
    n[2 * h + 1] = r * sin(a);
  }
}

/* ---- workload description ------------------------------------------- */
typedef struct {
  uint64_t seed;
  int32_t k;              /* draft tokens per chain */
  int32_t vocab;          /* V */
  int32_t dtype;          /* SG_FP32 / SG_BF16 */
  int32_t batch_total;    /* B of the whole workload (for the regime split) */
  double sigma_a;         /* target logit scale, chains b < split */
  double sigma_b;         /* target logit scale, chains b >= split */
  int32_t split;          /* first chain using sigma_b */
  int32_t n_boost;        /* boosted ids per target row (distinct) */
  double boost;           /* added to boosted ids */
  int32_t draft_mode;     /* 0: draft = target + N(0, draft_sigma^2); 1: independent N(0, draft_sigma^2) */
  double draft_sigma;
  int32_t temp_mode;      /* 0: fixed temp_lo; 1: per chain U[temp_lo, temp_hi] */
  double temp_lo, temp_hi;
} sg_workload;

static double target_sigma(const sg_workload* w, int64_t b) { return b < w->split ? w->sigma_a : w->sigma_b; }

float sg_temperature(const sg_workload* w, int64_t b) {
  if (w->temp_mode == 0) return (float)w->temp_lo;
  double u = sg_uniform(w->seed, ST_TEMP, (uint64_t)b, 0);
  return (float)(w->temp_lo + (w->temp_hi - w->temp_lo) * u);
}

/* Boosted ids: the first n_boost distinct values of floor(u * V) on stream 4. */
static int boosted_ids(const sg_workload* w, uint64_t row, int32_t* ids) {
  int n = 0;
  uint64_t col = 0;
  while (n < w->n_boost) {
    uint32_t word = word_at(w->seed, ST_BOOST, row, col++);
    int32_t id = (int32_t)(((uint64_t)(word >> 8) * (uint64_t)w->vocab) >> 24);
    int dup = 0;
    for (int i = 0; i < n; ++i) dup |= (ids[i] == id);
    if (!dup) ids[n++] = id;
    if (col > (uint64_t)w->n_boost * 64 + 1024) break;
  }
  return n;
}

/* One logit row as fp32 values before storage rounding. */
static void target_row_f32(const sg_workload* w, int64_t b, int i, float* out) {
  const int64_t V = w->vocab;
  const uint64_t row = (uint64_t)b * (uint64_t)(w->k + 1) + (uint64_t)i;
  const double s = target_sigma(w, b);
  double n[4];
  for (int64_t j = 0; j < V; j += 4) {
    normals4(w->seed, ST_TARGET, row, (uint64_t)(j >> 2), n);
    for (int t = 0; t < 4 && j + t < V; ++t) out[j + t] = (float)(s * n[t]);
  }
  if (w->n_boost > 0) {
    int32_t ids[256];
    int nb = boosted_ids(w, row, ids);
    for (int t = 0; t < nb; ++t) out[ids[t]] = (float)((double)out[ids[t]] + w->boost);
  }
}

static void store_row(const float* src, int64_t V, int dtype, void* dst) {
  if (dtype == SG_FP32) {
    memcpy(dst, src, (size_t)V * 4);
  } else {
    uint16_t* d = (uint16_t*)dst;
    for (int64_t j = 0; j < V; ++j) d[j] = f32_to_bf16(src[j]);
  }
}
static void load_row(const void* src, int64_t V, int dtype, float* dst) {
  if (dtype == SG_FP32) {
    memcpy(dst, src, (size_t)V * 4);
  } else {
    const uint16_t* s = (const uint16_t*)src;
    for (int64_t j = 0; j < V; ++j) dst[j] = bf16_to_f32(s[j]);
  }
}

/* Draft row i of chain b: the stored target row plus noise, or independent normals. */
static void draft_row_f32(const sg_workload* w, int64_t b, int i, const float* target_stored, float* out) {
  const int64_t V = w->vocab;
  const uint64_t row = (uint64_t)b * (uint64_t)w->k + (uint64_t)i;
  double n[4];
  for (int64_t j = 0; j < V; j += 4) {
    normals4(w->seed, ST_DRAFT, row, (uint64_t)(j >> 2), n);
    for (int t = 0; t < 4 && j + t < V; ++t) {
      double base = w->draft_mode == 0 ? (double)target_stored[j + t] : 0.0;
      out[j + t] = (float)(base + w->draft_sigma * n[t]);
    }
  }
}

/* Gumbel-max: the index maximising z_j + T * g_j with g_j = -log(-log(u_j)),
 * u_j on the half-shifted lattice of stream 2.  For T == 0 this is the
 * plain argmax (lowest index among equal values).  The Gumbel-max trick draws
 * exactly from softmax(z / T) (Gumbel 1954; Maddison et al. 2014). */
static int32_t gumbel_argmax(const sg_workload* w, uint64_t row, const float* z, double T) {
  const int64_t V = w->vocab;
  double best = -INFINITY;
  int32_t arg = 0;
  uint32_t wd[4];
  for (int64_t j = 0; j < V; ++j) {
    double v = (double)z[j];
    if (T > 0.0) {
      if ((j & 3) == 0) block4(w->seed, ST_GUMBEL, row, (uint64_t)(j >> 2), wd);
      double u = ((double)(wd[j & 3] >> 8) + 0.5) * (1.0 / 16777216.0);
      v += T * (-log(-log(u)));
    }
    if (v > best) { best = v; arg = (int32_t)j; }
  }
  return arg;
}

/* ---- chain generation ------------------------------------------------ */
typedef struct {
  const sg_workload* w;
  int64_t b0, nb;        /* chains [b0, b0 + nb) of the workload */
  int64_t first, stride; /* this thread's share of the nb chains */
  void* target;          /* [nb, k+1, V] */
  void* draft;           /* [nb, k, V]   */
  int32_t* tokens;       /* [nb, k]      */
  float* temps;          /* [nb]         */
  float* uniforms;       /* [nb, k+1]    */
} sg_job;

static void* gen_worker(void* arg) {
  sg_job* J = (sg_job*)arg;
  const sg_workload* w = J->w;
  const int64_t V = w->vocab, k = w->k;
  const size_t es = w->dtype == SG_FP32 ? 4 : 2;
  float* tf = (float*)malloc((size_t)V * 4);
  float* ts = (float*)malloc((size_t)V * 4);
  float* df = (float*)malloc((size_t)V * 4);
  float* ds = (float*)malloc((size_t)V * 4);
  for (int64_t lb = J->first; lb < J->nb; lb += J->stride) {
    const int64_t b = J->b0 + lb;
    const float T = sg_temperature(w, b);
    if (J->temps) J->temps[lb] = T;
    if (J->uniforms)
      for (int64_t i = 0; i <= k; ++i) J->uniforms[lb * (k + 1) + i] = sg_uniform(w->seed, ST_VERIFY, (uint64_t)b, (uint64_t)i);
    for (int64_t i = 0; i <= k; ++i) {
      target_row_f32(w, b, (int)i, tf);
      char* trow = (char*)J->target + ((size_t)(lb * (k + 1) + i) * (size_t)V) * es;
      store_row(tf, V, w->dtype, trow);
      if (i == k) break;
      load_row(trow, V, w->dtype, ts);
      draft_row_f32(w, b, (int)i, ts, df);
      char* drow = (char*)J->draft + ((size_t)(lb * k + i) * (size_t)V) * es;
      store_row(df, V, w->dtype, drow);
      if (J->tokens) {
        load_row(drow, V, w->dtype, ds);
        J->tokens[lb * k + i] = gumbel_argmax(w, (uint64_t)(b * k + i), ds, (double)T);
      }
    }
  }
  free(tf); free(ts); free(df); free(ds);
  return NULL;
}

/* Generate chains [b0, b0 + nb) of the workload into caller-owned host
 * buffers.  Any of tokens / temps / uniforms may be NULL.  Returns 0 on
 * success.  The result does not depend on nthreads. */
int sg_generate(const sg_workload* w, int64_t b0, int64_t nb, void* target, void* draft,
                int32_t* tokens, float* temps, float* uniforms, int nthreads) {
  if (!w || w->k < 1 || w->vocab < 1 || nb < 0 || b0 < 0 || !target || !draft) return 1;
  if (w->dtype != SG_FP32 && w->dtype != SG_BF16) return 2;
  if (w->n_boost < 0 || w->n_boost > 256 || w->n_boost > w->vocab) return 3;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > nb) nthreads = (int)(nb > 0 ? nb : 1);
  pthread_t th[256];
  sg_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (sg_job){w, b0, nb, t, nthreads, target, draft, tokens, temps, uniforms};
  }
  if (nthreads == 1) {
    gen_worker(&jobs[0]);
    return 0;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, gen_worker, &jobs[t]) != 0) break;
    started++;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  for (int t = started; t < nthreads; ++t) gen_worker(&jobs[t]);
  return 0;
}

/* Independent uniforms [n_rows, n_cols] of one stream (rows row0..row0+n_rows-1). */
void sg_uniforms(uint64_t seed, uint32_t stream, uint64_t row0, int64_t n_rows, int64_t n_cols, float* out) {
  for (int64_t r = 0; r < n_rows; ++r)
    for (int64_t c = 0; c < n_cols; ++c)
      out[r * n_cols + c] = sg_uniform(seed, stream, row0 + (uint64_t)r, (uint64_t)c);
}

/* Gumbel-max samples of `rows` rows of logits (for drawing drafts from a given
 * distribution in tests): row r uses Gumbel row id row0 + r of stream 2. */
void sg_gumbel_argmax_rows(uint64_t seed, const void* logits, int dtype, int64_t rows, int64_t V,
                           const float* temps, uint64_t row0, int32_t* out) {
  sg_workload w;
  memset(&w, 0, sizeof w);
  w.seed = seed; w.vocab = (int32_t)V; w.dtype = dtype;
  float* z = (float*)malloc((size_t)V * 4);
  const size_t es = dtype == SG_FP32 ? 4 : 2;
  for (int64_t r = 0; r < rows; ++r) {
    load_row((const char*)logits + (size_t)r * (size_t)V * es, V, dtype, z);
    out[r] = gumbel_argmax(&w, row0 + (uint64_t)r, z, (double)temps[r]);
  }
  free(z);
}
