/*
 * lkv_oracle.c -- plain, slow, single-threaded CPU oracle (test infrastructure
 * only; see lkv_oracle.h for the sources, the precision rules and the build
 * flags). Every loop runs in the order the definition states; there is no
 * blocking, fusion or reordering.
 */
#include "lkv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element access                                                            */

float lkvo_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t lkvo_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u); /* round to nearest, ties to even */
  return (uint16_t)(u >> 16);
}

static float elem(const void *p, int dtype, int64_t i) {
  if (dtype == LKVO_BF16) return lkvo_bf16_to_f32(((const uint16_t *)p)[i]);
  return ((const float *)p)[i];
}

static size_t elem_size(int dtype) { return dtype == LKVO_BF16 ? 2u : 4u; }

static const void *row_ptr(const void *base, int dtype, int64_t row, int32_t d) {
  return (const char *)base + (size_t)row * (size_t)d * elem_size(dtype);
}

/* ------------------------------------------------------------------------ */
/* seeded initialisation                                                     */

/* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; constants as in Vigna's public-domain
 * splitmix64.c): state += golden gamma, then the variant-13 mix. */
static uint64_t splitmix64_next(uint64_t *state) {
  uint64_t z = (*state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

void lkvo_splitmix64(uint64_t seed, int32_t count, uint64_t *out) {
  uint64_t st = seed;
  for (int32_t i = 0; i < count; ++i) out[i] = splitmix64_next(&st);
}

int lkvo_init_indices(int64_t n, int32_t c, uint64_t seed, int64_t *idx_out) {
  if (c < 1 || (int64_t)c > n) return -1;
  int64_t *perm = (int64_t *)malloc((size_t)n * sizeof *perm);
  if (!perm) return -1;
  for (int64_t i = 0; i < n; ++i) perm[i] = i;
  uint64_t st = seed;
  for (int32_t i = 0; i < c; ++i) {
    uint64_t r = splitmix64_next(&st);
    int64_t j = (int64_t)i + (int64_t)(r % (uint64_t)(n - i));
    int64_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
    idx_out[i] = perm[i];
  }
  free(perm);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* K-means [LouisKV notes, 关键设计 2: K-means over the prefill keys, centroid  */
/* = mean of the cluster's keys, used as the retrieval index]                */

double lkvo_sqdist(const void *key, int dtype, const float *cent, int32_t d) {
  double acc = 0.0;
  for (int32_t j = 0; j < d; ++j) {
    double diff = (double)elem(key, dtype, j) - (double)cent[j];
    double sq = diff * diff;
    acc = acc + sq;
  }
  return acc;
}

void lkvo_assign(const void *keys, int dtype, int64_t n, int32_t d,
                 const float *cent, int32_t c, int32_t *assign_out,
                 double *gap_out) {
  for (int64_t i = 0; i < n; ++i) {
    const void *k = row_ptr(keys, dtype, i, d);
    int32_t best = 0;
    double d1 = lkvo_sqdist(k, dtype, cent, d);
    double d2 = INFINITY;
    for (int32_t j = 1; j < c; ++j) {
      double dj = lkvo_sqdist(k, dtype, cent + (size_t)j * d, d);
      if (dj < d1) {
        d2 = d1;
        d1 = dj;
        best = j;
      } else if (dj < d2) {
        d2 = dj;
      }
    }
    assign_out[i] = best;
    if (gap_out) {
      double kk = 0.0, cc = 0.0;
      for (int32_t j = 0; j < d; ++j) {
        double kv = elem(k, dtype, j), cv = cent[(size_t)best * d + j];
        kk += kv * kv;
        cc += cv * cv;
      }
      gap_out[i] = (c > 1) ? (d2 - d1) / (kk + cc) : INFINITY;
    }
  }
}

void lkvo_update(const void *keys, int dtype, int64_t n, int32_t d,
                 const int32_t *assign, int32_t c, float *cent,
                 int32_t *count_out, int64_t *inexact_out) {
  double *sum = (double *)calloc((size_t)c * d, sizeof *sum);
  int64_t inexact = 0;
  for (int32_t j = 0; j < c; ++j) count_out[j] = 0;
  /* token order: each cluster's members are added in increasing token index */
  for (int64_t i = 0; i < n; ++i) {
    int32_t j = assign[i];
    count_out[j] += 1;
    const void *k = row_ptr(keys, dtype, i, d);
    for (int32_t t = 0; t < d; ++t) {
      double a = sum[(size_t)j * d + t], b = (double)elem(k, dtype, t);
      double s = a + b;
      /* two-sum error term: nonzero iff the addition rounded */
      double bb = s - a;
      double err = (a - (s - bb)) + (b - bb);
      if (err != 0.0) ++inexact;
      sum[(size_t)j * d + t] = s;
    }
  }
  for (int32_t j = 0; j < c; ++j) {
    if (count_out[j] == 0) continue; /* empty cluster keeps its centroid */
    for (int32_t t = 0; t < d; ++t)
      cent[(size_t)j * d + t] =
          (float)(sum[(size_t)j * d + t] / (double)count_out[j]);
  }
  free(sum);
  if (inexact_out) *inexact_out += inexact;
}

void lkvo_operand(const float *cent, int64_t count, int dtype, float *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = (dtype == LKVO_BF16) ? lkvo_bf16_to_f32(lkvo_f32_to_bf16(cent[i]))
                                  : cent[i];
}

double lkvo_objective(const void *keys, int dtype, int64_t n, int32_t d,
                      const float *cent, const int32_t *assign) {
  double j = 0.0;
  for (int64_t i = 0; i < n; ++i)
    j += lkvo_sqdist(row_ptr(keys, dtype, i, d), dtype,
                     cent + (size_t)assign[i] * d, d);
  return j;
}

int lkvo_kmeans(const void *keys, int dtype, int64_t n, int32_t d, int32_t c,
                int32_t iters, uint64_t seed, float *cent_out,
                int32_t *assign_out, int32_t *count_out, float *trace_cent,
                int32_t *trace_assign, int64_t *inexact_out) {
  if (iters < 1 || c < 1 || (int64_t)c > n || d < 1) return -1;
  int64_t *idx = (int64_t *)malloc((size_t)c * sizeof *idx);
  float *op = (float *)malloc((size_t)c * d * sizeof *op);
  if (!idx || !op) {
    free(idx);
    free(op);
    return -1;
  }
  lkvo_init_indices(n, c, seed, idx);
  for (int32_t j = 0; j < c; ++j)
    for (int32_t t = 0; t < d; ++t)
      cent_out[(size_t)j * d + t] = elem(keys, dtype, idx[j] * d + t);
  if (inexact_out) *inexact_out = 0;
  if (trace_cent) memcpy(trace_cent, cent_out, (size_t)c * d * sizeof(float));
  for (int32_t it = 0; it < iters; ++it) {
    lkvo_operand(cent_out, (int64_t)c * d, dtype, op);
    lkvo_assign(keys, dtype, n, d, op, c, assign_out, NULL);
    lkvo_update(keys, dtype, n, d, assign_out, c, cent_out, count_out,
                inexact_out);
    if (trace_assign)
      memcpy(trace_assign + (size_t)it * n, assign_out, (size_t)n * sizeof(int32_t));
    if (trace_cent)
      memcpy(trace_cent + (size_t)(it + 1) * c * d, cent_out,
             (size_t)c * d * sizeof(float));
  }
  free(idx);
  free(op);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* semantic boundary [LouisKV notes, 关键设计 1]                              */

float lkvo_boundary_r32(const void *q_prev, const void *q_cur, int dtype,
                        int32_t h, int32_t d) {
  float r = 0.0f;
  for (int32_t head = 0; head < h; ++head) {
    float dot = 0.0f, na = 0.0f, nb = 0.0f;
    for (int32_t j = 0; j < d; ++j) {
      float a = elem(q_prev, dtype, (int64_t)head * d + j);
      float b = elem(q_cur, dtype, (int64_t)head * d + j);
      dot = fmaf(a, b, dot);
      na = fmaf(a, a, na);
      nb = fmaf(b, b, nb);
    }
    float den = sqrtf(na) * sqrtf(nb);
    float cs = (den > 0.0f) ? dot / den : 0.0f;
    r = r + cs;
  }
  return r / (float)h;
}

double lkvo_boundary_r64(const void *q_prev, const void *q_cur, int dtype,
                         int32_t h, int32_t d) {
  double r = 0.0;
  for (int32_t head = 0; head < h; ++head) {
    double dot = 0.0, na = 0.0, nb = 0.0;
    for (int32_t j = 0; j < d; ++j) {
      double a = elem(q_prev, dtype, (int64_t)head * d + j);
      double b = elem(q_cur, dtype, (int64_t)head * d + j);
      dot += a * b;
      na += a * a;
      nb += b * b;
    }
    double den = sqrt(na) * sqrt(nb);
    r += (den > 0.0) ? dot / den : 0.0;
  }
  return r / (double)h;
}

/* ------------------------------------------------------------------------ */
/* group-consistent scoring and budgeted selection [LouisKV notes, 关键设计 3] */

void lkvo_group_scores(const void *q, int dtype, int32_t g, int32_t d,
                       const float *cent, int32_t u, float *scores_out) {
  float *qbar = (float *)malloc((size_t)d * sizeof *qbar);
  for (int32_t j = 0; j < d; ++j) {
    float acc = elem(q, dtype, j);
    for (int32_t h = 1; h < g; ++h) acc = acc + elem(q, dtype, (int64_t)h * d + j);
    qbar[j] = acc;
  }
  for (int32_t k = 0; k < u; ++k) {
    float s = 0.0f;
    for (int32_t j = 0; j < d; ++j) s = fmaf(qbar[j], cent[(size_t)k * d + j], s);
    scores_out[k] = s;
  }
  free(qbar);
}

/* (score descending, id ascending) */
static int precedes(const float *s, int32_t a, int32_t b) {
  if (s[a] != s[b]) return s[a] > s[b];
  return a < b;
}

int32_t lkvo_select(const float *scores, const int32_t *len, int32_t u,
                    int32_t budget, int32_t *sel_out, int32_t *n_tok_out) {
  /* plain insertion sort of the ids by the selection order */
  int32_t *order = (int32_t *)malloc((size_t)(u > 0 ? u : 1) * sizeof *order);
  for (int32_t i = 0; i < u; ++i) {
    int32_t x = i, p = i;
    while (p > 0 && precedes(scores, x, order[p - 1])) {
      order[p] = order[p - 1];
      --p;
    }
    order[p] = x;
  }
  int32_t n_sel = 0, tok = 0;
  for (int32_t i = 0; i < u; ++i) {
    int32_t id = order[i];
    if (tok + len[id] > budget) break; /* first unit that does not fit */
    tok += len[id];
    sel_out[n_sel++] = id;
  }
  free(order);
  *n_tok_out = tok;
  return n_sel;
}

int32_t lkvo_select_skip(const float *scores, const int32_t *len, int32_t u,
                         int32_t budget, int32_t *sel_out, int32_t *n_tok_out) {
  int32_t *order = (int32_t *)malloc((size_t)(u > 0 ? u : 1) * sizeof *order);
  for (int32_t i = 0; i < u; ++i) {
    int32_t x = i, p = i;
    while (p > 0 && precedes(scores, x, order[p - 1])) {
      order[p] = order[p - 1];
      --p;
    }
    order[p] = x;
  }
  int32_t n_sel = 0, tok = 0;
  for (int32_t i = 0; i < u; ++i) {
    int32_t id = order[i];
    if (tok + len[id] > budget) continue; /* does not fit: skip it */
    tok += len[id];
    sel_out[n_sel++] = id;
  }
  free(order);
  *n_tok_out = tok;
  return n_sel;
}

/* ------------------------------------------------------------------------ */
/* attention over the retrieved + local tokens [LouisKV notes, flowchart:     */
/* Attention over retrieved or reused critical KV]                           */

void lkvo_attention(const void *q, int dtype, int32_t g, int32_t d,
                    const void *k_rows, const void *v_rows, int64_t n,
                    double *out) {
  double *logit = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof *logit);
  double scale = 1.0 / sqrt((double)d);
  for (int32_t h = 0; h < g; ++h) {
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
      double dot = 0.0;
      for (int32_t j = 0; j < d; ++j)
        dot += (double)elem(q, dtype, (int64_t)h * d + j) *
               (double)elem(k_rows, dtype, i * d + j);
      logit[i] = dot * scale;
      if (logit[i] > m) m = logit[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      logit[i] = exp(logit[i] - m);
      z += logit[i];
    }
    for (int32_t j = 0; j < d; ++j) {
      double acc = 0.0;
      for (int64_t i = 0; i < n; ++i)
        acc += logit[i] * (double)elem(v_rows, dtype, i * d + j);
      out[(size_t)h * d + j] = (n > 0) ? acc / z : 0.0;
    }
  }
  free(logit);
}

/* ------------------------------------------------------------------------ */
/* ParisKV-style selector [ParisKV technical summary, 核心算法创新 1-2]        */

void lkvo_paris_signs(uint64_t seed, int32_t d, int8_t *sign_out) {
  uint64_t st = seed, word = 0;
  for (int32_t j = 0; j < d; ++j) {
    if (j % 64 == 0) word = splitmix64_next(&st);
    sign_out[j] = (int8_t)(((word >> (j % 64)) & 1u) ? -1 : 1);
  }
}

/* density of |x| up to its constant, and its integral by composite Simpson */
static double sphere_marginal(double x, int32_t m) { return pow(1.0 - x * x, 0.5 * (m - 3)); }

static double simpson(double a, double b, int32_t m, int moment) {
  const int n = 20000; /* even */
  const double h = (b - a) / n;
  double acc = 0.0;
  for (int i = 0; i <= n; ++i) {
    const double x = a + h * i;
    double f = sphere_marginal(x, m) * (moment ? x : 1.0);
    acc += f * (i == 0 || i == n ? 1.0 : (i % 2 ? 4.0 : 2.0));
  }
  return acc * h / 3.0;
}

int lkvo_paris_levels(int32_t m, float *thr_out, float *lev_out) {
  if (m < 2) return -1;
  const double total = simpson(0.0, 1.0, m, 0);
  double t[9];
  t[0] = 0.0;
  t[8] = 1.0;
  for (int l = 1; l < 8; ++l) {
    double lo = 0.0, hi = 1.0; /* P(|x| < t) = l / 8 by bisection */
    for (int it = 0; it < 60; ++it) {
      const double mid = 0.5 * (lo + hi);
      if (simpson(0.0, mid, m, 0) / total < l / 8.0) lo = mid;
      else hi = mid;
    }
    t[l] = 0.5 * (lo + hi);
    thr_out[l - 1] = (float)(t[l] * t[l]);
  }
  for (int l = 0; l < 8; ++l)
    lev_out[l] = (float)(simpson(t[l], t[l + 1], m, 1) / simpson(t[l], t[l + 1], m, 0));
  return 0;
}

static int hadamard_sign(int32_t i, int32_t j) {
  unsigned x = (unsigned)(i & j), par = 0;
  while (x) { par ^= x & 1u; x >>= 1; }
  return par ? -1 : 1;
}

/* the rotation's signs H_ij D_j, [d][d] */
static int8_t *paris_matrix(int32_t d, const int8_t *sign) {
  int8_t *hd = (int8_t *)malloc((size_t)d * d);
  if (!hd) return NULL;
  for (int32_t i = 0; i < d; ++i)
    for (int32_t j = 0; j < d; ++j) hd[(size_t)i * d + j] = (int8_t)(hadamard_sign(i, j) * sign[j]);
  return hd;
}

static void paris_encode_hd(const uint16_t *key, int32_t d, const int8_t *hd, int32_t m,
                            const float *thr, const float *lev, uint8_t *bucket_out,
                            uint8_t *level_out, float *w_out) {
  int64_t *k40 = (int64_t *)malloc((size_t)d * sizeof *k40);
  int64_t *y = (int64_t *)malloc((size_t)d * sizeof *y);
  for (int32_t j = 0; j < d; ++j) k40[j] = (int64_t)((double)lkvo_bf16_to_f32(key[j]) * 0x1p40);
  for (int32_t i = 0; i < d; ++i) {
    int64_t acc = 0;
    for (int32_t j = 0; j < d; ++j) acc += (int64_t)hd[(size_t)i * d + j] * k40[j];
    y[i] = acc;
  }
  for (int32_t b = 0; b < d / m; ++b) {
    const int64_t *yb = y + (size_t)b * m;
    unsigned bits = 0;
    double n2 = 0.0;
    for (int32_t j = 0; j < m; ++j) {
      if (yb[j] < 0) bits |= 1u << j;
      n2 = n2 + (double)yb[j] * (double)yb[j];
    }
    bucket_out[b] = (uint8_t)bits;
    double num = 0.0, den = 0.0;
    for (int32_t j = 0; j < m; ++j) {
      const double sq = (double)yb[j] * (double)yb[j];
      int l = 0;
      for (int k = 0; k < 7; ++k)
        if (sq >= (double)thr[k] * n2) l = k + 1;
      level_out[(size_t)b * m + j] = (uint8_t)l;
      const double v = (yb[j] < 0 ? -1.0 : 1.0) * (double)lev[l];
      num = num + (double)yb[j] * v;
      den = den + v * v;
    }
    w_out[b] = (float)(num / den * 0x1p-40 / sqrt((double)d));
  }
  free(k40);
  free(y);
}

void lkvo_paris_encode(const uint16_t *key, int32_t d, const int8_t *sign, int32_t m,
                       const float *thr, const float *lev, uint8_t *bucket_out,
                       uint8_t *level_out, float *w_out) {
  int8_t *hd = paris_matrix(d, sign);
  if (!hd) return;
  paris_encode_hd(key, d, hd, m, thr, lev, bucket_out, level_out, w_out);
  free(hd);
}

void lkvo_paris_rotate_query(const void *q, int dtype, int32_t g, int32_t d,
                             const int8_t *sign, float *qrot_out) {
  for (int32_t j = 0; j < d; ++j) {
    float acc = elem(q, dtype, j);
    for (int32_t h = 1; h < g; ++h) acc = acc + elem(q, dtype, (int64_t)h * d + j);
    qrot_out[j] = sign[j] < 0 ? -acc : acc;
  }
  for (int32_t h = 1; h < d; h *= 2)
    for (int32_t i = 0; i < d; i += 2 * h)
      for (int32_t j = i; j < i + h; ++j) {
        const float a = qrot_out[j], b = qrot_out[j + h];
        qrot_out[j] = a + b;
        qrot_out[j + h] = a - b;
      }
}

/* rankings by (value desc, id asc), sorted with the C library's qsort */
typedef struct { int32_t v; int64_t id; } rank_i;
typedef struct { float v; int64_t id; } rank_f;
static int cmp_rank_i(const void *pa, const void *pb) {
  const rank_i *a = (const rank_i *)pa, *b = (const rank_i *)pb;
  if (a->v != b->v) return a->v > b->v ? -1 : 1;
  return a->id < b->id ? -1 : (a->id > b->id);
}
static int cmp_rank_f(const void *pa, const void *pb) {
  const rank_f *a = (const rank_f *)pa, *b = (const rank_f *)pb;
  if (a->v != b->v) return a->v > b->v ? -1 : 1;
  return a->id < b->id ? -1 : (a->id > b->id);
}

int64_t lkvo_paris_select(const float *qrot, int32_t d, int32_t m, int32_t rho,
                          int64_t n_cand, int32_t budget, int64_t n,
                          const uint8_t *bucket, const uint8_t *level, const float *w,
                          const float *lev, int64_t *sel_out, int32_t *coarse_out,
                          float *est_out) {
  const int32_t nb = d / m, np = 1 << m;
  int32_t *vote = (int32_t *)calloc((size_t)nb * np, sizeof *vote);
  float *sim = (float *)malloc((size_t)np * sizeof *sim);
  int32_t *coarse = (int32_t *)calloc((size_t)(n > 0 ? n : 1), sizeof *coarse);
  float *est = (float *)calloc((size_t)(n > 0 ? n : 1), sizeof *est);
  rank_i *order = (rank_i *)malloc((size_t)(n > 0 ? n : 1) * sizeof *order);
  /* the rho best sign centroids of each subspace and their votes */
  for (int32_t b = 0; b < nb; ++b) {
    for (int32_t p = 0; p < np; ++p) {
      float s = 0.0f;
      for (int32_t j = 0; j < m; ++j) {
        const float x = qrot[(size_t)b * m + j];
        s = s + (((p >> j) & 1) ? -x : x);
      }
      sim[p] = s;
    }
    for (int32_t r = 0; r < rho && r < np; ++r) {
      int32_t best = -1;
      for (int32_t p = 0; p < np; ++p) {
        if (vote[(size_t)b * np + p]) continue;
        if (best < 0 || sim[p] > sim[best] || (sim[p] == sim[best] && p < best)) best = p;
      }
      vote[(size_t)b * np + best] = rho - r;
    }
  }
  for (int64_t i = 0; i < n; ++i) {
    int32_t c = 0;
    for (int32_t b = 0; b < nb; ++b) c += vote[(size_t)b * np + bucket[(size_t)i * nb + b]];
    coarse[i] = c;
  }
  /* candidates: the n_cand best coarse scores */
  for (int64_t i = 0; i < n; ++i) {
    order[i].v = coarse[i];
    order[i].id = i;
  }
  qsort(order, (size_t)n, sizeof *order, cmp_rank_i);
  const int64_t nc = n_cand < n ? n_cand : n;
  for (int64_t c = 0; c < nc; ++c) {
    const int64_t i = order[c].id;
    float e = 0.0f;
    for (int32_t b = 0; b < nb; ++b) {
      float dot = 0.0f;
      for (int32_t j = 0; j < m; ++j) {
        const size_t x = (size_t)b * m + j;
        const float v = ((bucket[(size_t)i * nb + b] >> j) & 1) ? -lev[level[(size_t)i * d + x]]
                                                                 : lev[level[(size_t)i * d + x]];
        dot = fmaf(v, qrot[x], dot);
      }
      e = fmaf(w[(size_t)i * nb + b], dot, e);
    }
    est[i] = e;
  }
  /* the budget best candidates by the estimate */
  rank_f *cand = (rank_f *)malloc((size_t)(nc > 0 ? nc : 1) * sizeof *cand);
  for (int64_t c = 0; c < nc; ++c) {
    cand[c].v = est[order[c].id];
    cand[c].id = order[c].id;
  }
  qsort(cand, (size_t)nc, sizeof *cand, cmp_rank_f);
  const int64_t k = budget < nc ? budget : nc;
  for (int64_t c = 0; c < k; ++c) sel_out[c] = cand[c].id;
  if (coarse_out) memcpy(coarse_out, coarse, (size_t)n * sizeof *coarse);
  if (est_out) memcpy(est_out, est, (size_t)n * sizeof *est);
  free(vote); free(sim); free(coarse); free(est); free(order); free(cand);
  return k;
}

/* ------------------------------------------------------------------------ */
/* decode: boundary -> segment close -> append/evict -> retrieve -> attend   */

int lkvo_decode(const lkvo_decode_args *a, lkvo_decode_result *r) {
  const int dt = a->dtype;
  const int32_t hkv = a->n_kv_heads, g = a->group, d = a->head_dim;
  const int32_t h_all = hkv * g, c = a->n_clusters, L = a->local_buf;
  const int32_t T = a->n_steps;
  const int64_t n = a->n_prefill;
  const size_t es = elem_size(dt);
  const int paris = a->selector == LKVO_SELECT_PARIS;
  /* the ParisKV-style selector has no clusters (c = 0) */
  if (hkv < 1 || g < 1 || d < 1 || c < (paris ? 0 : 1) || L < 1 || T < 0 || n < 0) return -1;
  const int32_t ucap = c + T > 0 ? c + T : 1; /* every eviction removes at least one token */
  if (a->trigger < 0 || a->trigger > 2 || (a->trigger == 2 && a->interval < 1) ||
      a->fill < 0 || a->fill > 1 || a->page < 0 || a->per_head < 0 || a->per_head > 1)
    return -1;
  /* selections: one per KV head, or one per query head */
  const int32_t hs = a->per_head ? h_all : hkv, gs = a->per_head ? 1 : g;
  if (a->selector < 0 || a->selector > 1) return -1;
  if (paris && (dt != LKVO_BF16 || a->per_head || d % 8 || a->paris_rho < 1 ||
                a->paris_rho > 256 || a->paris_n_cand < 1))
    return -1;

  int rc = -1;
  /* ParisKV-style metadata of every prefill and decode token, per KV head */
  const int32_t pnb = d / 8;
  int8_t *psign = NULL;
  uint8_t *pbk = NULL, *plv = NULL;
  float *pw = NULL, *pq = NULL;
  int64_t *psel = NULL;
  float pthr[7], plev[8];
  /* cluster membership in token order, per kv head */
  int32_t *cnt = (int32_t *)calloc((size_t)hkv * (c > 0 ? c : 1), sizeof *cnt);
  int32_t *first = (int32_t *)malloc((size_t)hkv * (c + 1) * sizeof *first);
  int64_t *member = (int64_t *)malloc((size_t)(hkv * n > 0 ? hkv * n : 1) * sizeof *member);
  /* per kv head unit tables: operand centroid and length */
  float *op = (float *)malloc((size_t)hkv * ucap * d * sizeof *op);
  int32_t *ulen = (int32_t *)malloc((size_t)hkv * ucap * sizeof *ulen);
  /* active selection per kv head */
  /* with the ParisKV-style selector a selection lists tokens (up to budget) */
  const int64_t acap = paris ? (a->budget > 0 ? a->budget : 1) : ucap;
  int32_t *act = (int32_t *)malloc((size_t)hs * acap * sizeof *act);
  int32_t *act_n = (int32_t *)calloc((size_t)hs, sizeof *act_n);
  int32_t *act_tok = (int32_t *)calloc((size_t)hs, sizeof *act_tok);
  /* closed, not yet evicted segments: FIFO of [start, end) */
  int32_t *cl_s = (int32_t *)malloc((size_t)(T + 1) * sizeof *cl_s);
  int32_t *cl_e = (int32_t *)malloc((size_t)(T + 1) * sizeof *cl_e);
  float *scores = (float *)malloc((size_t)ucap * sizeof *scores);
  float *segc = (float *)malloc((size_t)hkv * d * sizeof *segc);
  double *segsum = (double *)malloc((size_t)d * sizeof *segsum);
  char *kg = (char *)malloc((size_t)(n + T + 1) * d * es);
  char *vg = (char *)malloc((size_t)(n + T + 1) * d * es);
  if (!cnt || !first || !member || !op || !ulen || !act || !act_n ||
      !act_tok || !cl_s || !cl_e || !scores || !segc || !segsum || !kg || !vg)
    goto done;

  if (paris) {
    const size_t ntot = (size_t)hkv * (size_t)(n + T);
    psign = (int8_t *)malloc((size_t)d);
    pbk = (uint8_t *)malloc(ntot * pnb);
    plv = (uint8_t *)malloc(ntot * d);
    pw = (float *)malloc(ntot * pnb * sizeof *pw);
    pq = (float *)malloc((size_t)d * sizeof *pq);
    psel = (int64_t *)malloc((size_t)acap * sizeof *psel);
    if (!psign || !pbk || !plv || !pw || !pq || !psel) goto done;
    lkvo_paris_signs(a->paris_seed, d, psign);
    lkvo_paris_levels(8, pthr, plev);
    int8_t *hd = paris_matrix(d, psign);
    if (!hd) goto done;
    for (int32_t kh = 0; kh < hkv; ++kh)
      for (int64_t i = 0; i < n + T; ++i) {
        const uint16_t *kr = i < n ? (const uint16_t *)a->keys + ((size_t)kh * n + i) * d
                                   : (const uint16_t *)a->k_new + ((size_t)(i - n) * hkv + kh) * d;
        const size_t x = (size_t)kh * (n + T) + i;
        paris_encode_hd(kr, d, hd, 8, pthr, plev, pbk + x * pnb, plv + x * d, pw + x * pnb);
      }
    free(hd);
  }

  for (int32_t kh = 0; kh < hkv && !paris; ++kh) {
    const int32_t *as = a->assign + (size_t)kh * n;
    int32_t *ct = cnt + (size_t)kh * c;
    int32_t *fs = first + (size_t)kh * (c + 1);
    for (int64_t i = 0; i < n; ++i) {
      if (as[i] < 0 || as[i] >= c) goto done;
      ct[as[i]] += 1;
    }
    fs[0] = 0;
    for (int32_t j = 0; j < c; ++j) fs[j + 1] = fs[j] + ct[j];
    int32_t *fill = (int32_t *)calloc((size_t)c, sizeof *fill);
    if (!fill) goto done;
    for (int64_t i = 0; i < n; ++i) {
      int32_t j = as[i];
      member[(size_t)kh * n + fs[j] + fill[j]++] = i;
    }
    free(fill);
    lkvo_operand(a->cent + (size_t)kh * c * d, (int64_t)c * d, dt,
                 op + (size_t)kh * ucap * d);
    for (int32_t j = 0; j < c; ++j) ulen[(size_t)kh * ucap + j] = ct[j];
  }

  int32_t n_units = c, n_ev = 0, n_forced = 0;
  int32_t win_start = 0, open_start = 0, cl_head = 0, cl_tail = 0;

  for (int32_t t = 0; t < T; ++t) {
    const void *qt = row_ptr(a->q, dt, (int64_t)t * h_all, d);
    /* 1. boundary test (r_t is computed and recorded under every policy) */
    int flag = 1;
    float r32 = 0.0f;
    double r64 = 0.0;
    if (t > 0) {
      const void *qp = row_ptr(a->q, dt, (int64_t)(t - 1) * h_all, d);
      r32 = lkvo_boundary_r32(qp, qt, dt, h_all, d);
      r64 = lkvo_boundary_r64(qp, qt, dt, h_all, d);
      if (a->trigger == LKVO_TRIGGER_ADAPTIVE) flag = r32 < a->tau;
      else if (a->trigger == LKVO_TRIGGER_INTERVAL) flag = t % a->interval == 0;
    }
    /* 2. a boundary (or, with pages, a full page) closes the open segment;
     *    token t starts the next one */
    const int cut = a->page > 0 ? (t - open_start >= a->page) : flag;
    if (cut && t > 0 && open_start < t) {
      cl_s[cl_tail] = open_start;
      cl_e[cl_tail] = t;
      ++cl_tail;
      open_start = t;
    }
    /* 3. make room for token t: evict whole segments, oldest first; with no
     *    closed segment left, cut the open one */
    while ((t - win_start) + 1 > L) {
      int32_t s0, s1;
      if (cl_head < cl_tail) {
        s0 = cl_s[cl_head];
        s1 = cl_e[cl_head];
        ++cl_head;
      } else {
        s0 = open_start;
        s1 = t;
        open_start = t;
        ++n_forced;
      }
      if (n_ev >= r->max_segs) goto done;
      for (int32_t kh = 0; kh < hkv; ++kh) {
        for (int32_t j = 0; j < d; ++j) segsum[j] = 0.0;
        for (int32_t tt = s0; tt < s1; ++tt)
          for (int32_t j = 0; j < d; ++j)
            segsum[j] = segsum[j] +
                        (double)elem(a->k_new, dt, ((int64_t)tt * hkv + kh) * d + j);
        for (int32_t j = 0; j < d; ++j)
          segc[(size_t)kh * d + j] = (float)(segsum[j] / (double)(s1 - s0));
        lkvo_operand(segc + (size_t)kh * d, d, dt,
                     op + ((size_t)kh * ucap + n_units) * d);
        ulen[(size_t)kh * ucap + n_units] = s1 - s0;
      }
      r->seg_start[n_ev] = s0;
      r->seg_len[n_ev] = s1 - s0;
      if (r->seg_cent)
        memcpy(r->seg_cent + (size_t)n_ev * hkv * d, segc,
               (size_t)hkv * d * sizeof(float));
      ++n_ev;
      ++n_units;
      win_start = s1;
    }
    /* 4. token t enters the local buffer [win_start, t] */
    /* 5. retrieval on a boundary step, against the pool after evictions */
    if (flag && paris) {
      /* tokens: the prefill, then the decode tokens before the buffer */
      for (int32_t kh = 0; kh < hkv; ++kh) {
        const int64_t nreg = n + win_start;
        const size_t x0 = (size_t)kh * (n + T);
        const void *qg = row_ptr(a->q, dt, (int64_t)t * h_all + (int64_t)kh * g, d);
        lkvo_paris_rotate_query(qg, dt, g, d, psign, pq);
        /* the region is contiguous in the metadata: prefill i at i, decode t' at n + t' */
        const int64_t k = lkvo_paris_select(pq, d, 8, a->paris_rho, a->paris_n_cand, a->budget, nreg,
                                            pbk + x0 * pnb, plv + x0 * d, pw + x0 * pnb, plev, psel,
                                            NULL, NULL);
        for (int64_t c = 0; c < k; ++c) act[(size_t)kh * acap + c] = (int32_t)psel[c];
        act_n[kh] = (int32_t)k;
        act_tok[kh] = (int32_t)k;
      }
    } else if (flag) {
      /* selection j scores with the sum of query heads j*gs .. j*gs+gs-1
       * (its group, or the one head) against its KV head's units */
      for (int32_t j = 0; j < hs; ++j) {
        const int32_t kh = j * gs / g;
        const void *qg = row_ptr(a->q, dt, (int64_t)t * h_all + (int64_t)j * gs, d);
        lkvo_group_scores(qg, dt, gs, d, op + (size_t)kh * ucap * d, n_units, scores);
        if (a->fill == LKVO_FILL_SKIP)
          act_n[j] = lkvo_select_skip(scores, ulen + (size_t)kh * ucap, n_units,
                                      a->budget, act + (size_t)j * acap, &act_tok[j]);
        else
          act_n[j] = lkvo_select(scores, ulen + (size_t)kh * ucap, n_units,
                                 a->budget, act + (size_t)j * acap, &act_tok[j]);
      }
    }
    /* 6. attention of each query head over its selection + buffer */
    if (!a->attn_mask || a->attn_mask[t]) {
      for (int32_t j = 0; j < hs; ++j) {
        const int32_t kh = j * gs / g;
        int64_t m = 0;
        for (int32_t s = 0; s < act_n[j]; ++s) {
          int32_t u = act[(size_t)j * acap + s];
          if (paris) { /* a token: prefill u, or decode token u - n */
            const void *ks = u < n ? row_ptr(a->keys, dt, (int64_t)kh * n + u, d)
                                   : row_ptr(a->k_new, dt, (int64_t)(u - n) * hkv + kh, d);
            const void *vs = u < n ? row_ptr(a->values, dt, (int64_t)kh * n + u, d)
                                   : row_ptr(a->v_new, dt, (int64_t)(u - n) * hkv + kh, d);
            memcpy(kg + m * d * es, ks, d * es);
            memcpy(vg + m * d * es, vs, d * es);
            ++m;
          } else if (u < c) {
            const int32_t *fs = first + (size_t)kh * (c + 1);
            for (int32_t p = fs[u]; p < fs[u + 1]; ++p) {
              int64_t i = member[(size_t)kh * n + p];
              memcpy(kg + m * d * es, row_ptr(a->keys, dt, (int64_t)kh * n + i, d), d * es);
              memcpy(vg + m * d * es, row_ptr(a->values, dt, (int64_t)kh * n + i, d), d * es);
              ++m;
            }
          } else {
            int32_t e = u - c;
            for (int32_t tt = r->seg_start[e]; tt < r->seg_start[e] + r->seg_len[e]; ++tt) {
              memcpy(kg + m * d * es, row_ptr(a->k_new, dt, (int64_t)tt * hkv + kh, d), d * es);
              memcpy(vg + m * d * es, row_ptr(a->v_new, dt, (int64_t)tt * hkv + kh, d), d * es);
              ++m;
            }
          }
        }
        for (int32_t tt = win_start; tt <= t; ++tt) {
          memcpy(kg + m * d * es, row_ptr(a->k_new, dt, (int64_t)tt * hkv + kh, d), d * es);
          memcpy(vg + m * d * es, row_ptr(a->v_new, dt, (int64_t)tt * hkv + kh, d), d * es);
          ++m;
        }
        const void *qg = row_ptr(a->q, dt, (int64_t)t * h_all + (int64_t)j * gs, d);
        lkvo_attention(qg, dt, gs, d, kg, vg, m,
                       r->out + ((size_t)t * h_all + (size_t)j * gs) * d);
      }
    }
    /* per-step record */
    if (r->flag) r->flag[t] = (uint8_t)flag;
    if (r->r32) r->r32[t] = r32;
    if (r->r64) r->r64[t] = r64;
    if (r->win_start) r->win_start[t] = win_start;
    if (r->n_units) r->n_units[t] = n_units;
    for (int32_t j = 0; j < hs; ++j) {
      if (r->n_sel) r->n_sel[(size_t)t * hs + j] = act_n[j];
      if (r->n_tok) r->n_tok[(size_t)t * hs + j] = act_tok[j];
      if (r->sel) {
        if (act_n[j] > r->max_sel) goto done;
        memcpy(r->sel + ((size_t)t * hs + j) * r->max_sel, act + (size_t)j * acap,
               (size_t)act_n[j] * sizeof(int32_t));
      }
    }
  }
  r->n_evicted = n_ev;
  r->n_forced = n_forced;
  rc = 0;

done:
  free(cnt); free(first); free(member); free(op); free(ulen); free(act);
  free(act_n); free(act_tok); free(cl_s); free(cl_e); free(scores);
  free(segc); free(segsum); free(kg); free(vg);
  free(psign); free(pbk); free(plv); free(pw); free(pq); free(psel);
  return rc;
}
