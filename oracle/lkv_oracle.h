/*
 * lkv_oracle.h -- plain, slow, single-threaded CPU oracle for LouisKV-style
 * KV-cache retrieval.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this code; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no source with the CUDA path.
 *
 * Sources (cited by page title and section):
 *   [LouisKV notes]  "LouisKV: Efficient KV Cache Retrieval for Long
 *                    Input-Output Sequences" (papernotes.org summary of the
 *                    ICLR 2026 paper): sections 方法详解/整体框架 (flowchart),
 *                    关键设计 1 (r_t formula), 关键设计 2 (clusters, segments,
 *                    local buffer), 关键设计 3 (group-consistent selection,
 *                    budgeted selection).
 *   [LouisKV blog]   "LouisKV: A New Approach to Efficient KV Cache Management
 *                    for Long Language Model Sequences" (edgentiq blog),
 *                    section "Decoupled Fine-Grained Management".
 *
 * Precision. Floating-point results are computed in double precision, with
 * two exceptions where a floating-point value decides an integer and the CUDA
 * kernels take that decision in single precision: the boundary statistic r_t
 * and the unit scores. For those the oracle evaluates the same single-precision
 * expression in the same operation order (documented at each function), so the
 * decision is the same on both sides. The K-means assignment is decided on the
 * double-precision squared distance.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (no FMA contraction:
 * every fused multiply-add in this file is an explicit fmaf call).
 */
#ifndef LKV_ORACLE_H
#define LKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { LKVO_FP32 = 0, LKVO_BF16 = 1 };

/* bfloat16 <-> float. Widening is exact; narrowing rounds to nearest even. */
float lkvo_bf16_to_f32(uint16_t b);
uint16_t lkvo_f32_to_bf16(float f);

/* K-means initialisation: the first c entries of a partial Fisher-Yates
 * shuffle of [0, n) driven by the splitmix64 sequence started at `seed`.
 * Returns 0, or -1 if c < 1 or c > n. [LouisKV notes, 关键设计 2]: the pages
 * fix no initialisation; this seeded rule is the reading adopted. */
int lkvo_init_indices(int64_t n, int32_t c, uint64_t seed, int64_t *idx_out);

/* The splitmix64 output sequence itself (for pinning against the published
 * reference values). */
void lkvo_splitmix64(uint64_t seed, int32_t count, uint64_t *out);

/* Squared Euclidean distance in double precision, summed over dimensions in
 * index order, each term (k_j - c_j)^2 formed with a separate subtract,
 * multiply and add. */
double lkvo_sqdist(const void *key, int dtype, const float *cent, int32_t d);

/* Lloyd assignment: assign_out[i] = argmin_j lkvo_sqdist(key_i, cent_j),
 * ties to the lowest j. `cent` holds the operand values (already rounded to
 * bf16 for bf16 keys). gap_out (optional): relative gap
 * (D_second - D_first) / (|k|^2 + |c_first|^2). */
void lkvo_assign(const void *keys, int dtype, int64_t n, int32_t d,
                 const float *cent, int32_t c, int32_t *assign_out,
                 double *gap_out);

/* Lloyd update: count_out[j] = #{i : assign[i] = j}; for non-empty j,
 * cent[j] = float( S_j / count_j ) with S_j the double-precision sum of the
 * member keys taken in token order. Empty clusters keep cent[j].
 * [LouisKV notes, 关键设计 2]: centroid = mean of the cluster's keys.
 * inexact_out (optional): set to the number of (cluster, dim) sums whose
 * double-precision accumulation rounded (detected with an exact two-sum). */
void lkvo_update(const void *keys, int dtype, int64_t n, int32_t d,
                 const int32_t *assign, int32_t c, float *cent,
                 int32_t *count_out, int64_t *inexact_out);

/* Operand centroid: bf16-rounded copy for bf16 keys, unchanged for fp32. */
void lkvo_operand(const float *cent, int64_t count, int dtype, float *out);

/* Objective J = sum_i sqdist(k_i, cent_{assign_i}) (cent = operand values). */
double lkvo_objective(const void *keys, int dtype, int64_t n, int32_t d,
                      const float *cent, const int32_t *assign);

/* Full K-means: init, then `iters` (>= 1) Lloyd rounds (assign with the
 * operand of the previous centroids, then update), no early stop.
 * trace_cent (optional): [iters+1][c][d] centroids before round 1..after round
 * iters; trace_assign (optional): [iters][n]. Returns 0 or -1. */
int lkvo_kmeans(const void *keys, int dtype, int64_t n, int32_t d, int32_t c,
                int32_t iters, uint64_t seed, float *cent_out,
                int32_t *assign_out, int32_t *count_out, float *trace_cent,
                int32_t *trace_assign, int64_t *inexact_out);

/* Boundary statistic r_t = (1/H) sum_h cos(q_{t-1}^h, q_t^h)
 * [LouisKV notes, 关键设计 1, formula r_t]. Single-precision form (the
 * decision value): per head, dot, |a|^2 and |b|^2 accumulate with fmaf in
 * index order; cos = dot / (sqrtf(|a|^2) * sqrtf(|b|^2)), 0 if that product is
 * 0; the head cosines are added in head order and the sum divided by H. */
float lkvo_boundary_r32(const void *q_prev, const void *q_cur, int dtype,
                        int32_t h, int32_t d);
/* The same statistic in double precision (for reporting the decision gap). */
double lkvo_boundary_r64(const void *q_prev, const void *q_cur, int dtype,
                         int32_t h, int32_t d);

/* Group-consistent unit scores [LouisKV notes, 关键设计 3 其二 and 关键设计 2
 * (dot product decides attention)]: qbar = sum of the group's g query heads
 * (single-precision adds in head order), s_u = qbar . cent_u accumulated with
 * fmaf in index order. `q` is [g][d]; `cent` is [u][d] operand values. */
void lkvo_group_scores(const void *q, int dtype, int32_t g, int32_t d,
                       const float *cent, int32_t u, float *scores_out);

/* Budgeted selection [LouisKV notes, 关键设计 3 其三]: order the units by
 * (score descending, id ascending); walk that order adding whole units while
 * the running token count stays <= budget; stop at the first unit that does
 * not fit. sel_out receives the ids in selection order. Returns the number of
 * units selected; *n_tok_out their total length. */
int32_t lkvo_select(const float *scores, const int32_t *len, int32_t u,
                    int32_t budget, int32_t *sel_out, int32_t *n_tok_out);

/* Skip-and-continue budget fill (a selection variant; the pages fix only the
 * stop-at-first-misfit rule above): walk the same (score descending, id
 * ascending) order and add every unit whose length still fits in what is left
 * of the budget, skipping the ones that do not. Same outputs as lkvo_select. */
int32_t lkvo_select_skip(const float *scores, const int32_t *len, int32_t u,
                         int32_t budget, int32_t *sel_out, int32_t *n_tok_out);

/* Softmax attention of g query heads over n rows, in double precision:
 * out_h = sum_i softmax_i(q_h . k_i / sqrt(d)) v_i. k_rows, v_rows: [n][d]. */
void lkvo_attention(const void *q, int dtype, int32_t g, int32_t d,
                    const void *k_rows, const void *v_rows, int64_t n,
                    double *out);

/* One (sequence, layer) decode run [LouisKV notes, 方法详解 flowchart and
 * 关键设计 1-2; LouisKV blog, Decoupled Fine-Grained Management]. */
typedef struct {
  int32_t dtype;
  int32_t n_kv_heads;   /* H_kv */
  int32_t group;        /* G query heads per KV head; H = H_kv * G */
  int32_t head_dim;     /* d */
  int64_t n_prefill;    /* N */
  int32_t n_clusters;   /* C */
  int32_t local_buf;    /* L >= 1 */
  int32_t n_steps;      /* T */
  float tau;
  int32_t budget;
  const void *keys;     /* [H_kv][N][d] prefill keys */
  const void *values;   /* [H_kv][N][d] prefill values */
  const int32_t *assign;/* [H_kv][N] cluster of each prefill token */
  const float *cent;    /* [H_kv][C][d] cluster centroids (fp32, unrounded) */
  const void *q;        /* [T][H][d] */
  const void *k_new;    /* [T][H_kv][d] */
  const void *v_new;    /* [T][H_kv][d] */
  const uint8_t *attn_mask; /* [T] compute attention only where nonzero; NULL = all */
  /* Retrieval policy; all zero is the method itself. The variants are the
   * baselines the pages compare it with [LouisKV notes, 研究背景与动机 (a
   * retrieval at every decode token, page-granular units) and 消融实验
   * (adaptive vs fixed step, fine-grained vs page units, group-consistent
   * selection)]. */
  int32_t trigger;      /* LKVO_TRIGGER_ADAPTIVE: t = 0 or r_t < tau;
                           LKVO_TRIGGER_EVERY: every step;
                           LKVO_TRIGGER_INTERVAL: t % interval == 0 */
  int32_t interval;     /* >= 1 with LKVO_TRIGGER_INTERVAL */
  int32_t fill;         /* LKVO_FILL_PREFIX (lkvo_select) or LKVO_FILL_SKIP (lkvo_select_skip) */
  int32_t page;         /* 0: the open decode segment closes at a retrieval step;
                           P >= 1: it closes once it holds P tokens (page units),
                           whatever the step does */
  int32_t per_head;     /* 0: one selection per KV head from the group's summed
                           query; 1: one per query head from its own query, and
                           each head attends its own selection */
  /* Selector: LKVO_SELECT_CLUSTERS (the method's units) or LKVO_SELECT_PARIS
   * (tokens ranked by the ParisKV-style coarse-to-fine pipeline below, over
   * the prefill tokens and the decode tokens that left the local buffer;
   * bf16 only, per_head 0). With PARIS the selection records hold token ids
   * (prefill token i, decode token t as n_prefill + t), best first. */
  int32_t selector;
  int32_t paris_rho;    /* sign centroids per subspace that vote */
  int32_t paris_n_cand; /* candidates kept for the rerank */
  uint64_t paris_seed;  /* sign flips of the rotation */
} lkvo_decode_args;

enum { LKVO_SELECT_CLUSTERS = 0, LKVO_SELECT_PARIS = 1 };

/* ------------------------------------------------------------------------ */
/* ParisKV-style selector [ParisKV technical summary, 核心算法创新 1 (l2
 * normalisation and a shared random orthogonal rotation by SRHT; analytic
 * sign centroids on the unit sphere) and 2 (collision voting over B
 * subspaces with the top-rho centroids of each, then a rerank of the
 * candidates by the calibrated estimate ||q|| sum_b w_b <v_b, q_b> from
 * 4-bit codes: 1 sign bit + 3 magnitude bits per coordinate from the Beta
 * prior that the rotation induces)]. Readings: the rotation is
 * H diag(D) / sqrt(d) with H the Sylvester-Hadamard matrix and D random
 * signs; a key is rotated exactly (its bf16 values as integers times 2^40);
 * the bucket of a subspace is the sign pattern of the rotated key there (the
 * nearest analytic centroid); the 3-bit magnitude of coordinate j of the
 * subspace direction u = y_b / |y_b| is the number of prior quantiles t_l
 * (l = 1..7, P(|x| < t_l) = l/8 for a coordinate x of a uniform unit vector
 * in R^m) at or below |u_j|, its value the prior's mean of |x| over that
 * bin; w_b = <y_b, v_b> / <v_b, v_b> (the least-squares scale of the
 * dequantised direction v_b, which holds |y_b| and the calibration); the
 * vote of the r-th best centroid (r = 0..rho-1) is rho - r; the constant
 * factor ||q|| of the estimate is dropped (it does not change the order). */

/* D_j = -1 where bit j % 64 of the (j / 64)-th splitmix64 output of seed is
 * set, else +1. */
void lkvo_paris_signs(uint64_t seed, int32_t d, int8_t *sign_out);

/* Quantiles and bin means of |x| for a coordinate x of a uniform unit vector
 * in R^m (density of x proportional to (1 - x^2)^((m-3)/2)), by Simpson
 * integration and bisection in double: thr_out[l-1] = float(t_l^2) for
 * l = 1..7, lev_out[l] = float(E[|x| : t_l <= |x| < t_{l+1}]) for l = 0..7
 * (t_0 = 0, t_8 = 1). Returns 0, or -1 for m < 2. */
int lkvo_paris_levels(int32_t m, float *thr_out, float *lev_out);

/* Metadata of one bf16 key (d dims, B = d / m subspaces, m = 8):
 * y = H D round_toward_zero(k * 2^40) in exact integers; bucket_out[b] = the
 * sign bits of y over subspace b (bit j set where y_{mb+j} < 0);
 * level_out[i] = #{l : y_i^2 >= thr[l] * n2_b} with n2_b = sum_j y_{mb+j}^2
 * (double products and adds in index order); w_out[b] = float of
 * (sum_j y_j v_j) / (sum_j v_j^2) * 2^-40 / sqrt(d), v_j = +-lev[level_j]
 * (double, index order). */
void lkvo_paris_encode(const uint16_t *key, int32_t d, const int8_t *sign, int32_t m,
                       const float *thr, const float *lev, uint8_t *bucket_out,
                       uint8_t *level_out, float *w_out);

/* The rotated group query in single precision: qbar = sum of the g heads
 * (adds in head order), x_j = D_j qbar_j, then the in-place fast Hadamard
 * butterfly over h = 1, 2, 4, ..., d/2 (pairs (j, j + h) -> (a + b, a - b)
 * within blocks of 2h, in index order). */
void lkvo_paris_rotate_query(const void *q, int dtype, int32_t g, int32_t d,
                             const int8_t *sign, float *qrot_out);

/* Token selection over n tokens with their metadata ([n][B] buckets, [n][d]
 * levels, [n][B] scales): per subspace the 2^m sign patterns p score
 * sim_p = sum_j (bit j of p ? -q_j : q_j) (single-precision adds in index
 * order); the best rho by (sim desc, p asc) vote rho - r; a token's coarse
 * score is the sum of its buckets' votes; the n_cand best tokens by (coarse
 * desc, id asc) are reranked by est = sum_b w_b dot_b, dot_b = sum_j v_j q_j
 * (fmaf chains in index order, est = fmaf(w_b, dot_b, est)); the budget best
 * by (est desc, id asc) are selected. sel_out receives their ids, best
 * first; coarse_out [n] and est_out [n] (optional) the scores (est only for
 * candidates, else 0). Returns the number selected. */
int64_t lkvo_paris_select(const float *qrot, int32_t d, int32_t m, int32_t rho,
                          int64_t n_cand, int32_t budget, int64_t n,
                          const uint8_t *bucket, const uint8_t *level, const float *w,
                          const float *lev, int64_t *sel_out, int32_t *coarse_out,
                          float *est_out);

enum { LKVO_TRIGGER_ADAPTIVE = 0, LKVO_TRIGGER_EVERY = 1, LKVO_TRIGGER_INTERVAL = 2 };
enum { LKVO_FILL_PREFIX = 0, LKVO_FILL_SKIP = 1 };

typedef struct {
  int32_t max_sel;      /* capacity of sel per (step, kv head) */
  int32_t max_segs;     /* capacity of the evicted-segment log */
  double *out;          /* [T][H][d] (steps masked out are left untouched) */
  uint8_t *flag;        /* [T] 1 = retrieval step */
  float *r32;           /* [T] decision value (0 at t = 0) */
  double *r64;          /* [T] double-precision r_t (0 at t = 0) */
  /* selection records: one per KV head, or per query head with per_head (Hs = H) */
  int32_t *n_sel;       /* [T][Hs] units in the active selection */
  int32_t *n_tok;       /* [T][Hs] tokens in the active selection */
  int32_t *sel;         /* [T][Hs][max_sel] active selection, selection order */
  int32_t *win_start;   /* [T] first decode token in the local buffer after the step */
  int32_t *n_units;     /* [T] units in the pool after the step's evictions */
  int32_t *seg_start;   /* [max_segs] first decode token of evicted segment e */
  int32_t *seg_len;     /* [max_segs] */
  float *seg_cent;      /* [max_segs][H_kv][d] or NULL */
  int32_t n_evicted;    /* out */
  int32_t n_forced;     /* out: segments cut because the buffer filled */
} lkvo_decode_result;

/* Returns 0, or -1 on bad arguments / capacity (max_sel < U or max_segs too
 * small) / allocation failure. */
int lkvo_decode(const lkvo_decode_args *a, lkvo_decode_result *r);

#ifdef __cplusplus
}
#endif
#endif
