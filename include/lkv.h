/*
 * lkv.h -- C ABI of liblkv, a single-GPU (GB300, sm_103a) implementation of
 * the data-parallel hot path of LouisKV-style KV-cache retrieval.
 *
 * Sources, cited by page title and section:
 *   [LouisKV notes]  "LouisKV: Efficient KV Cache Retrieval for Long
 *                    Input-Output Sequences" (papernotes.org summary):
 *                    方法详解/整体框架 (flowchart), 关键设计 1-3.
 *   [LouisKV blog]   "LouisKV: A New Approach to Efficient KV Cache Management
 *                    for Long Language Model Sequences": "Semantic-Aware
 *                    Adaptive Retrieval", "Decoupled Fine-Grained Management".
 *   [ParisKV]        "ParisKV" technical summary (gist.science): 系统级创新 1
 *                    (UVA offload: kernels fetch the chosen KV rows from host
 *                    memory directly).
 *
 * Conventions shared by every call:
 *   - d (head_dim) is 128. Query head h belongs to KV head h / group.
 *   - dtype LKV_DTYPE_BF16: keys, values and queries are bfloat16 (2 bytes,
 *     the upper half of an IEEE binary32); LKV_DTYPE_FP32: binary32.
 *     Accumulation is fp32 (attention, scores) or exact (centroid sums).
 *   - Pointers named "device" must be CUDA device (or managed) memory,
 *     readable by the current device; "host" pointers are ordinary host
 *     memory. The caller keeps ownership of everything it passes; the library
 *     copies what it needs to keep (keys and values into its own pool).
 *   - Calls that take device pointers are stream-ordered on the context's
 *     stream and return before the GPU work finishes; only lkv_sync,
 *     lkv_get_index and lkv_get_decode_state block.
 *   - Errors: every call returns an lkv_status; nothing is thrown across the
 *     ABI. lkv_last_error gives a one-line description. A device-side
 *     anomaly (capacity exceeded, a bounded wait that ran out) is recorded in
 *     the context and reported by the next lkv_sync as LKV_ECUDA /
 *     LKV_ECAPACITY / LKV_ETIMEOUT; a CUDA launch or runtime error is
 *     LKV_ECUDA and leaves the context unusable (LKV_ESTATE afterwards).
 */
#ifndef LKV_H
#define LKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LKV_OK = 0,
  LKV_EINVAL = 1,     /* bad argument, null pointer, shape outside the context */
  LKV_ENOMEM = 2,     /* device or pinned host allocation failed */
  LKV_ECUDA = 3,      /* CUDA runtime / launch error */
  LKV_ECAPACITY = 4,  /* more decode steps / units than the context was sized for */
  LKV_ESTATE = 5,     /* call out of order (decode before index) or broken context */
  LKV_ETIMEOUT = 6    /* a device-side bounded wait gave up */
} lkv_status;

typedef enum { LKV_DTYPE_FP32 = 0, LKV_DTYPE_BF16 = 1 } lkv_dtype;

typedef struct lkv_config {
  int32_t batch;        /* B sequences decoded together */
  int32_t n_layers;     /* attention layers with their own index and state */
  int32_t n_kv_heads;   /* H_kv */
  int32_t group;        /* G query heads per KV head (GQA), 1..8 */
  int32_t head_dim;     /* d; must be 128 */
  int32_t dtype;        /* lkv_dtype */
  int32_t local_buf;    /* L: tokens of the GPU local buffer of recent output
                           segments [LouisKV notes, 关键设计 2] */
  int32_t max_clusters; /* largest C a build may ask for */
  int64_t max_prefill;  /* largest N (prefill tokens per sequence), <= 2^18 */
  int32_t max_steps;    /* decode steps each layer may take */
  int32_t max_budget;   /* largest token budget a decode call may pass */
  int32_t offload;      /* 0: K/V pool in HBM. 1: prefill rows and evicted
                           segments in pinned host memory, read by the GPU
                           through unified virtual addressing [ParisKV, UVA
                           offload]; centroids and the local buffer stay in HBM */
  void *stream;         /* cudaStream_t for all work; NULL = legacy stream */
} lkv_config;

typedef struct lkv_ctx lkv_ctx;

/* Allocate a context sized by *cfg (device memory for the pool, index,
 * decode state and scratch; pinned host memory for the offloaded pool).
 * Ownership: the caller owns *cfg; the context owns everything it allocates
 * and frees it in lkv_destroy. Errors: LKV_EINVAL (shape), LKV_ENOMEM,
 * LKV_ECUDA. */
lkv_status lkv_create(const lkv_config *cfg, lkv_ctx **out);
void lkv_destroy(lkv_ctx *ctx);

/* Prefill index build for one layer [LouisKV notes, 关键设计 2; LouisKV blog,
 * Prefill Stage]: for every (sequence, KV head), K-means over its n_tokens
 * keys with n_clusters clusters and exactly `iters` Lloyd rounds (no early
 * stop); each cluster's centroid is the mean of its member keys and becomes
 * the retrieval index of a unit made of those tokens. The K/V rows are then
 * copied into the pool, grouped by cluster. Resets the layer's decode state.
 *
 * keys, values: device, [B][H_kv][n_tokens][d] in the context dtype.
 * Initialisation: slice s = b*H_kv + h takes as initial centroids the keys at
 * the first n_clusters indices of a partial Fisher-Yates shuffle of
 * [0, n_tokens) driven by the splitmix64 sequence seeded with seed + s.
 * Assignment: argmin of the squared Euclidean distance, evaluated exactly
 * (double precision, index order) wherever the fast tensor-core distance
 * cannot separate the two best centroids; ties go to the lowest cluster id.
 * Centroid arithmetic: member sum exact (or double, token order), divided in
 * double, rounded once to fp32; an empty cluster keeps its centroid. For
 * bf16, the scoring operand is the centroid rounded to bf16.
 * Errors: LKV_EINVAL (layer, sizes above the context capacities,
 * n_clusters > n_tokens, iters < 1), LKV_ECUDA. */
lkv_status lkv_build_index(lkv_ctx *ctx, int32_t layer, const void *keys,
                           const void *values, int64_t n_tokens,
                           int32_t n_clusters, int32_t iters, uint64_t seed);

/* lkv_build_index pipelined behind a producer [LouisKV notes, 关键设计 2 and
 * 关键设计 3 其一: the clustering (and the offload of the pool) overlaps the
 * prefill forward pass instead of blocking it]. The context's stream first
 * waits for ready_event (a cudaEvent_t recorded by the producer once this
 * layer's keys and values are complete, or NULL), then runs the build of
 * lkv_build_index; done_event (a cudaEvent_t, or NULL) is recorded on the
 * context's stream when the build has finished reading keys and values, so
 * the producer may reuse those buffers after waiting for it. With the context
 * on its own stream the build of layer l runs beside the producer's work on
 * layer l + 1; builds of several layers run one after another (they share the
 * K-means scratch). Events stay owned by the caller. Same result and errors as
 * lkv_build_index, plus LKV_ECUDA if an event cannot be waited on or
 * recorded. */
lkv_status lkv_build_index_async(lkv_ctx *ctx, int32_t layer, const void *keys,
                                 const void *values, int64_t n_tokens,
                                 int32_t n_clusters, int32_t iters, uint64_t seed,
                                 void *ready_event, void *done_event);

/* Teacher-forced index: same as lkv_build_index but with the assignment and
 * fp32 centroids given instead of computed (for parity runs from an external
 * index). assign: device int32 [B][H_kv][n_tokens], values in [0, n_clusters);
 * centroids: device fp32 [B][H_kv][n_clusters][d]. */
lkv_status lkv_load_index(lkv_ctx *ctx, int32_t layer, const void *keys,
                          const void *values, int64_t n_tokens,
                          int32_t n_clusters, const int32_t *assign,
                          const float *centroids);

/* One decode step for layers [layer, layer + n_layers), every sequence
 * [LouisKV notes, flowchart and 关键设计 1-3]. Per (sequence, layer):
 *  1. r_t = (1/H) sum_h cos(q_{t-1}^h, q_t^h); retrieval triggers at t = 0
 *     or when r_t < tau. r_t is evaluated in fp32: per head dot and squared
 *     norms by fused multiply-add in index order, cos = dot / (sqrt(|a|^2) *
 *     sqrt(|b|^2)) (0 when that is 0), head cosines added in head order.
 *  2. On a trigger the open output segment closes; token t opens the next.
 *  3. While the local buffer cannot take token t (it holds L tokens), its
 *     oldest closed segment is evicted into the pool as a new unit whose
 *     index is the mean of its keys (per KV head); with no closed segment
 *     left the open segment is cut and evicted.
 *  4. k_new/v_new of token t enter the local buffer.
 *  5. On a trigger, per KV head (group-consistent selection), every unit is
 *     scored with s_u = qbar . c_u, qbar = sum of the group's query heads
 *     (fp32 adds in head order), the dot by fp32 fused multiply-add in index
 *     order; units are taken in (score desc, id asc) order while their token
 *     total stays <= budget, stopping at the first that does not fit.
 *     Without a trigger the previous selection is reused unchanged.
 *  6. out = softmax(q K^T / sqrt(d)) V over the selected units' tokens and
 *     the local buffer (fp32 accumulate).
 * q: device [B][n_layers][H][d]; k_new, v_new: device [B][n_layers][H_kv][d]
 * (context dtype); tau: threshold; budget: tokens per (sequence, layer, KV
 * head), 0..max_budget; local_buf must equal the context's L.
 * Outputs (device; any may be NULL except out):
 *   out            fp32 [B][n_layers][H][d]
 *   selected_units int32 [B][n_layers][H_kv][max_clusters + max_steps]:
 *                  the active selection, ascending unit id (clusters are
 *                  units 0..C-1, evicted segments C, C+1, ... in eviction
 *                  order); entries past n_selected are left untouched
 *   n_selected     int32 [B][n_layers][H_kv]
 *   boundary       uint8 [B][n_layers]: 1 where this step retrieved
 *   r_out          fp32  [B][n_layers]: r_t (0 at t = 0)
 * Errors: LKV_EINVAL, LKV_ESTATE (layer has no index), LKV_ECAPACITY (layer
 * already took max_steps steps), LKV_ECUDA. */
lkv_status lkv_decode_step(lkv_ctx *ctx, int32_t layer, int32_t n_layers,
                           const void *q, const void *k_new, const void *v_new,
                           float tau, int32_t budget, int32_t local_buf,
                           float *out, int32_t *selected_units,
                           int32_t *n_selected, uint8_t *boundary,
                           float *r_out);

/* n_steps consecutive decode steps of layers [layer, layer + n_layers): the
 * same computation as n_steps calls of lkv_decode_step, with step i's
 * tensors at i * (one step's size) from each base pointer:
 *   q [n_steps][B][n_layers][H][d], k_new/v_new [n_steps][B][n_layers][H_kv][d],
 *   out [n_steps][B][n_layers][H][d], selected_units
 *   [n_steps][B][n_layers][H_kv][max_clusters + max_steps], n_selected
 *   [n_steps][B][n_layers][H_kv], boundary and r_out [n_steps][B][n_layers].
 * The steps run from captured CUDA graphs of 2048, 512, 128 and 64 steps,
 * longest first, each no longer than the context's step slots (max_steps
 * rounded up to 64, at most 2048), cached per argument set, so the host
 * issues one launch per graph; fewer than 64 left over run one at a time. Inside the graph one kernel runs the boundary tests and
 * segment bookkeeping of 64 steps at a time (they depend on the inputs
 * only); then, for an HBM pool (bf16, 4 or 8 query heads per KV head, at
 * most 1024 slices), one kernel scores and selects every retrieval of those
 * 64 steps side by side, and each step's attention runs on one of 16 side
 * streams, overlapping the attentions of other steps and the next chunk's
 * boundary and selection work (otherwise each step's selection runs on its
 * own, as in lkv_decode_step). The boundary flags, r_t and selections are
 * those of lkv_decode_step, and the attention outputs agree with it within
 * fp32 rounding (the split of a slice's rows over warps can differ). With
 * profiling enabled (lkv_set_profiling) the same kernels are launched one
 * after another on the context's stream (a boundary and a selection launch
 * per 64 steps where the chunked selection applies, else per step), each
 * bracketed by CUDA events. All layers of the call must have taken the same
 * number of steps
 * (LKV_EINVAL). Errors as lkv_decode_step. */
lkv_status lkv_decode_steps(lkv_ctx *ctx, int32_t layer, int32_t n_layers,
                            int32_t n_steps, const void *q, const void *k_new,
                            const void *v_new, float tau, int32_t budget,
                            int32_t local_buf, float *out, int32_t *selected_units,
                            int32_t *n_selected, uint8_t *boundary, float *r_out);

/* Retrieval policy of a context: the method itself (all fields zero, the
 * default) or one of the baselines the pages measure it against [LouisKV
 * notes, 研究背景与动机: earlier systems retrieve at every decode token and
 * manage KV in fixed pages; 消融实验: adaptive vs fixed retrieval step,
 * fine-grained vs page units, group-consistent selection]:
 *   trigger   LKV_TRIGGER_ADAPTIVE: retrieve at t = 0 or when r_t < tau.
 *             LKV_TRIGGER_EVERY: at every step. LKV_TRIGGER_INTERVAL: when
 *             t % interval == 0. r_t is computed and reported (r_out) under
 *             every trigger; tau matters only to the adaptive one.
 *   interval  >= 1 with LKV_TRIGGER_INTERVAL, else ignored.
 *   fill      LKV_FILL_PREFIX: units are taken in (score desc, id asc) order
 *             until the first that does not fit. LKV_FILL_SKIP: a unit that
 *             does not fit is skipped and the walk goes on, so every later
 *             unit that still fits is taken (a slice with more than 4096 units
 *             falls back to the prefix and lkv_sync reports LKV_ECAPACITY).
 *   page      0: an output segment closes at each retrieval step (step 2 of
 *             lkv_decode_step). P >= 1: it closes as soon as it holds P tokens
 *             whatever the trigger (fixed pages of the output; combine with
 *             lkv_build_pages for page units of the input).
 *   per_head  0: group-consistent selection (one per KV head from the sum of
 *             its query heads). 1: one selection per query head, scored with
 *             that head's own query (s_u = q_h . c_u) and filled to the budget
 *             on its own; each head attends its own selection and the local
 *             buffer (the rows are read once for the union of the group's
 *             selections). The decode outputs selected_units and n_selected
 *             then have one record per query head: [..][H][max_clusters +
 *             max_steps] and [..][H]. Needs an HBM pool, bf16, group 4 or 8,
 *             at most 1024 slices, max_prefill + max_steps < 2^24 and at most
 *             4096 units in a slice (LKV_ECAPACITY from lkv_sync beyond);
 *             the first call with per_head = 1 allocates the per-head
 *             records (LKV_ENOMEM).
 * The policy applies to the decode calls that follow (graphs captured before
 * are dropped; the call waits for the context's stream). Errors: LKV_EINVAL,
 * LKV_ENOMEM, LKV_ECUDA. */
enum { LKV_TRIGGER_ADAPTIVE = 0, LKV_TRIGGER_EVERY = 1, LKV_TRIGGER_INTERVAL = 2 };
enum { LKV_FILL_PREFIX = 0, LKV_FILL_SKIP = 1 };
typedef struct lkv_policy {
  int32_t trigger;
  int32_t interval;
  int32_t fill;
  int32_t page;
  int32_t per_head;
} lkv_policy;
lkv_status lkv_set_policy(lkv_ctx *ctx, const lkv_policy *policy);

/* Page-unit index for one layer, in place of lkv_build_index (the units of
 * the page-granular baselines [CTkvr, 1.1: block indexes mean-pool runs of
 * consecutive tokens]): unit j of every (sequence, KV head) holds prefill
 * tokens [j*page, (j+1)*page) (the last may be shorter), its index vector the
 * mean of their keys with the centroid arithmetic of lkv_build_index. Units:
 * ceil(n_tokens / page), at most max_clusters. keys, values as in
 * lkv_build_index. Resets the layer's decode state. Errors: LKV_EINVAL,
 * LKV_ECUDA. */
lkv_status lkv_build_pages(lkv_ctx *ctx, int32_t layer, const void *keys,
                           const void *values, int64_t n_tokens, int32_t page);

/* ParisKV-style token selector, a second workload on the same pool and
 * attention [ParisKV technical summary, 核心算法创新 1-2]. The prefill of the
 * layer is not clustered: its rows go to the pool in token order, and every
 * token (prefill, and each decode token as it is appended) gets compact
 * metadata of its key: the key, as exact integers k * 2^40 (bf16 values of
 * magnitude 2^-33 .. 2^22), is rotated by H diag(D) (H the 128 x 128
 * Sylvester-Hadamard matrix, D random signs from splitmix64(seed): bit j % 64
 * of output j / 64 set means -1) and split into 16 subspaces of 8; per
 * subspace the bucket is the sign pattern (the nearest of the 256 analytic
 * centroids), the code holds 3 magnitude bits per coordinate (how many of the
 * prior's 7 thresholds, lkv_paris_levels, the squared coordinate of the unit
 * subspace direction reaches), and w = <y_b, v_b> / <v_b, v_b> / (2^40 *
 * sqrt(128)) scales the dequantised direction v_b (signs times the prior's
 * bin means). At a retrieval step of a (sequence, layer, KV head), over the
 * prefill tokens and the decode tokens that left the local buffer: the
 * group's summed query (fp32 adds in head order) is rotated by the same D
 * and H (single-precision butterfly, strides 1, 2, ..., 64); in every
 * subspace the rho sign patterns with the largest sum of +-q (ties to the
 * lower pattern) give the tokens in their bucket rho, rho - 1, ..., 1 votes;
 * the n_cand tokens with the most votes (ties to the lower token) are
 * reranked by est = sum_b w_b <v_b, q_b> (fp32 fused multiply-adds, b and
 * then coordinate order); the `budget` best by (est desc, token asc) are the
 * selection, and every head of the group attends them and the local buffer.
 * Retrieval steps, segments and the local buffer follow the context's policy
 * as with clusters. selected_units then lists pool rows (prefill token i at
 * row i, decode token t at max_prefill + t), ascending.
 * keys, values: device bf16 [B][H_kv][n_tokens][d]. rho 1..15, n_cand
 * 1..4096; the first call fixes rho, n_cand and seed for the context (a
 * later call with others is LKV_EINVAL), allocates the metadata of every
 * pool row (144 bytes per row) and the vote scratch of the 128 step slots
 * (128 bytes per row) (LKV_ENOMEM), and drops captured graphs. The
 * context must be bf16, with an HBM pool, group 4 or 8, at most 1024
 * slices, max_clusters + max_steps >= max_budget, and no layer built by
 * lkv_build_index, lkv_build_pages or lkv_load_index (and those calls are
 * LKV_EINVAL on it afterwards); per-query-head selection does not apply.
 * Errors: LKV_EINVAL, LKV_ENOMEM, LKV_ECUDA. */
typedef struct lkv_paris_params {
  int32_t rho;
  int32_t n_cand;
  uint64_t seed;
} lkv_paris_params;
lkv_status lkv_build_paris(lkv_ctx *ctx, int32_t layer, const void *keys, const void *values,
                           int64_t n_tokens, const lkv_paris_params *params);

/* The ParisKV-style prior tables (host only, no GPU): for a coordinate x of
 * a uniform unit vector in R^8, thr[l-1] = float(t_l^2) where P(|x| < t_l) =
 * l / 8 (l = 1..7), and lev[l] = float(E[|x| : t_l <= |x| < t_{l+1}]) for
 * l = 0..7 (t_0 = 0, t_8 = 1). Errors: LKV_EINVAL (null pointer). */
lkv_status lkv_paris_levels(float *thr, float *lev);

/* Which kernel screens the K-means distances before the exact settlement.
 * LKV_FILTER_TENSOR (the default): tcgen05 tensor-core tiles, used for bf16
 * keys; fp32 keys always take the SIMT filter. LKV_FILTER_SIMT: the fp32
 * FMA filter for every dtype. Both certify their decisions against the exact
 * double-precision distance ("LouisKV ... Long Input-Output Sequences",
 * 关键设计 2: keys go to their nearest centroid), so the assignment and the
 * centroids do not depend on the choice; only the speed does.
 * Errors: LKV_EINVAL (null context or unknown value). */
enum { LKV_FILTER_TENSOR = 0, LKV_FILTER_SIMT = 1 };
lkv_status lkv_set_kmeans_filter(lkv_ctx *ctx, int32_t filter);

/* Per-kernel launch counts (always kept) and CUDA-event durations (kept while
 * profiling is enabled: each launch is bracketed by events on the context
 * stream). */
typedef struct lkv_kernel_stat {
  char name[24];
  int64_t launches;
  double total_ms;
} lkv_kernel_stat;

lkv_status lkv_set_profiling(lkv_ctx *ctx, int32_t enable);

/* Blocking. stats: host array of capacity entries (one per kernel kind; the
 * number of kinds goes to *n_stats). counters (optional, host int64[6]):
 * rows attended (K and V rows read by the attention), attention slices
 * processed, units scored, rows gathered from host memory, units selected,
 * tokens selected. reset != 0 zeroes everything afterwards. */
lkv_status lkv_get_profile(lkv_ctx *ctx, lkv_kernel_stat *stats, int32_t capacity,
                           int32_t *n_stats, int64_t *counters, int32_t reset);

/* Copy one (layer, sequence, KV head) index to host memory (blocks until the
 * context's stream is idle). Any output pointer may be NULL.
 *   centroids host fp32 [capacity][d]: units 0..n_units-1 (clusters, then
 *             evicted segments); unit_len, unit_row host int32 [capacity]:
 *             token count and first pool row of each unit (cluster rows are
 *             contiguous in the pool; segment rows start at max_prefill + the
 *             segment's first decode position); assign host int32 [n_tokens]
 *             (cluster of each prefill token); perm host int32 [n_tokens]:
 *             prefill token stored at pool row i.
 * *n_units receives the number of units; LKV_ECAPACITY if it exceeds
 * capacity (nothing copied). */
lkv_status lkv_get_index(lkv_ctx *ctx, int32_t layer, int32_t seq,
                         int32_t kv_head, int32_t capacity, float *centroids,
                         int32_t *unit_len, int32_t *unit_row, int32_t *assign,
                         int32_t *perm, int32_t *n_units);

typedef struct lkv_decode_state {
  int32_t t;            /* decode tokens appended so far */
  int32_t win_start;    /* first decode position held in the local buffer */
  int32_t open_start;   /* first decode position of the open segment */
  int32_t n_clusters;   /* C */
  int32_t n_units;      /* C + evicted segments (selectable units) */
  int32_t n_closed;     /* segments closed so far (evicted or not) */
  int32_t n_evicted;
  int32_t n_forced;     /* segments cut because the buffer filled */
  int64_t n_refined;    /* K-means assignments settled in double precision */
  int64_t n_inexact;    /* centroid sums that needed the double fallback */
} lkv_decode_state;

/* Allocation-free K-means of one (sequence, KV head) slice. The pages have
 * no counterpart to this call; it exists for callers that must not allocate
 * GPU memory themselves or through us: a process whose device memory is
 * owned by another allocator (a serving engine or framework that reserves
 * the whole GPU up front, so an extra cudaMalloc fails or fragments its
 * pool), or code that must not risk the implicit device synchronisation of
 * cudaMalloc/cudaFree. It computes exactly what lkv_build_index computes for
 * one slice (same Lloyd rounds, same bit-exact centroids and assignment),
 * without the K/V pool. The initialisation is drawn from `seed` as given:
 * lkv_build_index seeds slice s = b*H_kv + h with its seed + s, so to
 * reproduce slice s of a build, pass the build's seed + s.
 * keys: device, [n_tokens][d] in dtype; centroids: device fp32
 * [n_clusters][d], out; assign: device int32 [n_tokens], out; stream: a
 * cudaStream_t or NULL. Nothing is allocated: every intermediate lives in one
 * fixed array inside the library (about 2.7 MB, held by every GPU that loads
 * the library until the process exits), which limits n_tokens to 32768 and
 * n_clusters to 2048 (LKV_EINVAL beyond). All calls on a GPU share that
 * array and it keeps the previous call's contents, so calls that may
 * overlap on the GPU (different streams, different host threads) race: order
 * them on one stream. The first call on each device looks up the array's
 * device address and sets kernel attributes, so make that first call before
 * any stream capture; the address is kept for the life of the process, so
 * calls after a cudaDeviceReset are not supported. Asynchronous on stream;
 * errors returned at once: LKV_EINVAL, LKV_ECUDA (text via
 * lkv_last_error(NULL)). Device-side anomalies of the call (an overflowing
 * settlement queue, a failed invariant check) are recorded in the array and
 * kept until lkv_kmeans_static_status collects them. */
lkv_status lkv_kmeans_static(const void *keys, int32_t dtype, int64_t n_tokens,
                             int32_t n_clusters, int32_t iters, uint64_t seed,
                             float *centroids, int32_t *assign, void *stream);

/* Blocking companion of lkv_kmeans_static (it allocates nothing either):
 * waits for `stream`, then reports and clears the device-side anomalies that
 * the lkv_kmeans_static calls on the current device recorded since the last
 * status call: LKV_OK, LKV_ECAPACITY, LKV_ETIMEOUT or LKV_ECUDA (text via
 * lkv_last_error(NULL)). */
lkv_status lkv_kmeans_static_status(void *stream);

/* Blocking read of one (layer, sequence) decode state. */
lkv_status lkv_get_decode_state(lkv_ctx *ctx, int32_t layer, int32_t seq,
                                lkv_decode_state *out);

/* Host-link ceiling for the offload gather [ParisKV, 系统级创新 1: kernels
 * read the chosen K/V rows from host memory over UVA]: one kernel streams
 * `bytes` of pinned host memory (cudaHostAlloc / cudaHostRegister) into
 * device memory with plain 16-byte loads over UVA, a contiguous read with the
 * load pattern of the gather. host_src: pinned host, dev_dst: device, both
 * 16-byte aligned, bytes a multiple of 16. Asynchronous on `stream`
 * (cudaStream_t or NULL). Errors: LKV_EINVAL, LKV_ECUDA (text via
 * lkv_last_error(NULL)). */
lkv_status lkv_uva_read(const void *host_src, void *dev_dst, int64_t bytes, void *stream);

/* Single-launch read ceiling of device memory (no counterpart in the pages):
 * one kernel reads `bytes` of device memory at dev_src with plain 16-byte
 * loads over a grid that fills the GPU, and writes nothing the caller sees.
 * A decode step's attention reads its rows in one launch; timing this call
 * with CUDA events on the same number of bytes (L2 overwritten first) gives
 * the rate one launch of that size reaches. dev_src: device memory, 16-byte
 * aligned; bytes a multiple of 16. Asynchronous on `stream` (cudaStream_t or
 * NULL). Errors: LKV_EINVAL, LKV_ECUDA (text via lkv_last_error(NULL)). */
lkv_status lkv_read_ceiling(const void *dev_src, int64_t bytes, void *stream);

/* Failure-path check (no counterpart in the pages): launches, on the
 * context's stream, one CTA that waits on a barrier that nothing completes.
 * The wait gives up after limit_ns nanoseconds (0..1e9, else LKV_EINVAL) and
 * records the timeout in the context exactly as a decode or K-means kernel
 * whose bounded wait ran out, so the next lkv_sync returns LKV_ETIMEOUT and
 * clears it; the context stays usable. Asynchronous. */
lkv_status lkv_diag_wait_timeout(lkv_ctx *ctx, int64_t limit_ns);

/* Wait for the context's stream; report device-side anomalies. */
lkv_status lkv_sync(lkv_ctx *ctx);

/* Text of the last error on this context ("" if none); valid until the next
 * call on the context. NULL ctx: the last lkv_create failure. */
const char *lkv_last_error(const lkv_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif
