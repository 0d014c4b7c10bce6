// lkv_internal.cuh -- device-side layout and helpers shared by the liblkv
// translation units (K-means build, decode step, C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace lkv {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 8;
constexpr int kMaxParts = 64;      // token parts of the stable counting sort
constexpr int kAttnChunk = 64;     // tokens per attention work item
constexpr int kRing = 32;          // plan slots and attention scratch slots (see Pipe)
constexpr int kAttnStreams = 16;   // attention streams of a pipelined capture
constexpr int kChunk = 64;         // decode steps whose boundary tests one launch runs
constexpr int kMaxSlots = 32 * kChunk;  // step slots (queries, views) at most: the steps of the longest graph
constexpr int kAttnMaxSplit = 8;   // CTAs per slice in one attention launch, at most
constexpr int kStreamMaxSlices = 1024;  // slices of one call the streaming attention takes

// Error bits recorded on the device and reported by lkv_sync.
enum : int32_t {
  kErrCapacity = 1,  // a unit / selection / list capacity would overflow
  kErrTimeout = 2,   // a bounded device-side wait gave up
  kErrInternal = 4,  // an invariant check failed
};

// Decode state of one (layer, sequence).
struct DecState {
  int32_t t;           // decode tokens appended so far
  int32_t win_start;   // first decode position in the local buffer
  int32_t open_start;  // first decode position of the open segment
  int32_t n_clusters;  // C
  int32_t n_units;     // C + n_evicted
  int32_t n_closed;    // segments closed so far; segment e is unit C + e
  int32_t n_evicted;   // closed segments that left the buffer
  int32_t n_forced;
  int32_t flag;        // this step retrieves
  float r;             // this step's r_t
  int32_t seg_slow;    // open segment holds a value outside the exact-sum range
  int32_t plan;        // selection-plan slot (0..plan_ring-1) in force; a retrieval step advances it
  int32_t n_prefill;   // prefill tokens (read by the ParisKV-style selector)
};

// Everything a kernel needs to find the context's data. Per-slice arrays are
// indexed by the global slice gs = (layer * B + b) * Hkv + h; per-sequence
// arrays by lb = layer * B + b. Strides are in elements.
struct CtxView {
  int dtype;          // 0 fp32, 1 bf16
  int B, Hkv, G, d;
  int L;              // local buffer tokens
  int64_t n_cap;      // max prefill rows per slice
  int32_t t_cap;      // max decode steps
  int32_t u_cap;      // max units per slice (C_cap + T_cap)
  int32_t bud_cap;    // max token budget
  int32_t sel_cap;    // selected tokens a plan can hold: min(bud_cap, n_cap + t_cap)
  int32_t need_pieces;  // a reader of the copy pieces exists (host offload gather or the scalar attention)
  int offload;
  int64_t S_all;      // slices of all layers (n_layers * B * Hkv)
  int32_t n_lb;       // (layer, sequence) pairs (n_layers * B)
  // pool: prefill rows [0, n_cap) and evicted-segment rows [n_cap, n_cap+t_cap)
  void *pool_k, *pool_v;      // slice stride pool_rows * d (HBM or pinned host)
  int64_t pool_rows;
  // decode region (local buffer rows), decode position t at row t
  void *dec_k, *dec_v;        // slice stride dec_rows * d
  int64_t dec_rows;
  void *stage_k, *stage_v;    // offload only: [plan slot][slice][bud_cap][d]
  void *cent_op;              // [slice][u_cap][d] scoring operand (dtype)
  float *cent32;              // [slice][u_cap][d]
  int32_t *unit_row;          // [slice][u_cap]
  int32_t *unit_len;          // [slice][u_cap]
  int32_t *assign;            // [slice][n_cap]
  int32_t *perm;              // [slice][n_cap]
  DecState *st;               // [lb]
  void *q_prev;               // [lb][H][d] (dtype)
  int32_t n_slots;            // step slots: max_steps rounded up to kChunk, at most kMaxSlots
  float *q_attn;              // [n_slots step slots][lb][H][d] queries * log2(e)/sqrt(d), fp32
  int4 *aview;                // [n_slots][lb] (t, win_start, plan slot, 2 * units + flag)
  int4 *adesc;                // [n_slots][slice] (t, win_start, plan slot, selected tokens),
                              // written by the selection kernel on every step
  int64_t *segsum;            // [slice][d] exact fixed-point sums (bf16) or
                              // doubles reinterpreted (fp32)
  float *scores;              // chunk selection: [kChunk][slice][u_cap] per step of the chunk, else [slice][u_cap]
  // the selection plan, one copy per plan slot: [plan_ring][slice]...
  int32_t plan_ring;          // plan slots: 2 * kChunk + 1 with chunk selection, else kRing
  int32_t chunk_sel;          // one selection launch per chunk of steps (see launch_decode_steps)
  int32_t *sel;               // [plan_ring][slice][u_cap] selected unit ids, ascending
  int32_t *n_sel;             // [plan_ring][slice]
  int32_t *n_tok;             // [plan_ring][slice]
  int32_t *sel_rows;          // [plan_ring][slice][sel_cap] pool row of each selected token (HBM pool only)
  int4 *pieces;               // [slice][max_pieces] (src row, first token, length, 0)
  int32_t *chunk_piece;       // [slice][max_chunks + 1] first piece of each chunk
  int4 *chunk_pieces;         // [plan_ring][slice][max_chunks][64] the pieces of each chunk
  int32_t *chunk_count;       // [plan_ring][slice][max_chunks] pieces in each chunk
  int32_t max_pieces;
  int32_t *attn_count;        // [kRing][slice] attention CTAs / warps done (last one combines), by step slot mod kRing
  float *attn_wpart;          // [kRing][w_cap][G * d + 2 * G] per-warp partials of the streaming attention
  int32_t *sel_count;         // [kRing][slice] scoring CTAs done (the last one selects), by step slot mod kRing
  int32_t w_cap;              // warps the streaming attention may use in one launch
  float *attn_part;           // [kRing][slice][kAttnMaxSplit][G * d + 2 * G] CTA partials
  int32_t max_chunks;
  int32_t *err;               // device error bits (shared by all layers)
  int64_t *counters;          // [kCounters] work counters (see CounterId)
  // retrieval policy (all zero: the method; see lkv_policy)
  int32_t pol_trigger;        // 0 r_t < tau, 1 every step, 2 every pol_interval-th step
  int32_t pol_interval;
  int32_t pol_fill;           // 0 stop at the first unit that does not fit, 1 skip it and go on
  int32_t pol_page;           // 0: segments close at retrieval steps; P: once they hold P tokens
  int32_t pol_per_head;       // 1: a selection per query head (the attention reads their union)
  // per-query-head selection only (allocated when that policy is first set):
  uint8_t *sel_mask;          // [plan_ring][slice][u_cap] query heads that selected each listed unit
  int32_t *hsel_n;            // [plan_ring][slice][kMaxGroup] units selected by each query head
  int32_t *hsel_tok;          // [plan_ring][slice][kMaxGroup] their tokens
  // ParisKV-style token selector (all layers; set by lkv_build_paris)
  int32_t paris;              // 1: retrievals select tokens by the coarse-to-fine pipeline
  int32_t paris_rho;          // sign centroids per subspace that vote (1..15)
  int32_t paris_n_cand;       // candidates kept for the rerank (1..4096)
  uint64_t paris_sign[2];     // bit j set: coordinate j of the key / query is negated
  float paris_thr[7];         // prior thresholds on x^2
  float paris_lev[8];         // prior bin means of |x|
  uint8_t *pk_bucket;         // [slice][pool_rows][16] bucket (sign pattern) per subspace
  uint8_t *pk_code;           // [slice][pool_rows][64] 3-bit magnitude levels, two per byte
  float *pk_w;                // [slice][pool_rows][16] calibrated scale per subspace
  uint8_t *pk_score;          // [kChunk][slice][pk_pitch] vote sums of a step's region tokens (by step slot mod kChunk)
  int64_t pk_pitch;           // pool_rows rounded up to a multiple of 16
};

// Retrieval triggers and budget fills of the policy.
enum : int32_t { kTrigAdaptive = 0, kTrigEvery = 1, kTrigInterval = 2 };
enum : int32_t { kFillPrefix = 0, kFillSkip = 1 };

// Plan-slot views of the selection plan (plan_ring slots).
__host__ __device__ __forceinline__ int32_t *plan_sel(const CtxView &v, int p, int64_t gs) {
  return v.sel + ((int64_t)p * v.S_all + gs) * v.u_cap;
}
__host__ __device__ __forceinline__ int32_t *plan_nsel(const CtxView &v, int p, int64_t gs) {
  return v.n_sel + (int64_t)p * v.S_all + gs;
}
__host__ __device__ __forceinline__ int32_t *plan_ntok(const CtxView &v, int p, int64_t gs) {
  return v.n_tok + (int64_t)p * v.S_all + gs;
}
__host__ __device__ __forceinline__ int32_t *plan_sel_rows(const CtxView &v, int p, int64_t gs) {
  return v.sel_rows + ((int64_t)p * v.S_all + gs) * v.sel_cap;
}
__host__ __device__ __forceinline__ uint8_t *plan_sel_mask(const CtxView &v, int p, int64_t gs) {
  return v.sel_mask + ((int64_t)p * v.S_all + gs) * v.u_cap;
}
__host__ __device__ __forceinline__ int32_t *plan_hsel_n(const CtxView &v, int p, int64_t gs) {
  return v.hsel_n + ((int64_t)p * v.S_all + gs) * kMaxGroup;
}
__host__ __device__ __forceinline__ int32_t *plan_hsel_tok(const CtxView &v, int p, int64_t gs) {
  return v.hsel_tok + ((int64_t)p * v.S_all + gs) * kMaxGroup;
}
// Per-query-head selection stores the union's token rows with the mask of
// the heads that selected them in the top byte (pool rows stay below 2^24).
constexpr int kRowBits = 24;
constexpr int32_t kRowMask = (1 << kRowBits) - 1;
__host__ __device__ __forceinline__ int4 *plan_chunk_pieces(const CtxView &v, int p, int64_t gs) {
  return v.chunk_pieces + ((int64_t)p * v.S_all + gs) * v.max_chunks * 64;
}
__host__ __device__ __forceinline__ int32_t *plan_chunk_count(const CtxView &v, int p, int64_t gs) {
  return v.chunk_count + ((int64_t)p * v.S_all + gs) * v.max_chunks;
}

// Work counters accumulated on the device (read by lkv_get_profile).
enum CounterId : int { kCntAttnRows = 0, kCntScoreUnits = 1, kCntGatherRows = 2,
                       kCntAttnSlices = 3, kCntSelUnits = 4, kCntSelTokens = 5, kCounters = 8 };

// Kernel kinds for launch counting and event timing.
enum ProfKind : int {
  kPBoundary = 0, kPScore, kPGather, kPAttn,
  kPKmInit, kPKmOperand, kPKmAssign, kPKmRefine, kPKmSort, kPKmUpdate, kPKmPool, kPKmAssignTc,
  kPSelect,
  kPNum
};

// Host-side launch counter and (when enabled) CUDA-event timer: begin/end
// bracket the launches of one kernel kind on the context stream.
struct Prof {
  bool timing = false;
  bool counting = true;
  int64_t launches[kPNum] = {};
  double ms[kPNum] = {};
  struct Rec { int kind; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  int open_kind = -1;
  cudaEvent_t open_a = nullptr;

  cudaEvent_t take() {
    if (pool.empty()) {
      cudaEvent_t e = nullptr;
      cudaEventCreate(&e);
      return e;
    }
    cudaEvent_t e = pool.back();
    pool.pop_back();
    return e;
  }
  void begin(int kind, cudaStream_t s, int n = 1) {
    if (counting) launches[kind] += n;
    if (!timing) return;
    open_kind = kind;
    open_a = take();
    cudaEventRecord(open_a, s);
  }
  void end(cudaStream_t s) {
    if (!timing || open_kind < 0) return;
    cudaEvent_t b = take();
    cudaEventRecord(b, s);
    recs.push_back({open_kind, open_a, b});
    open_kind = -1;
    if (recs.size() >= 8192) resolve();
  }
  void resolve() {
    if (recs.empty()) return;
    cudaEventSynchronize(recs.back().b);
    for (const Rec &r : recs) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) ms[r.kind] += t;
      pool.push_back(r.a);
      pool.push_back(r.b);
    }
    recs.clear();
  }
  void release() {
    resolve();
    for (cudaEvent_t e : pool) cudaEventDestroy(e);
    pool.clear();
  }
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int DT>
__device__ __forceinline__ float load_elem(const void *p, int64_t i) {
  if constexpr (DT == 1) return bf16_bits_to_f32(((const uint16_t *)p)[i]);
  else return ((const float *)p)[i];
}

template <int DT>
__device__ __forceinline__ void store_elem(void *p, int64_t i, float v) {
  if constexpr (DT == 1) ((uint16_t *)p)[i] = f32_to_bf16_bits(v);
  else ((float *)p)[i] = v;
}

template <int DT>
constexpr int elem_bytes() { return DT == 1 ? 2 : 4; }

// Monotone map of a float (with -0 folded onto +0) to uint32 such that a
// larger score gives a SMALLER key: ascending key order = descending score.
__device__ __forceinline__ uint32_t desc_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  uint32_t asc = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ~asc;
}

// Exact fixed-point accumulation of bf16 values: v * 2^40 as int64 is exact
// for 2^-33 <= |v| < 32 (biased exponent 94..131) and the sum of up to 2^18
// such terms cannot overflow. Values outside 94..e_hi (other than zero) set
// *slow so the caller can fall back to double-precision token-order sums.
// The exact sum equals a token-order double sum only while every partial
// sum fits 53 bits, i.e. stays below 2^13 in magnitude: callers bound the
// sum of magnitudes, either through e_hi and the number of terms or with a
// running sum of |v|.
__device__ __forceinline__ int64_t bf16_fixed40(uint16_t bits, int *slow, uint32_t e_hi = 131u) {
  uint32_t e = (bits >> 7) & 0xffu;
  uint32_t m = bits & 0x7fu;
  if (e == 0 && m == 0) return 0;
  if (e < 94u || e > e_hi) { *slow = 1; return 0; }
  int64_t mag = (int64_t)(128u + m) << (e - 94u);
  return (bits & 0x8000u) ? -mag : mag;
}

__device__ __forceinline__ double fixed40_to_double(int64_t v) {
  // one correctly rounded conversion, then an exact power-of-two scale
  return __ll2double_rn(v) * 0x1p-40;
}

__device__ __forceinline__ void set_err(int32_t *err, int32_t bits) {
  atomicOr(err, bits);
}

// ---------------------------------------------------------------- launchers

struct KmeansScratch {
  float *knorm;        // [S][n_cap]
  float *c2;           // [S][c2_pitch]: |c|^2 of the operand centroids
  int32_t c2_pitch;    // c_cap rounded up to a multiple of 256
  uint16_t *c2b;       // [S][c2_pitch][16] bf16: -|c|^2 / 2 as a high part and remainder, then zeros
  float *cstat;        // [S][2]: max |c|, max |c|^2
  int32_t *cnt_part;   // [S][kMaxParts][c_cap] counts, then running offsets
  int32_t *count;      // [S][c_cap]
  int32_t *offs;       // [S][c_cap]
  int4 *amb;           // [S * n_cap] ambiguous assignments
  int32_t *amb_count;  // [2]: two-candidate entries (front), crowded entries (back)
  int64_t *n_refined;  // [1] running total
  int64_t *n_inexact;  // [1] running total
  int64_t *init_idx;   // [S][c_cap]
};

// K-means build of one layer (all slices). keys/values: [S][n][d] device.
cudaError_t launch_kmeans_build(const CtxView &v, int layer, const KmeansScratch &ks,
                                const void *keys, const void *values, int64_t n,
                                int32_t c, int32_t iters, bool use_tc,
                                cudaStream_t stream, Prof &prof);
// Page-mean index of one layer: unit j holds prefill tokens [j*page,
// (j+1)*page) of every slice, its index vector the mean of their keys.
cudaError_t launch_page_index(const CtxView &v, int layer, const KmeansScratch &ks,
                              const void *keys, const void *values, int64_t n, int32_t page,
                              cudaStream_t stream, Prof &prof);
// ParisKV-style index of one layer: the pool in token order (no clusters)
// and every prefill token's metadata.
cudaError_t launch_paris_index(const CtxView &v, int layer, const KmeansScratch &ks,
                               const void *keys, const void *values, int64_t n,
                               cudaStream_t stream, Prof &prof);
// Prior thresholds (x^2) and bin means of |x| for m = 8 (host, closed form).
void paris_levels_host(float thr[7], float lev[8]);
// Pool and unit table from a given assignment and fp32 centroids.
cudaError_t launch_load_index(const CtxView &v, int layer, const KmeansScratch &ks,
                              const void *keys, const void *values, int64_t n,
                              int32_t c, const int32_t *assign,
                              const float *cent, cudaStream_t stream, Prof &prof);

// Inputs and outputs of one decode step are found at base + k * stride where
// k = (tokens the sequence's layer had appended before this step) - base_t:
// a single-step call passes strides 0; a multi-step call passes per-step
// strides (and bases shifted so that base_t = 0), so that one captured step
// replays unchanged from a CUDA graph.
struct StepArgs {
  const void *q, *k_new, *v_new;   // [B][nl][H][d], [B][nl][Hkv][d]
  int32_t base_t;                  // decode position of the call's first step
  int64_t stride_q, stride_kv;     // elements between consecutive steps' inputs
  int64_t stride_out, stride_sel, stride_nsel, stride_b;  // outputs, per step
  float tau;
  int32_t budget;
  float *out;                      // [B][nl][H][d]
  int32_t *selected_units;         // [B][nl][Hkv][u_cap] or null
  int32_t *n_selected;             // [B][nl][Hkv] or null
  uint8_t *boundary;               // [B][nl] or null
  float *r_out;                    // [B][nl] or null
  int32_t l0;                      // first layer of this call
  int32_t slot;                    // step slot (queries, views): the step's index in a
                                   // captured graph (0 .. n_slots - 1), else 0; the
                                   // attention's scratch is slot mod kRing
  int32_t nl;                      // layers in this call
};

// Streams and events of a pipelined multi-step capture, three lanes:
//  - one boundary kernel per chunk of kChunk steps on the capture stream
//    (the decode state chain), writing every step's slot (queries and view);
//    the chunks of a graph use distinct slots;
//  - scoring/selection (and the offload gather) on `sel`, the chunk's steps
//    after its boundary kernel (b_done), each step after the previous one
//    (programmatic dependent launch). Every kSelWaitStride-th step's
//    selection i also waits for step i - kAttnStreams's attention: then at
//    any selection j the attentions still running are within the
//    kAttnStreams + kSelWaitStride - 1 steps before j (fewer than kRing), so
//    a retrieval's plan slot ((retrievals so far) mod kRing) is read by no
//    running attention, and step j's attention scratch (j mod kRing) is
//    free. Selections read the step's view, never the live state, and a
//    boundary kernel only writes units above the unit count a pending
//    selection reads;
//  - step i's attention on attn[i % kAttnStreams], after its selection (sel_done).
// With chunk selection the selection lane runs one launch per chunk instead,
// each after its chunk's boundary kernel and the previous chunk's selection,
// and chunk j's selection also waits until every attention of chunk j - 2
// has finished (chunk_done): the attentions still running then belong to
// chunk j - 1, whose steps and chunk j's are at most 2 * kChunk retrievals
// apart, so with plan_ring = 2 * kChunk + 1 no plan slot that a running
// attention reads is written.
constexpr int kSelWaitStride = 8;
static_assert(kAttnStreams + kSelWaitStride - 1 < kRing, "plan ring too small for the attentions in flight");
struct Pipe {
  cudaStream_t sel;
  cudaStream_t attn[kAttnStreams];
  cudaEvent_t b_done, sel_done;
  cudaEvent_t attn_done[kAttnStreams];
  // chunk selection: chunk j's attentions all done (joined on `join`), in
  // three rotating events; chunk j + 2's selection waits for it (see
  // launch_decode_steps)
  cudaStream_t join;
  cudaEvent_t chunk_done[3];
  int step;  // index of the chunk's first step in the capture
};

// n_steps consecutive decode steps (step i in slot a.slot + i): one boundary
// launch for all of them, then each step's scoring, selection and attention;
// with `pipe` (graph capture only) the lanes are forked as described above.
cudaError_t launch_decode_steps(const CtxView &v, const StepArgs &a, int n_steps, cudaStream_t stream,
                                Prof &prof, const Pipe *pipe = nullptr);
// Streaming read of `bytes` (a multiple of 16) of pinned host memory into
// device memory by plain 16-byte loads over UVA (the host-link ceiling).
cudaError_t launch_uva_read(const void *host_src, void *dev_dst, int64_t bytes, cudaStream_t stream);
cudaError_t launch_read_ceiling(const void *src, int64_t bytes, cudaStream_t stream);
// One CTA whose bounded wait on a barrier nobody completes runs out after
// limit_ns and records kErrTimeout (tests the failure path).
cudaError_t launch_diag_wait(const CtxView &v, uint64_t limit_ns, cudaStream_t stream);
// Error text of calls that have no context (read with lkv_last_error(NULL)).
void set_unbound_error(const char *msg);
// Per-warp partial slots the streaming attention needs on a GPU with `sms`
// multiprocessors (the most warps one launch may use).
int stream_warp_cap(int sms);
// One-time kernel attributes (dynamic shared memory limits), before any capture.
cudaError_t prepare_kernels(int dtype, int group);

}  // namespace lkv
