// api.cu -- the C ABI of liblkv (declared in include/lkv.h): context
// allocation, argument checks, stream-ordered launches, blocking queries.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/lkv.h"
#include "lkv_internal.cuh"
#include "paris.cuh"

using lkv::CtxView;
using lkv::DecState;
using lkv::KmeansScratch;

struct GraphEntry {
  lkv::StepArgs args{};
  int steps = 0;
  cudaGraphExec_t exec = nullptr;
};

struct lkv_ctx {
  lkv_config cfg{};
  CtxView v{};
  KmeansScratch ks{};
  cudaStream_t stream = nullptr;
  cudaStream_t capture = nullptr;   // private stream for CUDA-graph capture
  lkv::Pipe pipe{};                 // side streams and events of a pipelined capture
  lkv::Prof prof;
  std::vector<GraphEntry> graphs;
  std::vector<void *> dev;
  std::vector<void *> host;
  std::vector<int32_t> steps;     // decode steps taken per layer
  std::vector<int8_t> built;      // index present per layer (1 clusters or pages, 2 ParisKV-style)
  std::vector<int64_t> n_tokens;  // prefill tokens per layer
  std::vector<int32_t> n_clusters;
  std::string err;
  bool broken = false;
  bool use_tc = true;             // tensor-core distance filter for bf16 keys
  int alloc_index = 0;
  int fail_at = -1;               // host-side allocation-failure injection
  uint64_t paris_seed = 0;        // seed of the ParisKV-style selector's signs
};

static thread_local std::string g_create_error;

namespace lkv {
// Error text of calls that have no context (read with lkv_last_error(NULL)).
void set_unbound_error(const char *msg) { g_create_error = msg; }
}  // namespace lkv

static lkv_status fail(lkv_ctx *c, lkv_status s, const std::string &msg) {
  if (c) c->err = msg;
  else g_create_error = msg;
  return s;
}

static lkv_status cuda_fail(lkv_ctx *c, cudaError_t e, const char *where) {
  if (c) c->broken = true;
  return fail(c, LKV_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

static void *dalloc(lkv_ctx *c, size_t bytes, lkv_status *st) {
  if (*st != LKV_OK) return nullptr;
  if (c->fail_at >= 0 && c->alloc_index++ == c->fail_at) {
    *st = fail(c, LKV_ENOMEM, "injected allocation failure");
    return nullptr;
  }
  void *p = nullptr;
  if (cudaMalloc(&p, bytes < 16 ? 16 : bytes) != cudaSuccess) {
    cudaGetLastError();
    *st = fail(c, LKV_ENOMEM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
    return nullptr;
  }
  c->dev.push_back(p);
  return p;
}

static void *halloc(lkv_ctx *c, size_t bytes, lkv_status *st) {
  if (*st != LKV_OK) return nullptr;
  if (c->fail_at >= 0 && c->alloc_index++ == c->fail_at) {
    *st = fail(c, LKV_ENOMEM, "injected allocation failure");
    return nullptr;
  }
  void *p = nullptr;
  if (cudaHostAlloc(&p, bytes < 16 ? 16 : bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    cudaGetLastError();
    *st = fail(c, LKV_ENOMEM, "pinned host allocation of " + std::to_string(bytes) + " bytes failed");
    return nullptr;
  }
  c->host.push_back(p);
  return p;
}

static void free_all(lkv_ctx *c) {
  for (GraphEntry &g : c->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  c->graphs.clear();
  c->prof.release();
  if (c->capture) cudaStreamDestroy(c->capture);
  c->capture = nullptr;
  for (int i = 0; i < lkv::kAttnStreams; ++i) {
    if (c->pipe.attn[i]) cudaStreamDestroy(c->pipe.attn[i]);
    if (c->pipe.attn_done[i]) cudaEventDestroy(c->pipe.attn_done[i]);
    c->pipe.attn[i] = nullptr;
    c->pipe.attn_done[i] = nullptr;
  }
  for (int i = 0; i < 3; ++i) {
    if (c->pipe.chunk_done[i]) cudaEventDestroy(c->pipe.chunk_done[i]);
    c->pipe.chunk_done[i] = nullptr;
  }
  if (c->pipe.join) cudaStreamDestroy(c->pipe.join);
  c->pipe.join = nullptr;
  if (c->pipe.sel_done) cudaEventDestroy(c->pipe.sel_done);
  if (c->pipe.b_done) cudaEventDestroy(c->pipe.b_done);
  if (c->pipe.sel) cudaStreamDestroy(c->pipe.sel);
  c->pipe.sel_done = c->pipe.b_done = nullptr;
  c->pipe.sel = nullptr;
  for (void *p : c->dev) cudaFree(p);
  for (void *p : c->host) cudaFreeHost(p);
  c->dev.clear();
  c->host.clear();
}

// splitmix64 (Steele, Lea and Flood, OOPSLA 2014), the seeded source of the
// K-means initialisation.
static uint64_t splitmix64_next(uint64_t &state) {
  uint64_t z = (state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// First c entries of a partial Fisher-Yates shuffle of [0, n).
static void init_indices(int64_t n, int32_t c, uint64_t seed, int64_t *out,
                         std::vector<int64_t> &perm) {
  perm.resize((size_t)n);
  for (int64_t i = 0; i < n; ++i) perm[(size_t)i] = i;
  uint64_t st = seed;
  for (int32_t i = 0; i < c; ++i) {
    const uint64_t r = splitmix64_next(st);
    const int64_t j = (int64_t)i + (int64_t)(r % (uint64_t)(n - i));
    std::swap(perm[(size_t)i], perm[(size_t)j]);
    out[i] = perm[(size_t)i];
  }
}

extern "C" {

lkv_status lkv_create(const lkv_config *cfg, lkv_ctx **out) {
  if (!cfg || !out) return fail(nullptr, LKV_EINVAL, "null argument");
  *out = nullptr;
  const lkv_config &k = *cfg;
  if (k.head_dim != 128) return fail(nullptr, LKV_EINVAL, "head_dim must be 128");
  if (!(k.group == 1 || k.group == 2 || k.group == 4 || k.group == 8))
    return fail(nullptr, LKV_EINVAL, "group must be 1, 2, 4 or 8");
  if (k.n_kv_heads < 1 || k.n_kv_heads > 16) return fail(nullptr, LKV_EINVAL, "n_kv_heads must be 1..16");
  if (k.batch < 1 || k.n_layers < 1) return fail(nullptr, LKV_EINVAL, "batch and n_layers must be >= 1");
  if (k.dtype != LKV_DTYPE_FP32 && k.dtype != LKV_DTYPE_BF16) return fail(nullptr, LKV_EINVAL, "bad dtype");
  if (k.local_buf < 1) return fail(nullptr, LKV_EINVAL, "local_buf must be >= 1");
  if (k.max_clusters < 1 || k.max_clusters > 12288) return fail(nullptr, LKV_EINVAL, "max_clusters must be 1..12288");
  if (k.max_prefill < 1 || k.max_prefill > (int64_t(1) << 18)) return fail(nullptr, LKV_EINVAL, "max_prefill must be 1..2^18");
  if (k.max_steps < 1 || k.max_budget < 0) return fail(nullptr, LKV_EINVAL, "max_steps >= 1 and max_budget >= 0 required");
  if ((int64_t)k.max_clusters + k.max_steps >= (int64_t(1) << 30)) return fail(nullptr, LKV_EINVAL, "too many units");
  if (k.max_budget > (int64_t(1) << 30)) return fail(nullptr, LKV_EINVAL, "max_budget too large");

  lkv_ctx *c = new lkv_ctx();
  c->cfg = k;
  c->stream = (cudaStream_t)k.stream;
  if (const char *e = std::getenv("LKV_FAIL_ALLOC_AFTER")) c->fail_at = std::atoi(e);
  const int B = k.batch, NL = k.n_layers, Hkv = k.n_kv_heads, G = k.group, d = 128;
  const int H = Hkv * G;
  const size_t es = k.dtype == LKV_DTYPE_BF16 ? 2 : 4;
  const int64_t n_cap = k.max_prefill;
  const int32_t t_cap = k.max_steps, c_cap = k.max_clusters, u_cap = c_cap + t_cap;
  const int64_t S_all = (int64_t)NL * B * Hkv, LB = (int64_t)NL * B, S = (int64_t)B * Hkv;
  const int64_t pool_rows = n_cap + t_cap;
  const int32_t max_chunks = (k.max_budget + k.local_buf + lkv::kAttnChunk - 1) / lkv::kAttnChunk;

  lkv_status st = LKV_OK;
  CtxView &v = c->v;
  v.dtype = k.dtype;
  v.pol_interval = 1;
  v.B = B; v.Hkv = Hkv; v.G = G; v.d = d; v.L = k.local_buf;
  v.n_cap = n_cap; v.t_cap = t_cap; v.u_cap = u_cap; v.bud_cap = k.max_budget;
  v.offload = k.offload ? 1 : 0;
  // the tensor-core attention (bf16, 4 or 8 query heads per KV head) reads
  // the per-token rows; the pieces serve the host gather and the scalar attention
  v.need_pieces = (v.offload || !(k.dtype == 1 && (G == 4 || G == 8))) ? 1 : 0;
  // the streaming attention over an HBM pool takes its selections from one
  // launch per chunk of steps, with a plan ring for two chunks
  v.chunk_sel = (!v.offload && !v.need_pieces && S_all <= lkv::kStreamMaxSlices) ? 1 : 0;
  v.plan_ring = v.chunk_sel ? 2 * lkv::kChunk + 1 : lkv::kRing;
  const int64_t R = v.plan_ring;
  v.S_all = S_all;
  v.n_lb = (int32_t)LB;
  v.pool_rows = pool_rows;
  if (!k.offload) {
    v.pool_k = dalloc(c, S_all * pool_rows * d * es, &st);
    v.pool_v = dalloc(c, S_all * pool_rows * d * es, &st);
    if (st == LKV_OK) {
      v.dec_k = (char *)v.pool_k + n_cap * d * es;
      v.dec_v = (char *)v.pool_v + n_cap * d * es;
    }
    v.dec_rows = pool_rows;
  } else {
    v.pool_k = halloc(c, S_all * pool_rows * d * es, &st);
    v.pool_v = halloc(c, S_all * pool_rows * d * es, &st);
    v.dec_k = dalloc(c, S_all * t_cap * d * es, &st);
    v.dec_v = dalloc(c, S_all * t_cap * d * es, &st);
    v.dec_rows = t_cap;
    v.stage_k = dalloc(c, R * S_all * (int64_t)k.max_budget * d * es, &st);  // per plan slot
    v.stage_v = dalloc(c, R * S_all * (int64_t)k.max_budget * d * es, &st);
  }
  v.cent_op = dalloc(c, S_all * u_cap * d * es, &st);
  v.cent32 = (float *)dalloc(c, S_all * u_cap * d * 4, &st);
  v.unit_row = (int32_t *)dalloc(c, S_all * u_cap * 4, &st);
  v.unit_len = (int32_t *)dalloc(c, S_all * u_cap * 4, &st);
  v.assign = (int32_t *)dalloc(c, S_all * n_cap * 4, &st);
  v.perm = (int32_t *)dalloc(c, S_all * n_cap * 4, &st);
  v.st = (DecState *)dalloc(c, LB * sizeof(DecState), &st);
  v.q_prev = dalloc(c, LB * H * d * es, &st);
  // step slots: a captured graph of up to kMaxSlots steps, no longer than
  // the context's steps need
  v.n_slots = (int32_t)std::min<int64_t>(lkv::kMaxSlots, ((int64_t)t_cap + lkv::kChunk - 1) / lkv::kChunk * lkv::kChunk);
  const int64_t NS = v.n_slots;
  v.q_attn = (float *)dalloc(c, NS * LB * H * d * 4, &st);  // per step slot
  v.aview = (int4 *)dalloc(c, NS * LB * sizeof(int4), &st);
  v.adesc = (int4 *)dalloc(c, NS * S_all * sizeof(int4), &st);
  v.segsum = (int64_t *)dalloc(c, S_all * d * 8, &st);
  v.scores = (float *)dalloc(c, (v.chunk_sel ? lkv::kChunk : 1) * S_all * u_cap * 4, &st);
  // the selection plan, one copy per plan slot
  v.sel = (int32_t *)dalloc(c, R * S_all * u_cap * 4, &st);
  v.n_sel = (int32_t *)dalloc(c, R * S_all * 4, &st);
  v.n_tok = (int32_t *)dalloc(c, R * S_all * 4, &st);
  v.sel_cap = (int32_t)std::min<int64_t>(k.max_budget, (int64_t)n_cap + t_cap);
  if (!k.offload) v.sel_rows = (int32_t *)dalloc(c, R * S_all * (int64_t)v.sel_cap * 4, &st);
  v.max_chunks = max_chunks;
  v.attn_count = (int32_t *)dalloc(c, lkv::kRing * S_all * 4, &st);
  v.sel_count = (int32_t *)dalloc(c, lkv::kRing * S_all * 4, &st);
  v.attn_part = (float *)dalloc(c, lkv::kRing * S_all * lkv::kAttnMaxSplit *
                                       (int64_t)(k.group * d + 2 * k.group) * 4, &st);
  if (st == LKV_OK) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      sms = 160;
    }
    v.w_cap = lkv::stream_warp_cap(sms);
  }
  v.attn_wpart = (float *)dalloc(c, lkv::kRing * (int64_t)v.w_cap *
                                        (int64_t)(k.group * d + 2 * k.group) * 4, &st);
  v.max_pieces = u_cap + max_chunks;
  const int64_t pc = v.need_pieces ? 1 : 0;  // the copy pieces exist only where a reader needs them
  v.pieces = (int4 *)dalloc(c, pc * S_all * (int64_t)v.max_pieces * sizeof(int4), &st);
  v.chunk_piece = (int32_t *)dalloc(c, pc * S_all * (int64_t)(max_chunks + 1) * 4, &st);
  v.chunk_pieces = (int4 *)dalloc(c, pc * R * S_all * (int64_t)max_chunks * lkv::kAttnChunk * sizeof(int4), &st);
  v.chunk_count = (int32_t *)dalloc(c, pc * R * S_all * (int64_t)max_chunks * 4, &st);
  v.err = (int32_t *)dalloc(c, 4, &st);
  v.counters = (int64_t *)dalloc(c, lkv::kCounters * 8, &st);

  KmeansScratch &ks = c->ks;
  ks.knorm = (float *)dalloc(c, S * n_cap * 4, &st);
  ks.c2_pitch = (c_cap + 255) / 256 * 256;
  ks.c2 = (float *)dalloc(c, S * ks.c2_pitch * 4, &st);
  ks.c2b = (uint16_t *)dalloc(c, S * ks.c2_pitch * 32, &st);
  ks.cstat = (float *)dalloc(c, S * 2 * 4, &st);
  ks.cnt_part = (int32_t *)dalloc(c, S * lkv::kMaxParts * c_cap * 4, &st);
  ks.count = (int32_t *)dalloc(c, S * c_cap * 4, &st);
  ks.offs = (int32_t *)dalloc(c, S * c_cap * 4, &st);
  ks.amb = (int4 *)dalloc(c, S * n_cap * sizeof(int4), &st);
  ks.amb_count = (int32_t *)dalloc(c, 8, &st);  // front and back ends of the queue
  ks.n_refined = (int64_t *)dalloc(c, 8, &st);
  ks.n_inexact = (int64_t *)dalloc(c, 8, &st);
  ks.init_idx = (int64_t *)dalloc(c, S * c_cap * 8, &st);
  if (st != LKV_OK) {
    g_create_error = c->err;
    free_all(c);
    delete c;
    return st;
  }
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMemsetAsync(v.st, 0, LB * sizeof(DecState), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.attn_count, 0, lkv::kRing * S_all * 4, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.sel_count, 0, lkv::kRing * S_all * 4, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.err, 0, 4, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ks.n_refined, 0, 8, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ks.n_inexact, 0, 8, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.counters, 0, lkv::kCounters * 8, c->stream);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->capture, cudaStreamNonBlocking);
  for (int i = 0; i < lkv::kAttnStreams; ++i) {
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->pipe.attn[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->pipe.attn_done[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->pipe.sel_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->pipe.b_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->pipe.sel, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->pipe.join, cudaStreamNonBlocking);
  for (int i = 0; i < 3; ++i)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->pipe.chunk_done[i], cudaEventDisableTiming);
  if (e == cudaSuccess) e = lkv::prepare_kernels(k.dtype, k.group);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    g_create_error = std::string("initialisation: ") + cudaGetErrorString(e);
    free_all(c);
    delete c;
    return LKV_ECUDA;
  }
  c->steps.assign(NL, 0);
  c->built.assign(NL, 0);
  c->n_tokens.assign(NL, 0);
  c->n_clusters.assign(NL, 0);
  *out = c;
  return LKV_OK;
}

void lkv_destroy(lkv_ctx *c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  free_all(c);
  delete c;
}

static lkv_status check_usable(lkv_ctx *c) {
  if (!c) return LKV_EINVAL;
  if (c->broken) return fail(c, LKV_ESTATE, "context is unusable after a CUDA error");
  return LKV_OK;
}

lkv_status lkv_build_index(lkv_ctx *c, int32_t layer, const void *keys, const void *values,
                           int64_t n, int32_t nc, int32_t iters, uint64_t seed) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (c->v.paris) return fail(c, LKV_EINVAL, "the context uses the ParisKV-style selector");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(c, LKV_EINVAL, "layer out of range");
  if (!keys || !values) return fail(c, LKV_EINVAL, "null keys or values");
  if (n < 1 || n > c->cfg.max_prefill) return fail(c, LKV_EINVAL, "n_tokens outside 1..max_prefill");
  if (nc < 1 || nc > c->cfg.max_clusters || nc > n)
    return fail(c, LKV_EINVAL, "n_clusters outside 1..min(max_clusters, n_tokens)");
  if (iters < 1) return fail(c, LKV_EINVAL, "iters must be >= 1");
  const int S = c->cfg.batch * c->cfg.n_kv_heads;
  std::vector<int64_t> idx((size_t)S * nc), perm;
  for (int sl = 0; sl < S; ++sl) init_indices(n, nc, seed + (uint64_t)sl, idx.data() + (size_t)sl * nc, perm);
  cudaError_t e = cudaMemcpyAsync(c->ks.init_idx, idx.data(), idx.size() * 8, cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess) e = lkv::launch_kmeans_build(c->v, layer, c->ks, keys, values, n, nc, iters, c->use_tc, c->stream, c->prof);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_index");
  c->built[layer] = 1;
  c->steps[layer] = 0;
  c->n_tokens[layer] = n;
  c->n_clusters[layer] = nc;
  return LKV_OK;
}

lkv_status lkv_build_index_async(lkv_ctx *c, int32_t layer, const void *keys, const void *values,
                                 int64_t n, int32_t nc, int32_t iters, uint64_t seed, void *ready_event,
                                 void *done_event) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (ready_event) {
    cudaError_t e = cudaStreamWaitEvent(c->stream, (cudaEvent_t)ready_event, 0);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_index_async: waiting for ready_event");
  }
  s = lkv_build_index(c, layer, keys, values, n, nc, iters, seed);
  if (s != LKV_OK) return s;
  if (done_event) {
    cudaError_t e = cudaEventRecord((cudaEvent_t)done_event, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_index_async: recording done_event");
  }
  return LKV_OK;
}

lkv_status lkv_load_index(lkv_ctx *c, int32_t layer, const void *keys, const void *values,
                          int64_t n, int32_t nc, const int32_t *assign, const float *cent) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (c->v.paris) return fail(c, LKV_EINVAL, "the context uses the ParisKV-style selector");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(c, LKV_EINVAL, "layer out of range");
  if (!keys || !values || !assign || !cent) return fail(c, LKV_EINVAL, "null argument");
  if (n < 1 || n > c->cfg.max_prefill) return fail(c, LKV_EINVAL, "n_tokens outside 1..max_prefill");
  if (nc < 1 || nc > c->cfg.max_clusters) return fail(c, LKV_EINVAL, "n_clusters outside 1..max_clusters");
  cudaError_t e = lkv::launch_load_index(c->v, layer, c->ks, keys, values, n, nc, assign, cent, c->stream, c->prof);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_load_index");
  c->built[layer] = 1;
  c->steps[layer] = 0;
  c->n_tokens[layer] = n;
  c->n_clusters[layer] = nc;
  return LKV_OK;
}

static lkv_status check_step_args(lkv_ctx *c, int32_t layer, int32_t nl, int32_t n_steps,
                                  const void *q, const void *k_new, const void *v_new, float tau,
                                  int32_t budget, int32_t local_buf, const float *out) {
  if (nl < 1 || layer < 0 || layer + nl > c->cfg.n_layers) return fail(c, LKV_EINVAL, "layer range out of bounds");
  if (!q || !k_new || !v_new || !out) return fail(c, LKV_EINVAL, "null input or output");
  if (n_steps < 0) return fail(c, LKV_EINVAL, "n_steps must be >= 0");
  if (budget < 0 || budget > c->cfg.max_budget) return fail(c, LKV_EINVAL, "budget outside 0..max_budget");
  if (local_buf != c->cfg.local_buf) return fail(c, LKV_EINVAL, "local_buf differs from the context's");
  if (tau != tau) return fail(c, LKV_EINVAL, "tau is NaN");
  for (int l = layer; l < layer + nl; ++l) {
    if (!c->built[l]) return fail(c, LKV_ESTATE, "layer " + std::to_string(l) + " has no index");
    if (c->steps[l] != c->steps[layer])
      return fail(c, LKV_EINVAL, "layers decoded in one call must have taken the same number of steps");
    if ((int64_t)c->steps[l] + n_steps > c->cfg.max_steps) return fail(c, LKV_ECAPACITY, "max_steps reached");
  }
  return LKV_OK;
}

static lkv::StepArgs step_args(lkv_ctx *c, int32_t layer, int32_t nl, bool multi, const void *q,
                               const void *k_new, const void *v_new, float tau, int32_t budget,
                               float *out, int32_t *sel, int32_t *nsel, uint8_t *bnd, float *r) {
  lkv::StepArgs a{};
  a.q = q; a.k_new = k_new; a.v_new = v_new;
  a.tau = tau; a.budget = budget;
  a.out = out; a.selected_units = sel; a.n_selected = nsel;
  a.boundary = bnd; a.r_out = r;
  a.l0 = layer; a.nl = nl;
  a.base_t = 0;
  if (multi) {
    const int64_t B = c->cfg.batch, Hkv = c->cfg.n_kv_heads, H = Hkv * c->cfg.group;
    const int64_t Hs = c->v.pol_per_head ? H : Hkv;  // selection records per query or KV head
    const size_t es = c->cfg.dtype == LKV_DTYPE_BF16 ? 2 : 4;
    a.stride_q = B * nl * H * 128;
    a.stride_kv = B * nl * Hkv * 128;
    a.stride_out = B * nl * H * 128;
    a.stride_sel = B * nl * Hs * (int64_t)c->v.u_cap;
    a.stride_nsel = B * nl * Hs;
    a.stride_b = B * nl;
    // kernels address step t (the absolute decode position) at base + t *
    // stride; shifting every base back by the call's first position makes
    // the arguments, and so a cached graph, identical for every call that
    // walks the same full-length buffers chunk by chunk
    const uint64_t t0 = (uint64_t)c->steps[layer];
    auto shift = [t0](const void *p, int64_t stride, size_t eb) -> uintptr_t {
      return p ? (uintptr_t)p - (uintptr_t)(t0 * (uint64_t)stride * eb) : 0;
    };
    a.q = (const void *)shift(q, a.stride_q, es);
    a.k_new = (const void *)shift(k_new, a.stride_kv, es);
    a.v_new = (const void *)shift(v_new, a.stride_kv, es);
    a.out = (float *)shift(out, a.stride_out, 4);
    a.selected_units = (int32_t *)shift(sel, a.stride_sel, 4);
    a.n_selected = (int32_t *)shift(nsel, a.stride_nsel, 4);
    a.boundary = (uint8_t *)shift(bnd, a.stride_b, 1);
    a.r_out = (float *)shift(r, a.stride_b, 4);
  }
  return a;
}

lkv_status lkv_decode_step(lkv_ctx *c, int32_t layer, int32_t nl, const void *q,
                           const void *k_new, const void *v_new, float tau, int32_t budget,
                           int32_t local_buf, float *out, int32_t *selected_units,
                           int32_t *n_selected, uint8_t *boundary, float *r_out) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  s = check_step_args(c, layer, nl, 1, q, k_new, v_new, tau, budget, local_buf, out);
  if (s != LKV_OK) return s;
  lkv::StepArgs a = step_args(c, layer, nl, false, q, k_new, v_new, tau, budget, out,
                              selected_units, n_selected, boundary, r_out);
  cudaError_t e = lkv::launch_decode_steps(c->v, a, 1, c->stream, c->prof);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_decode_step");
  for (int l = layer; l < layer + nl; ++l) c->steps[l] += 1;
  return LKV_OK;
}

// Graph of `steps` consecutive decode steps with these arguments (cached).
static cudaError_t step_graph(lkv_ctx *c, const lkv::StepArgs &a, int steps, cudaGraphExec_t *out) {
  for (GraphEntry &g : c->graphs)
    if (g.steps == steps && std::memcmp(&g.args, &a, sizeof a) == 0) {
      *out = g.exec;
      return cudaSuccess;
    }
  lkv::Prof quiet;
  quiet.counting = false;
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamBeginCapture(c->capture, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return e;
  // step i's attention overlaps step i + 1's boundary test and selection
  // (step and plan slots keep their inputs apart)
  lkv::Pipe pipe = c->pipe;
  for (int i = 0; i < steps && e == cudaSuccess; i += lkv::kChunk) {
    lkv::StepArgs ai = a;
    ai.slot = i;
    pipe.step = i;
    e = lkv::launch_decode_steps(c->v, ai, std::min(lkv::kChunk, steps - i), c->capture, quiet, &pipe);
  }
  // join every lane back into the capture stream
  for (int i = 0; i < lkv::kAttnStreams && i < steps && e == cudaSuccess; ++i)
    e = cudaStreamWaitEvent(c->capture, c->pipe.attn_done[(steps - 1 - i) % lkv::kAttnStreams], 0);
  if (e == cudaSuccess && steps > 0) e = cudaEventRecord(c->pipe.sel_done, c->pipe.sel);
  if (e == cudaSuccess && steps > 0) e = cudaStreamWaitEvent(c->capture, c->pipe.sel_done, 0);
  if (e == cudaSuccess && steps > 0 && c->v.chunk_sel)  // the join lane's last record
    e = cudaStreamWaitEvent(c->capture, c->pipe.chunk_done[((steps - 1) / lkv::kChunk) % 3], 0);
  cudaError_t e2 = cudaStreamEndCapture(c->capture, &graph);
  if (e == cudaSuccess) e = e2;
  cudaGraphExec_t exec = nullptr;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
  if (graph) cudaGraphDestroy(graph);
  if (e != cudaSuccess) return e;
  if (c->graphs.size() >= 8) {
    cudaGraphExecDestroy(c->graphs.front().exec);
    c->graphs.erase(c->graphs.begin());
  }
  GraphEntry g;
  g.args = a;
  g.steps = steps;
  g.exec = exec;
  c->graphs.push_back(g);
  *out = exec;
  return cudaSuccess;
}

lkv_status lkv_decode_steps(lkv_ctx *c, int32_t layer, int32_t nl, int32_t n_steps,
                            const void *q, const void *k_new, const void *v_new, float tau,
                            int32_t budget, int32_t local_buf, float *out,
                            int32_t *selected_units, int32_t *n_selected, uint8_t *boundary,
                            float *r_out) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  s = check_step_args(c, layer, nl, n_steps, q, k_new, v_new, tau, budget, local_buf, out);
  if (s != LKV_OK) return s;
  if (n_steps == 0) return LKV_OK;
  lkv::StepArgs a = step_args(c, layer, nl, true, q, k_new, v_new, tau, budget, out,
                              selected_units, n_selected, boundary, r_out);
  cudaError_t e = cudaSuccess;
  if (c->prof.timing && c->v.chunk_sel) {
    // profiled: the graph's kernels (a boundary and a selection launch per
    // chunk of steps, then the steps' attentions) one after another on the
    // context stream, each bracketed by events
    for (int i = 0; i < n_steps && e == cudaSuccess; i += lkv::kChunk) {
      lkv::StepArgs ai = a;
      ai.slot = 0;
      e = lkv::launch_decode_steps(c->v, ai, std::min(lkv::kChunk, n_steps - i), c->stream, c->prof);
    }
  } else if (c->prof.timing) {
    for (int i = 0; i < n_steps && e == cudaSuccess; ++i) e = lkv::launch_decode_steps(c->v, a, 1, c->stream, c->prof);
  } else {
    // captured graphs of 2048 steps (32 boundary chunks, as far as the step
    // slots reach), then of 512, 128 and 64 for what is left, then single
    // steps
    int done = 0;
    for (const int gl : {lkv::kMaxSlots, 8 * lkv::kChunk, 2 * lkv::kChunk, lkv::kChunk}) {
      if (gl > c->v.n_slots) continue;
      const int reps = (n_steps - done) / gl;
      if (reps == 0 || e != cudaSuccess) continue;
      cudaGraphExec_t exec = nullptr;
      e = step_graph(c, a, gl, &exec);
      for (int r = 0; r < reps && e == cudaSuccess; ++r) e = cudaGraphLaunch(exec, c->stream);
      if (e == cudaSuccess && c->prof.counting) {
        // per graph: a boundary launch per chunk; selection (per chunk or per
        // step), attention and the offload gather per step
        c->prof.launches[lkv::kPBoundary] += (int64_t)reps * (gl / lkv::kChunk);
        c->prof.launches[lkv::kPSelect] += (int64_t)reps * (c->v.chunk_sel ? gl / lkv::kChunk : gl);
        c->prof.launches[lkv::kPAttn] += (int64_t)reps * gl;
        if (c->v.offload) c->prof.launches[lkv::kPGather] += (int64_t)reps * gl;
      }
      done += reps * gl;
    }
    for (int i = done; i < n_steps && e == cudaSuccess; ++i) e = lkv::launch_decode_steps(c->v, a, 1, c->stream, c->prof);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_decode_steps");
  for (int l = layer; l < layer + nl; ++l) c->steps[l] += n_steps;
  return LKV_OK;
}

lkv_status lkv_set_policy(lkv_ctx *c, const lkv_policy *p) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (!p) return fail(c, LKV_EINVAL, "null policy");
  if (p->trigger < LKV_TRIGGER_ADAPTIVE || p->trigger > LKV_TRIGGER_INTERVAL)
    return fail(c, LKV_EINVAL, "unknown trigger");
  if (p->trigger == LKV_TRIGGER_INTERVAL && p->interval < 1) return fail(c, LKV_EINVAL, "interval must be >= 1");
  if (p->fill != LKV_FILL_PREFIX && p->fill != LKV_FILL_SKIP) return fail(c, LKV_EINVAL, "unknown fill");
  if (p->page < 0) return fail(c, LKV_EINVAL, "page must be >= 0");
  if (p->per_head != 0 && p->per_head != 1) return fail(c, LKV_EINVAL, "per_head must be 0 or 1");
  if (p->per_head && c->v.paris) return fail(c, LKV_EINVAL, "per-head selection does not apply to the ParisKV-style selector");
  CtxView &v = c->v;
  if (p->per_head) {
    // the union of the heads' selections is read by the streaming attention
    // from per-token rows in HBM, with the heads' mask in the rows' top byte
    if (v.offload || v.need_pieces || v.S_all > lkv::kStreamMaxSlices)
      return fail(c, LKV_EINVAL, "per-head selection needs an HBM pool, bf16, 4 or 8 query heads per KV head "
                                 "and at most 1024 slices");
    if (v.pool_rows >= (int64_t(1) << lkv::kRowBits))
      return fail(c, LKV_EINVAL, "per-head selection needs max_prefill + max_steps < 2^24");
  }
  // the graphs captured the previous policy in their kernel arguments
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_set_policy");
  if (p->per_head && !v.sel_mask) {
    // first use: the union's rows (up to G budgets), the heads' masks and counts
    lkv_status st = LKV_OK;
    const int64_t R = v.plan_ring;
    const int32_t cap = (int32_t)std::min<int64_t>((int64_t)c->cfg.group * c->cfg.max_budget, v.pool_rows);
    int32_t *rows = (int32_t *)dalloc(c, R * v.S_all * (int64_t)cap * 4, &st);
    uint8_t *mask = (uint8_t *)dalloc(c, R * v.S_all * (int64_t)v.u_cap, &st);
    int32_t *hn = (int32_t *)dalloc(c, R * v.S_all * lkv::kMaxGroup * 4, &st);
    int32_t *ht = (int32_t *)dalloc(c, R * v.S_all * lkv::kMaxGroup * 4, &st);
    if (st != LKV_OK) return st;
    e = cudaMemsetAsync(hn, 0, R * v.S_all * lkv::kMaxGroup * 4, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(ht, 0, R * v.S_all * lkv::kMaxGroup * 4, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_set_policy");
    v.sel_rows = rows;
    v.sel_cap = cap;
    v.sel_mask = mask;
    v.hsel_n = hn;
    v.hsel_tok = ht;
  }
  for (GraphEntry &g : c->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  c->graphs.clear();
  c->v.pol_trigger = p->trigger;
  c->v.pol_interval = p->trigger == LKV_TRIGGER_INTERVAL ? p->interval : 1;
  c->v.pol_fill = p->fill;
  c->v.pol_page = p->page;
  c->v.pol_per_head = p->per_head;
  return LKV_OK;
}

lkv_status lkv_build_pages(lkv_ctx *c, int32_t layer, const void *keys, const void *values, int64_t n,
                           int32_t page) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (c->v.paris) return fail(c, LKV_EINVAL, "the context uses the ParisKV-style selector");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(c, LKV_EINVAL, "layer out of range");
  if (!keys || !values) return fail(c, LKV_EINVAL, "null keys or values");
  if (n < 1 || n > c->cfg.max_prefill) return fail(c, LKV_EINVAL, "n_tokens outside 1..max_prefill");
  if (page < 1) return fail(c, LKV_EINVAL, "page must be >= 1");
  const int64_t nc = (n + page - 1) / page;
  if (nc > c->cfg.max_clusters) return fail(c, LKV_EINVAL, "ceil(n_tokens / page) exceeds max_clusters");
  cudaError_t e = lkv::launch_page_index(c->v, layer, c->ks, keys, values, n, page, c->stream, c->prof);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_pages");
  c->built[layer] = 1;
  c->steps[layer] = 0;
  c->n_tokens[layer] = n;
  c->n_clusters[layer] = (int32_t)nc;
  return LKV_OK;
}

lkv_status lkv_paris_levels(float *thr, float *lev) {
  if (!thr || !lev) {
    lkv::set_unbound_error("lkv_paris_levels: null pointer");
    return LKV_EINVAL;
  }
  lkv::paris_levels_host(thr, lev);
  return LKV_OK;
}

lkv_status lkv_build_paris(lkv_ctx *c, int32_t layer, const void *keys, const void *values, int64_t n,
                           const lkv_paris_params *p) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  CtxView &v = c->v;
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(c, LKV_EINVAL, "layer out of range");
  if (!keys || !values || !p) return fail(c, LKV_EINVAL, "null argument");
  if (n < 1 || n > c->cfg.max_prefill) return fail(c, LKV_EINVAL, "n_tokens outside 1..max_prefill");
  if (p->rho < 1 || p->rho > lkv::kParisMaxRho) return fail(c, LKV_EINVAL, "rho must be 1..15");
  if (p->n_cand < 1 || p->n_cand > lkv::kParisMaxCand) return fail(c, LKV_EINVAL, "n_cand must be 1..4096");
  if (v.dtype != LKV_DTYPE_BF16 || v.offload || v.need_pieces || v.S_all > lkv::kStreamMaxSlices)
    return fail(c, LKV_EINVAL, "the ParisKV-style selector needs bf16, an HBM pool, group 4 or 8 and at most "
                               "1024 slices");
  if ((int64_t)v.u_cap < c->cfg.max_budget)
    return fail(c, LKV_EINVAL, "max_clusters + max_steps must be >= max_budget (selected tokens are listed)");
  if (v.pol_per_head) return fail(c, LKV_EINVAL, "per-head selection does not apply to the ParisKV-style selector");
  for (int l = 0; l < c->cfg.n_layers; ++l)
    if (c->built[l] == 1) return fail(c, LKV_EINVAL, "a layer of the context was built with clusters or pages");
  if (v.paris && (v.paris_rho != p->rho || v.paris_n_cand != p->n_cand || c->paris_seed != p->seed))
    return fail(c, LKV_EINVAL, "rho, n_cand and seed are fixed by the context's first lkv_build_paris");
  if (!v.paris) {
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_paris");
    lkv_status st = LKV_OK;
    const int64_t rows = v.S_all * v.pool_rows;
    uint8_t *bk = (uint8_t *)dalloc(c, rows * lkv::kParisSub, &st);
    uint8_t *code = (uint8_t *)dalloc(c, rows * 64, &st);
    float *w = (float *)dalloc(c, rows * lkv::kParisSub * 4, &st);
    const int64_t pitch = (v.pool_rows + 15) / 16 * 16;
    uint8_t *score = (uint8_t *)dalloc(c, (int64_t)lkv::kChunk * v.S_all * pitch, &st);
    if (st != LKV_OK) return st;
    for (GraphEntry &g : c->graphs)
      if (g.exec) cudaGraphExecDestroy(g.exec);
    c->graphs.clear();
    uint64_t sm = p->seed;
    v.paris_sign[0] = splitmix64_next(sm);
    v.paris_sign[1] = splitmix64_next(sm);
    lkv::paris_levels_host(v.paris_thr, v.paris_lev);
    v.paris_rho = p->rho;
    v.paris_n_cand = p->n_cand;
    v.pk_bucket = bk;
    v.pk_code = code;
    v.pk_w = w;
    v.pk_score = score;
    v.pk_pitch = pitch;
    v.paris = 1;
    c->paris_seed = p->seed;
  }
  cudaError_t e = lkv::launch_paris_index(v, layer, c->ks, keys, values, n, c->stream, c->prof);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_build_paris");
  c->built[layer] = 2;
  c->steps[layer] = 0;
  c->n_tokens[layer] = n;
  c->n_clusters[layer] = 0;
  return LKV_OK;
}

static const char *kKindNames[lkv::kPNum] = {
    "lkv_boundary", "lkv_score", "lkv_gather_offload", "lkv_attn",
    "kmeans_init", "kmeans_operand", "kmeans_assign", "kmeans_refine", "kmeans_sort",
    "kmeans_update", "kmeans_pool", "kmeans_assign_tc", "lkv_select"};

lkv_status lkv_set_kmeans_filter(lkv_ctx *ctx, int32_t filter) {
  if (!ctx) return fail(nullptr, LKV_EINVAL, "null context");
  if (filter != LKV_FILTER_TENSOR && filter != LKV_FILTER_SIMT)
    return fail(ctx, LKV_EINVAL, "unknown K-means filter");
  ctx->use_tc = filter == LKV_FILTER_TENSOR;
  return LKV_OK;
}

lkv_status lkv_set_profiling(lkv_ctx *c, int32_t enable) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  c->prof.timing = enable != 0;
  return LKV_OK;
}

lkv_status lkv_get_profile(lkv_ctx *c, lkv_kernel_stat *stats, int32_t capacity, int32_t *n_stats,
                           int64_t *counters, int32_t reset) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  s = lkv_sync(c);
  if (s != LKV_OK) return s;
  c->prof.resolve();
  if (n_stats) *n_stats = lkv::kPNum;
  for (int k = 0; k < lkv::kPNum && stats && k < capacity; ++k) {
    std::memset(stats[k].name, 0, sizeof stats[k].name);
    std::strncpy(stats[k].name, kKindNames[k], sizeof stats[k].name - 1);
    stats[k].launches = c->prof.launches[k];
    stats[k].total_ms = c->prof.ms[k];
  }
  if (counters) {
    int64_t h[lkv::kCounters] = {};
    cudaError_t e = cudaMemcpy(h, c->v.counters, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_get_profile");
    counters[0] = h[lkv::kCntAttnRows];
    counters[1] = h[lkv::kCntAttnSlices];
    counters[2] = h[lkv::kCntScoreUnits];
    counters[3] = h[lkv::kCntGatherRows];
    counters[4] = h[lkv::kCntSelUnits];
    counters[5] = h[lkv::kCntSelTokens];
  }
  if (reset) {
    for (int k = 0; k < lkv::kPNum; ++k) {
      c->prof.launches[k] = 0;
      c->prof.ms[k] = 0.0;
    }
    cudaError_t e = cudaMemset(c->v.counters, 0, lkv::kCounters * 8);
    if (e != cudaSuccess) return cuda_fail(c, e, "lkv_get_profile");
  }
  return LKV_OK;
}

lkv_status lkv_uva_read(const void *host_src, void *dev_dst, int64_t bytes, void *stream) {
  if (!host_src || !dev_dst || bytes < 0 || bytes % 16 != 0 ||
      ((uintptr_t)host_src | (uintptr_t)dev_dst) % 16 != 0) {
    lkv::set_unbound_error("lkv_uva_read: null pointer, or size/address not a multiple of 16");
    return LKV_EINVAL;
  }
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host_src);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    lkv::set_unbound_error("lkv_uva_read: host_src is not pinned host memory");
    return LKV_EINVAL;
  }
  e = lkv::launch_uva_read(attr.devicePointer ? attr.devicePointer : host_src, dev_dst, bytes,
                           (cudaStream_t)stream);
  if (e != cudaSuccess) {
    lkv::set_unbound_error((std::string("lkv_uva_read: ") + cudaGetErrorString(e)).c_str());
    return LKV_ECUDA;
  }
  return LKV_OK;
}

lkv_status lkv_read_ceiling(const void *dev_src, int64_t bytes, void *stream) {
  if (!dev_src || bytes < 0 || bytes % 16 != 0 || (uintptr_t)dev_src % 16 != 0) {
    lkv::set_unbound_error("lkv_read_ceiling: null pointer, or size/address not a multiple of 16");
    return LKV_EINVAL;
  }
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, dev_src);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    lkv::set_unbound_error("lkv_read_ceiling: dev_src is not device memory");
    return LKV_EINVAL;
  }
  e = lkv::launch_read_ceiling(dev_src, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    lkv::set_unbound_error((std::string("lkv_read_ceiling: ") + cudaGetErrorString(e)).c_str());
    return LKV_ECUDA;
  }
  return LKV_OK;
}

lkv_status lkv_diag_wait_timeout(lkv_ctx *c, int64_t limit_ns) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (limit_ns < 0 || limit_ns > 1000000000) return fail(c, LKV_EINVAL, "limit_ns must be 0..1e9");
  cudaError_t e = lkv::launch_diag_wait(c->v, (uint64_t)limit_ns, c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_diag_wait_timeout");
  return LKV_OK;
}

lkv_status lkv_sync(lkv_ctx *c) {
  if (!c) return LKV_EINVAL;
  if (c->broken) return fail(c, LKV_ESTATE, "context is unusable after a CUDA error");
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_sync");
  int32_t bits = 0;
  e = cudaMemcpy(&bits, c->v.err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_sync");
  if (bits) {
    cudaMemset(c->v.err, 0, 4);
    if (bits & lkv::kErrTimeout) return fail(c, LKV_ETIMEOUT, "a device-side wait gave up");
    if (bits & lkv::kErrCapacity) return fail(c, LKV_ECAPACITY, "device-side capacity exceeded");
    return fail(c, LKV_ECUDA, "device-side invariant check failed");
  }
  return LKV_OK;
}

lkv_status lkv_get_index(lkv_ctx *c, int32_t layer, int32_t seq, int32_t kv_head,
                         int32_t capacity, float *centroids, int32_t *unit_len,
                         int32_t *unit_row, int32_t *assign, int32_t *perm, int32_t *n_units) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (layer < 0 || layer >= c->cfg.n_layers || seq < 0 || seq >= c->cfg.batch || kv_head < 0 ||
      kv_head >= c->cfg.n_kv_heads || !n_units)
    return fail(c, LKV_EINVAL, "index coordinates out of range");
  if (!c->built[layer]) return fail(c, LKV_ESTATE, "layer has no index");
  s = lkv_sync(c);
  if (s != LKV_OK) return s;
  const int64_t lb = (int64_t)layer * c->cfg.batch + seq;
  const int64_t gs = lb * c->cfg.n_kv_heads + kv_head;
  DecState st{};
  cudaError_t e = cudaMemcpy(&st, c->v.st + lb, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_get_index");
  *n_units = st.n_units;
  if (st.n_units > capacity) return fail(c, LKV_ECAPACITY, "capacity below n_units");
  const int64_t u_cap = c->v.u_cap, n = c->n_tokens[layer];
  if (centroids && e == cudaSuccess)
    e = cudaMemcpy(centroids, c->v.cent32 + gs * u_cap * 128, (size_t)st.n_units * 128 * 4, cudaMemcpyDeviceToHost);
  if (unit_len && e == cudaSuccess)
    e = cudaMemcpy(unit_len, c->v.unit_len + gs * u_cap, (size_t)st.n_units * 4, cudaMemcpyDeviceToHost);
  if (unit_row && e == cudaSuccess)
    e = cudaMemcpy(unit_row, c->v.unit_row + gs * u_cap, (size_t)st.n_units * 4, cudaMemcpyDeviceToHost);
  if (assign && e == cudaSuccess)
    e = cudaMemcpy(assign, c->v.assign + gs * c->v.n_cap, (size_t)n * 4, cudaMemcpyDeviceToHost);
  if (perm && e == cudaSuccess)
    e = cudaMemcpy(perm, c->v.perm + gs * c->v.n_cap, (size_t)n * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_get_index");
  return LKV_OK;
}

lkv_status lkv_get_decode_state(lkv_ctx *c, int32_t layer, int32_t seq, lkv_decode_state *out) {
  lkv_status s = check_usable(c);
  if (s != LKV_OK) return s;
  if (!out || layer < 0 || layer >= c->cfg.n_layers || seq < 0 || seq >= c->cfg.batch)
    return fail(c, LKV_EINVAL, "state coordinates out of range");
  s = lkv_sync(c);
  if (s != LKV_OK) return s;
  DecState st{};
  int64_t refined = 0, inexact = 0;
  cudaError_t e = cudaMemcpy(&st, c->v.st + (int64_t)layer * c->cfg.batch + seq, sizeof st, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&refined, c->ks.n_refined, 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&inexact, c->ks.n_inexact, 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "lkv_get_decode_state");
  out->t = st.t;
  out->win_start = st.win_start;
  out->open_start = st.open_start;
  out->n_clusters = st.n_clusters;
  out->n_units = st.n_units;
  out->n_closed = st.n_closed;
  out->n_evicted = st.n_evicted;
  out->n_forced = st.n_forced;
  out->n_refined = refined;
  out->n_inexact = inexact;
  return LKV_OK;
}

const char *lkv_last_error(const lkv_ctx *c) {
  if (!c) return g_create_error.c_str();
  return c->err.c_str();
}

}  // extern "C"
