// decode.cu -- one decode step of LouisKV-style retrieval for a range of
// layers and all sequences [LouisKV notes, 方法详解 flowchart; 关键设计 1-3]:
//
//   k_step_boundary  r_t, trigger flag, segment close, local-buffer eviction,
//                    append of token t                      (1 CTA / (seq, layer))
//   k_score          s_u = qbar . c_u for every unit         (trigger steps only)
//   k_select         (score desc, id asc) budget prefix, plus the copy plan of
//                    the selected rows in 64-token chunks    (trigger steps only)
//   k_gather_offload selected rows host -> HBM staging (UVA; offload only)
//   k_attn           split-K softmax attention: each CTA stages one 64-token
//                    chunk of (selected rows ++ local buffer) with bulk copies,
//                    the last CTA of each (seq, layer, kv head) combines
//
// Inputs/outputs of step k of a call live at base + k * stride (StepArgs).
#include "lkv_internal.cuh"

namespace lkv {

constexpr int kMaxHeads = 128;
constexpr unsigned kFull = 0xffffffffu;

// 16-byte vector of elements starting at element offset i (16-byte aligned).
template <int DT>
__device__ __forceinline__ void load16(const void *base, int64_t i, float *out) {
  const uint4 raw = __ldg((const uint4 *)((const char *)base + i * elem_bytes<DT>()));
  if constexpr (DT == 1) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      out[2 * e] = __uint_as_float(w[e] << 16);
      out[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    out[0] = __uint_as_float(raw.x); out[1] = __uint_as_float(raw.y);
    out[2] = __uint_as_float(raw.z); out[3] = __uint_as_float(raw.w);
  }
}

// ---------------------------------------------------------------- mbarrier / bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}
// Wait for the phase to complete, giving up after limit_ns of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase, uint64_t limit_ns) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, phase))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// ---------------------------------------------------------------- boundary + segments

// Close segment [s0, s1) as unit C + n_closed: its index vector is the mean of
// its keys per kv head. Called by every thread of the block; returns false
// (uniformly) when the unit table is full.
template <int DT>
__device__ bool close_segment(const CtxView &v, DecState &st, int64_t lb, int s0, int s1) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int u = st.n_clusters + st.n_closed;
  if (u >= v.u_cap) {
    if (tid == 0) set_err(v.err, kErrCapacity);
    return false;
  }
  const int len = s1 - s0;
  const bool slow = st.seg_slow != 0;
  for (int k = tid; k < v.Hkv * kHeadDim; k += nth) {
    const int h = k / kHeadDim, dim = k % kHeadDim;
    const int64_t gs = lb * v.Hkv + h;
    double S;
    if constexpr (DT == 1) {
      if (!slow) {
        S = fixed40_to_double(v.segsum[gs * kHeadDim + dim]);
      } else {
        S = 0.0;
        for (int tt = s0; tt < s1; ++tt)
          S = __dadd_rn(S, (double)load_elem<DT>(v.dec_k, (gs * v.dec_rows + tt) * kHeadDim + dim));
      }
    } else {
      S = __longlong_as_double(v.segsum[gs * kHeadDim + dim]);
    }
    const float mean = __double2float_rn(__ddiv_rn(S, (double)len));
    const int64_t ci = (gs * v.u_cap + u) * kHeadDim + dim;
    v.cent32[ci] = mean;
    store_elem<DT>(v.cent_op, ci, mean);
    v.segsum[gs * kHeadDim + dim] = 0;
  }
  for (int h = tid; h < v.Hkv; h += nth) {
    const int64_t gs = lb * v.Hkv + h;
    v.unit_row[gs * v.u_cap + u] = (int32_t)(v.n_cap + s0);
    v.unit_len[gs * v.u_cap + u] = len;
  }
  __syncthreads();
  if (tid == 0) {
    st.n_closed += 1;
    st.seg_slow = 0;
  }
  __syncthreads();
  return true;
}

template <int DT>
__global__ void __launch_bounds__(1024) k_step_boundary(CtxView v, StepArgs a) {
  const int li = blockIdx.x / v.B, b = blockIdx.x % v.B;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int H = v.Hkv * v.G;
  const int tid = threadIdx.x, nth = blockDim.x;
  __shared__ DecState st;
  __shared__ float cosv[kMaxHeads];
  __shared__ int slow_any;
  if (tid == 0) {
    st = v.st[lb];
    slow_any = 0;
  }
  __syncthreads();
  const int t = st.t;
  const int64_t k = t - a.base_t;
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  const void *k_new = (const char *)a.k_new + k * a.stride_kv * elem_bytes<DT>();
  const void *v_new = (const char *)a.v_new + k * a.stride_kv * elem_bytes<DT>();
  const int64_t qoff = ((int64_t)b * a.nl + li) * H * kHeadDim;
  const int64_t kvoff = ((int64_t)b * a.nl + li) * v.Hkv * kHeadDim;

  // 1. r_t = (1/H) sum_h cos(q_{t-1}^h, q_t^h) in fp32, fixed operation order
  if (t > 0) {
    if (tid < H) {
      float dot = 0.f, na = 0.f, nb = 0.f;
      constexpr int per16 = 16 / elem_bytes<DT>();
#pragma unroll 2
      for (int j0 = 0; j0 < kHeadDim; j0 += per16) {
        float x[8], y[8];
        load16<DT>(v.q_prev, (lb * H + tid) * kHeadDim + j0, x);
        load16<DT>(q, qoff + (int64_t)tid * kHeadDim + j0, y);
#pragma unroll
        for (int e = 0; e < per16; ++e) {
          dot = __fmaf_rn(x[e], y[e], dot);
          na = __fmaf_rn(x[e], x[e], na);
          nb = __fmaf_rn(y[e], y[e], nb);
        }
      }
      const float den = __fmul_rn(__fsqrt_rn(na), __fsqrt_rn(nb));
      cosv[tid] = den > 0.f ? __fdiv_rn(dot, den) : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
      float r = 0.f;
      for (int h = 0; h < H; ++h) r = __fadd_rn(r, cosv[h]);
      r = __fdiv_rn(r, (float)H);
      st.r = r;
      st.flag = r < a.tau ? 1 : 0;
    }
  } else if (tid == 0) {
    st.r = 0.f;
    st.flag = 1;
  }
  __syncthreads();

  // 2. a boundary closes the open segment; token t opens the next one
  if (st.flag && t > 0 && st.open_start < t) {
    const int s0 = st.open_start;
    if (close_segment<DT>(v, st, lb, s0, t) && tid == 0) st.open_start = t;
    __syncthreads();
  }

  // 3. make room for token t: evict the oldest closed segment; with none
  //    left, cut the open segment and evict it
  for (int guard = 0; guard <= v.L + 1; ++guard) {
    __syncthreads();
    const bool need = (t - st.win_start) + 1 > v.L;
    const bool none_closed = st.n_evicted >= st.n_closed;
    __syncthreads();
    if (!need) break;
    if (none_closed) {
      const int s0 = st.open_start;
      if (s0 >= t || !close_segment<DT>(v, st, lb, s0, t)) {
        if (tid == 0) set_err(v.err, kErrInternal);
        break;
      }
      if (tid == 0) {
        st.open_start = t;
        st.n_forced += 1;
      }
      __syncthreads();
    }
    const int u = st.n_clusters + st.n_evicted;
    const int64_t gs0 = lb * v.Hkv;
    const int seg0 = v.unit_row[gs0 * v.u_cap + u] - (int32_t)v.n_cap;
    const int seg_len = v.unit_len[gs0 * v.u_cap + u];
    if (v.offload) {
      // the evicted rows move to the host pool (same relative rows)
      constexpr int per_row = kHeadDim * elem_bytes<DT>() / 16;
      const int64_t total = (int64_t)v.Hkv * seg_len * per_row;
      for (int64_t x = tid; x < total; x += nth) {
        const int h = (int)(x / ((int64_t)seg_len * per_row));
        const int rem = (int)(x % ((int64_t)seg_len * per_row));
        const int r = rem / per_row, c16 = rem % per_row;
        const int64_t gs = gs0 + h;
        const int64_t src = (gs * v.dec_rows + seg0 + r) * kHeadDim * elem_bytes<DT>() + c16 * 16;
        const int64_t dst = (gs * v.pool_rows + v.n_cap + seg0 + r) * kHeadDim * elem_bytes<DT>() + c16 * 16;
        *(uint4 *)((char *)v.pool_k + dst) = *(const uint4 *)((const char *)v.dec_k + src);
        *(uint4 *)((char *)v.pool_v + dst) = *(const uint4 *)((const char *)v.dec_v + src);
      }
    }
    __syncthreads();
    if (tid == 0) {
      st.win_start = seg0 + seg_len;
      st.n_evicted += 1;
      st.n_units = st.n_clusters + st.n_evicted;
    }
  }
  __syncthreads();

  // 4. token t enters the local buffer; its key joins the open segment's sum
  int slow = 0;
  for (int x = tid; x < v.Hkv * kHeadDim; x += nth) {
    const int h = x / kHeadDim, dim = x % kHeadDim;
    const int64_t gs = lb * v.Hkv + h;
    const int64_t di = (gs * v.dec_rows + t) * kHeadDim + dim;
    if constexpr (DT == 1) {
      const uint16_t kb = ((const uint16_t *)k_new)[kvoff + x];
      ((uint16_t *)v.dec_k)[di] = kb;
      ((uint16_t *)v.dec_v)[di] = ((const uint16_t *)v_new)[kvoff + x];
      v.segsum[gs * kHeadDim + dim] += bf16_fixed40(kb, &slow);
    } else {
      const float kf = ((const float *)k_new)[kvoff + x];
      ((float *)v.dec_k)[di] = kf;
      ((float *)v.dec_v)[di] = ((const float *)v_new)[kvoff + x];
      const double s = __longlong_as_double(v.segsum[gs * kHeadDim + dim]);
      v.segsum[gs * kHeadDim + dim] = __double_as_longlong(__dadd_rn(s, (double)kf));
    }
  }
  if (slow) atomicOr(&slow_any, 1);
  for (int x = tid; x < H * kHeadDim; x += nth) {
    if constexpr (DT == 1)
      ((uint16_t *)v.q_prev)[lb * H * kHeadDim + x] = ((const uint16_t *)q)[qoff + x];
    else
      ((float *)v.q_prev)[lb * H * kHeadDim + x] = ((const float *)q)[qoff + x];
  }
  __syncthreads();
  if (tid == 0) {
    if (slow_any) st.seg_slow = 1;
    st.t = t + 1;
    v.st[lb] = st;
    const int64_t o = (int64_t)b * a.nl + li;
    if (a.boundary) a.boundary[k * a.stride_b + o] = (uint8_t)st.flag;
    if (a.r_out) a.r_out[k * a.stride_b + o] = st.r;
  }
}

// ---------------------------------------------------------------- scoring

template <int DT>
__global__ void __launch_bounds__(256) k_score(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const DecState *stp = v.st + lb;
  if (!stp->flag) return;
  const int U = stp->n_units;
  const int64_t k = (stp->t - 1) - a.base_t;
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  __shared__ float qbar[kHeadDim];
  const int H = v.Hkv * v.G;
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * v.G) * kHeadDim;
  if (threadIdx.x < kHeadDim) {
    float acc = load_elem<DT>(q, qoff + threadIdx.x);
    for (int g = 1; g < v.G; ++g) acc = __fadd_rn(acc, load_elem<DT>(q, qoff + (int64_t)g * kHeadDim + threadIdx.x));
    qbar[threadIdx.x] = acc;
  }
  __syncthreads();
  constexpr int per16 = 16 / elem_bytes<DT>();
  for (int u = blockIdx.y * blockDim.x + threadIdx.x; u < U; u += gridDim.y * blockDim.x) {
    const int64_t base = (gs * v.u_cap + u) * kHeadDim;
    float s = 0.f;
#pragma unroll 4
    for (int j0 = 0; j0 < kHeadDim; j0 += per16) {
      float c[8];
      load16<DT>(v.cent_op, base + j0, c);
#pragma unroll
      for (int e = 0; e < per16; ++e) s = __fmaf_rn(qbar[j0 + e], c[e], s);
    }
    v.scores[gs * v.u_cap + u] = s;
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)U);
}

// ---------------------------------------------------------------- selection

__device__ __forceinline__ int32_t block_scan_excl(int32_t x, int32_t *wt, int32_t *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) wt[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int32_t w = lane < nw ? wt[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) wt[lane] = w;
    if (lane == nw - 1 && total) *total = w;
  }
  __syncthreads();
  const int32_t r = inc - x + (wid ? wt[wid - 1] : 0);
  __syncthreads();
  return r;
}

// Weighted radix select of the cut: the smallest key value K* (desc_key of a
// score) with sum_{key <= K*} len > budget. Units with key < K* all precede
// the first unit that does not fit; units with key == K* are taken in id
// order while they fit. Output: ascending unit ids, their first rows, the
// exclusive token prefix, and the copy plan: the selected rows cut into
// pieces that never cross a 64-token chunk boundary.
__global__ void __launch_bounds__(1024) k_select(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const DecState *stp = v.st + lb;
  if (!stp->flag) return;
  const int U = stp->n_units;
  const int budget = a.budget;
  const float *sc = v.scores + gs * v.u_cap;
  const int32_t *ln = v.unit_len + gs * v.u_cap;
  const int tid = threadIdx.x, nth = blockDim.x, wid = tid >> 5;
  __shared__ int32_t whist[32][256];
  __shared__ int32_t wt[32];
  __shared__ int32_t s_total, s_below, s_all, s_nsel, s_ntok, s_npieces;
  __shared__ uint32_t s_prefix, s_mask;

  int32_t part = 0;
  for (int u = tid; u < U; u += nth) part += ln[u];
  block_scan_excl(part, wt, &s_total);
  if (tid == 0) {
    s_all = s_total <= budget;
    s_prefix = 0;
    s_mask = 0;
    s_below = 0;
  }
  __syncthreads();
  if (!s_all) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int x = tid; x < 32 * 256; x += nth) (&whist[0][0])[x] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix, mask = s_mask;
      for (int u = tid; u < U; u += nth) {
        const uint32_t key = desc_key(sc[u]);
        if ((key & mask) == prefix) atomicAdd(&whist[wid][(key >> shift) & 255u], ln[u]);
      }
      __syncthreads();
      if (tid < 256) {
        int32_t tot = 0;
        for (int w = 0; w < 32; ++w) tot += whist[w][tid];
        whist[0][tid] = tot;
      }
      __syncthreads();
      if (tid < 32) {
        // warp scan over the 256 bins (8 per lane) for the bin where the
        // running weight first exceeds the budget
        int32_t loc[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) { loc[e] = whist[0][tid * 8 + e]; sum += loc[e]; }
        int32_t inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(kFull, inc, o);
          if (tid >= o) inc += y;
        }
        const int32_t base = s_below + inc - sum;
        int found = -1;
        int32_t run = base;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (found < 0 && run + loc[e] > budget) found = e;
          if (found < 0) run += loc[e];
        }
        const unsigned hit = __ballot_sync(kFull, found >= 0);
        const int src = hit ? __ffs(hit) - 1 : 31;
        const int digit = __shfl_sync(kFull, tid * 8 + (found >= 0 ? found : 7), src);
        const int32_t below = __shfl_sync(kFull, run, src);
        if (tid == 0) {
          s_below = below;
          s_prefix = prefix | ((uint32_t)digit << shift);
          s_mask = mask | (255u << shift);
        }
      }
      __syncthreads();
    }
  }
  const bool all = s_all != 0;
  const uint32_t kstar = s_prefix;
  const int32_t below = s_below;
  const int per = (U + nth - 1) / nth;
  const int u0 = tid * per, u1 = min(U, u0 + per);
  // exclusive id-order prefix of the tied units' lengths
  int32_t tl = 0;
  if (!all)
    for (int u = u0; u < u1; ++u)
      if (desc_key(sc[u]) == kstar) tl += ln[u];
  const int32_t tie_ex = block_scan_excl(tl, wt, nullptr);
  int32_t cnt = 0, toks = 0;
  {
    int32_t run = tie_ex;
    for (int u = u0; u < u1; ++u) {
      bool sel = all;
      if (!all) {
        const uint32_t key = desc_key(sc[u]);
        if (key < kstar) sel = true;
        else if (key == kstar) { run += ln[u]; sel = below + run <= budget; }
      }
      if (sel) { ++cnt; toks += ln[u]; }
    }
  }
  const int32_t cnt_ex = block_scan_excl(cnt, wt, &s_nsel);
  const int32_t tok_ex = block_scan_excl(toks, wt, &s_ntok);
  int32_t npc = 0;  // copy pieces of this thread's selected units
  {
    int32_t run = tie_ex, kk = cnt_ex, cum = tok_ex;
    int32_t *sel_out = v.sel + gs * v.u_cap;
    int32_t *row_out = v.rng_row + gs * v.u_cap;
    int32_t *cum_out = v.rng_cum + gs * (int64_t)(v.u_cap + 1);
    const int32_t *rows = v.unit_row + gs * v.u_cap;
    for (int u = u0; u < u1; ++u) {
      bool sel = all;
      if (!all) {
        const uint32_t key = desc_key(sc[u]);
        if (key < kstar) sel = true;
        else if (key == kstar) { run += ln[u]; sel = below + run <= budget; }
      }
      if (sel) {
        const int32_t len = ln[u];
        sel_out[kk] = u;
        row_out[kk] = rows[u];
        cum_out[kk] = cum;
        if (len > 0) npc += (cum + len - 1) / kAttnChunk - cum / kAttnChunk + 1;
        cum += len;
        ++kk;
      }
    }
  }
  const int32_t pc_ex = block_scan_excl(npc, wt, &s_npieces);
  {
    int32_t run = tie_ex, cum = tok_ex, p = pc_ex;
    int4 *pieces = v.pieces + gs * (int64_t)v.max_pieces;
    int32_t *cp = v.chunk_piece + gs * (int64_t)(v.max_chunks + 1);
    const int32_t *rows = v.unit_row + gs * v.u_cap;
    for (int u = u0; u < u1 && p - pc_ex < npc; ++u) {
      bool sel = all;
      if (!all) {
        const uint32_t key = desc_key(sc[u]);
        if (key < kstar) sel = true;
        else if (key == kstar) { run += ln[u]; sel = below + run <= budget; }
      }
      if (!sel) continue;
      int32_t len = ln[u], src = rows[u], f = cum;
      cum += len;
      while (len > 0) {
        const int32_t room = kAttnChunk - f % kAttnChunk;
        const int32_t n = len < room ? len : room;
        if (p < v.max_pieces) pieces[p] = make_int4(src, f, n, 0);
        if (f % kAttnChunk == 0 && f / kAttnChunk <= v.max_chunks) cp[f / kAttnChunk] = p;
        ++p;
        f += n;
        src += n;
        len -= n;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    v.n_sel[gs] = s_nsel;
    v.n_tok[gs] = s_ntok;
    v.rng_cum[gs * (int64_t)(v.u_cap + 1) + s_nsel] = s_ntok;
    const int nsc = (s_ntok + kAttnChunk - 1) / kAttnChunk;
    if (nsc <= v.max_chunks) v.chunk_piece[gs * (int64_t)(v.max_chunks + 1) + nsc] = s_npieces;
    if (s_ntok > budget || s_npieces > v.max_pieces) set_err(v.err, kErrInternal);
  }
}

// ---------------------------------------------------------------- offload gather

// Largest r with cum[r] <= f (cum ascending, cum[0] = 0, f < cum[n]).
__device__ __forceinline__ int find_range(const int32_t *cum, int n, int32_t f) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cum + mid) <= f) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int DT>
__global__ void __launch_bounds__(256) k_gather_offload(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  if (!v.st[lb].flag) return;
  const int ns = v.n_sel[gs], nt = v.n_tok[gs];
  const int32_t *cum = v.rng_cum + gs * (int64_t)(v.u_cap + 1);
  const int32_t *rows = v.rng_row + gs * v.u_cap;
  constexpr int rb = kHeadDim * elem_bytes<DT>();
  constexpr int per_row = rb / 16;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.y * (blockDim.x / 32);
  for (int f = blockIdx.y * (blockDim.x / 32) + threadIdx.x / 32; f < nt; f += warps) {
    const int r = find_range(cum, ns, f);
    const int64_t row = rows[r] + (f - cum[r]);
    if (lane < per_row) {
      const int64_t src = (gs * v.pool_rows + row) * rb + lane * 16;
      const int64_t dst = (gs * (int64_t)v.bud_cap + f) * rb + lane * 16;
      *(uint4 *)((char *)v.stage_k + dst) = __ldcg((const uint4 *)((const char *)v.pool_k + src));
      *(uint4 *)((char *)v.stage_v + dst) = __ldcg((const uint4 *)((const char *)v.pool_v + src));
    }
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    atomicAdd((unsigned long long *)&v.counters[kCntGatherRows], (unsigned long long)nt);
}

// ---------------------------------------------------------------- attention

constexpr int kAttnWarps = 4;
constexpr int kTokPerWarp = kAttnChunk / kAttnWarps;  // 16
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // 2 s

// Butterfly reduce-scatter of 32 per-lane partials (P == 32) or of 16
// partials replicated over both half-warps (P == 16): on return lane L holds
// the full sum of partial index L % P.
template <int P>
__device__ __forceinline__ float reduce_scatter(float (&x)[32], int lane) {
  if constexpr (P == 32) {
    const bool up = lane & 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float send = up ? x[j] : x[j + 16];
      const float keep = up ? x[j + 16] : x[j];
      x[j] = keep + __shfl_xor_sync(kFull, send, 16);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] += __shfl_xor_sync(kFull, x[j], 16);
  }
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    const bool up = lane & m;
#pragma unroll
    for (int j = 0; j < m; ++j) {
      const float send = up ? x[j] : x[j + m];
      const float keep = up ? x[j + m] : x[j];
      x[j] = keep + __shfl_xor_sync(kFull, send, m);
    }
  }
  return x[0];
}

template <int DT>
__device__ __forceinline__ void row4(const unsigned char *row, int lane, float (&o)[4]) {
  if constexpr (DT == 1) {
    const uint2 r = *(const uint2 *)(row + lane * 8);
    o[0] = __uint_as_float(r.x << 16); o[1] = __uint_as_float(r.x & 0xffff0000u);
    o[2] = __uint_as_float(r.y << 16); o[3] = __uint_as_float(r.y & 0xffff0000u);
  } else {
    const float4 r = *(const float4 *)(row + lane * 16);
    o[0] = r.x; o[1] = r.y; o[2] = r.z; o[3] = r.w;
  }
}

template <int DT, int G>
__global__ void __launch_bounds__(kAttnWarps * 32) k_attn(CtxView v, StepArgs a) {
  constexpr int RB = kHeadDim * elem_bytes<DT>();
  constexpr int TB = (32 / G) < kTokPerWarp ? (32 / G) : kTokPerWarp;  // tokens per batch
  constexpr int P = TB * G;                                           // partials per lane
  constexpr int NB = kTokPerWarp / TB;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *Ks = smem;                      // [64][RB]
  unsigned char *Vs = smem + kAttnChunk * RB;    // [64][RB]
  __shared__ __align__(8) uint64_t bar;
  __shared__ float qs[G][kHeadDim];
  __shared__ float ps[kAttnWarps][32];
  __shared__ float cs[kAttnWarps][G];
  __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
  __shared__ float wacc[kAttnWarps][G][kHeadDim];
  __shared__ int s_last, s_ok;

  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const DecState st = v.st[lb];
  const int t_cur = st.t - 1, ws = st.win_start;
  const int64_t k = t_cur - a.base_t;
  const int nt = v.n_tok[gs];
  const int total = nt + (t_cur - ws + 1);
  const int H = v.Hkv * G;
  const int nchunks = gridDim.y;
  const int chunk = blockIdx.y;
  const int f0 = chunk * kAttnChunk;
  const int nrow = max(0, min(kAttnChunk, total - f0));

  // --- stage the chunk's rows: warp 0 issues one bulk copy per piece
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (wid == 0) {
    int p0 = 0, p1 = 0;
    const unsigned char *selk, *selv;
    if (!v.offload) {
      selk = (const unsigned char *)v.pool_k + gs * v.pool_rows * RB;
      selv = (const unsigned char *)v.pool_v + gs * v.pool_rows * RB;
      if (f0 < nt) {
        const int32_t *cp = v.chunk_piece + gs * (int64_t)(v.max_chunks + 1);
        const int nsc = (nt + kAttnChunk - 1) / kAttnChunk;
        p0 = cp[chunk];
        p1 = (chunk + 1 < nsc) ? cp[chunk + 1] : cp[nsc];
      }
    } else {
      selk = (const unsigned char *)v.stage_k + gs * (int64_t)v.bud_cap * RB;
      selv = (const unsigned char *)v.stage_v + gs * (int64_t)v.bud_cap * RB;
    }
    uint32_t bytes = 0;
    const int4 *pieces = v.pieces + gs * (int64_t)v.max_pieces;
    for (int p = p0 + lane; p < p1; p += 32) bytes += 2u * (uint32_t)pieces[p].z * RB;
    const int win0 = max(f0, nt), win1 = f0 + nrow;  // local-buffer part of the chunk
    int sel_direct = 0;                              // offload: staged rows, one piece
    if (v.offload && f0 < nt) sel_direct = min(f0 + kAttnChunk, nt) - f0;
    if (lane == 0) {
      if (win1 > win0) bytes += 2u * (uint32_t)(win1 - win0) * RB;
      bytes += 2u * (uint32_t)sel_direct * RB;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) bytes += __shfl_xor_sync(kFull, bytes, o);
    if (lane == 0) mbar_arrive_expect_tx(&bar, bytes);
    __syncwarp();
    for (int p = p0 + lane; p < p1; p += 32) {
      const int4 pc = pieces[p];
      const int dr = pc.y - f0;
      bulk_g2s(Ks + dr * RB, selk + (int64_t)pc.x * RB, (uint32_t)pc.z * RB, &bar);
      bulk_g2s(Vs + dr * RB, selv + (int64_t)pc.x * RB, (uint32_t)pc.z * RB, &bar);
    }
    if (lane == 0) {
      if (sel_direct > 0) {
        bulk_g2s(Ks, selk + (int64_t)f0 * RB, (uint32_t)sel_direct * RB, &bar);
        bulk_g2s(Vs, selv + (int64_t)f0 * RB, (uint32_t)sel_direct * RB, &bar);
      }
      if (win1 > win0) {
        const int64_t r0 = gs * v.dec_rows + ws + (win0 - nt);
        bulk_g2s(Ks + (win0 - f0) * RB, (const unsigned char *)v.dec_k + r0 * RB,
                 (uint32_t)(win1 - win0) * RB, &bar);
        bulk_g2s(Vs + (win0 - f0) * RB, (const unsigned char *)v.dec_v + r0 * RB,
                 (uint32_t)(win1 - win0) * RB, &bar);
      }
    }
  }
  // query rows of the group, pre-scaled by log2(e)/sqrt(d) (scores in base 2)
  const float qscale = 1.4426950408889634f * rsqrtf((float)kHeadDim);
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
  for (int x = tid; x < G * kHeadDim; x += blockDim.x)
    qs[x / kHeadDim][x % kHeadDim] = load_elem<DT>(q, qoff + x) * qscale;
  if (tid == 0) s_ok = mbar_wait_bounded(&bar, 0, kWaitLimitNs) ? 1 : 0;
  __syncthreads();
  if (!s_ok) {
    // the copies did not land in time: record it and wait (bounded) once more
    // so that no copy is still writing this block's shared memory at exit
    if (tid == 0) {
      set_err(v.err, kErrTimeout);
      mbar_wait_bounded(&bar, 0, kWaitLimitNs);
    }
    __syncthreads();
  } else {
    mbar_wait_bounded(&bar, 0, kWaitLimitNs);  // completes at once; orders the reads below
  }

  float qr[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) qr[g][e] = qs[g][lane * 4 + e];

  const int own = lane % P;  // partial index (token own / G, head own % G) this lane owns
  float m_own = -INFINITY, l_own = 0.f;
  float acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;

#pragma unroll
  for (int bt = 0; bt < NB; ++bt) {
    const int r0 = wid * kTokPerWarp + bt * TB;
    float part[32];
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      float kk[4];
      row4<DT>(Ks + (r0 + i) * RB, lane, kk);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = qr[g][0] * kk[0];
        s = fmaf(qr[g][1], kk[1], s);
        s = fmaf(qr[g][2], kk[2], s);
        s = fmaf(qr[g][3], kk[3], s);
        part[i * G + g] = s;
      }
    }
#pragma unroll
    for (int j = P; j < 32; ++j) part[j] = 0.f;
    float s = reduce_scatter<P>(part, lane);
    if (r0 + own / G >= nrow) s = -INFINITY;
    float mx = s;
#pragma unroll
    for (int msk = G; msk < P; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, msk));
    const float m_new = fmaxf(m_own, mx);
    const float corr = (m_own == -INFINITY) ? 0.f : exp2f(m_own - m_new);
    const float p = (s == -INFINITY) ? 0.f : exp2f(s - m_new);
    l_own = l_own * corr + p;
    m_own = m_new;
    if (lane < P) ps[wid][lane] = p;
    if (lane < G) cs[wid][lane] = corr;
    __syncwarp();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float c = cs[wid][g];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] *= c;
    }
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      float vv[4];
      row4<DT>(Vs + (r0 + i) * RB, lane, vv);
      if (r0 + i >= nrow) vv[0] = vv[1] = vv[2] = vv[3] = 0.f;  // unwritten shared memory
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = ps[wid][i * G + g];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = fmaf(pg, vv[e], acc[g][e]);
      }
    }
    __syncwarp();
  }
  // per-head totals of this warp
#pragma unroll
  for (int msk = G; msk < P; msk <<= 1) l_own += __shfl_xor_sync(kFull, l_own, msk);
  if (lane < G) {
    wm[wid][lane] = m_own;
    wl[wid][lane] = l_own;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) wacc[wid][g][lane * 4 + e] = acc[g][e];
  __syncthreads();
  // merge the warps into the chunk partial
  const int64_t pbase = (gs * v.max_chunks + chunk) * G;
  for (int x = tid; x < G * kHeadDim; x += blockDim.x) {
    const int g = x / kHeadDim, dim = x % kHeadDim;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) mm = fmaxf(mm, wm[w][g]);
    float o = 0.f, z = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float sw = (wm[w][g] == -INFINITY) ? 0.f : exp2f(wm[w][g] - mm);
      o = fmaf(sw, wacc[w][g][dim], o);
      z = fmaf(sw, wl[w][g], z);
    }
    v.part_acc[(pbase + g) * kHeadDim + dim] = o;
    if (dim == 0) {
      v.part_ml[(pbase + g) * 2] = mm;
      v.part_ml[(pbase + g) * 2 + 1] = z;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&v.attn_count[gs], 1) == nchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA: combine the chunk partials, publish the outputs
  float *out = a.out + k * a.stride_out;
  const int64_t obase = (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
  for (int x = tid; x < G * kHeadDim; x += blockDim.x) {
    const int g = x / kHeadDim, dim = x % kHeadDim;
    float mm = -INFINITY;
    for (int c = 0; c < nchunks; ++c)
      mm = fmaxf(mm, __ldcg(&v.part_ml[((gs * v.max_chunks + c) * G + g) * 2]));
    float o = 0.f, z = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const int64_t pi = (gs * v.max_chunks + c) * G + g;
      const float mc = __ldcg(&v.part_ml[pi * 2]);
      if (mc == -INFINITY) continue;
      const float sw = exp2f(mc - mm);
      o = fmaf(sw, __ldcg(&v.part_acc[pi * kHeadDim + dim]), o);
      z = fmaf(sw, __ldcg(&v.part_ml[pi * 2 + 1]), z);
    }
    out[obase + x] = o / z;
  }
  const int64_t so = ((int64_t)b * a.nl + li) * v.Hkv + h;
  const int ns = v.n_sel[gs];
  if (a.selected_units) {
    const int32_t *sel = v.sel + gs * v.u_cap;
    int32_t *dst = a.selected_units + k * a.stride_sel + so * v.u_cap;
    for (int x = tid; x < ns; x += blockDim.x) dst[x] = sel[x];
  }
  if (tid == 0) {
    if (a.n_selected) a.n_selected[k * a.stride_nsel + so] = ns;
    v.attn_count[gs] = 0;
    atomicAdd((unsigned long long *)&v.counters[kCntAttnRows], (unsigned long long)total);
    atomicAdd((unsigned long long *)&v.counters[kCntAttnSlices], 1ull);
  }
}

// ---------------------------------------------------------------- host

template <int DT, int G>
constexpr size_t attn_smem() { return 2 * kAttnChunk * kHeadDim * elem_bytes<DT>(); }

template <int DT, int G>
static void launch_attn(const CtxView &v, const StepArgs &a, int slices, int nchunks,
                        cudaStream_t st) {
  k_attn<DT, G><<<dim3(slices, nchunks), kAttnWarps * 32, attn_smem<DT, G>(), st>>>(v, a);
}

template <int DT, int G>
static cudaError_t prep_attn() {
  return cudaFuncSetAttribute(k_attn<DT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem<DT, G>());
}

template <int DT>
static cudaError_t prep_dt(int group) {
  switch (group) {
    case 1: return prep_attn<DT, 1>();
    case 2: return prep_attn<DT, 2>();
    case 4: return prep_attn<DT, 4>();
    case 8: return prep_attn<DT, 8>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_kernels(int dtype, int group) {
  return dtype == 1 ? prep_dt<1>(group) : prep_dt<0>(group);
}

template <int DT>
static cudaError_t decode_t(const CtxView &v, const StepArgs &a, cudaStream_t st, Prof &prof) {
  const int slices = a.nl * v.B * v.Hkv;
  prof.begin(kPBoundary, st);
  k_step_boundary<DT><<<a.nl * v.B, 1024, 0, st>>>(v, a);
  prof.end(st);
  prof.begin(kPScore, st);
  k_score<DT><<<dim3(slices, kScoreCtasPerHead), 256, 0, st>>>(v, a);
  prof.end(st);
  prof.begin(kPSelect, st);
  k_select<<<slices, 1024, 0, st>>>(v, a);
  prof.end(st);
  if (v.offload) {
    prof.begin(kPGather, st);
    k_gather_offload<DT><<<dim3(slices, 16), 256, 0, st>>>(v, a);
    prof.end(st);
  }
  const int nchunks = (a.budget + v.L + kAttnChunk - 1) / kAttnChunk;
  prof.begin(kPAttn, st);
  switch (v.G) {
    case 1: launch_attn<DT, 1>(v, a, slices, nchunks, st); break;
    case 2: launch_attn<DT, 2>(v, a, slices, nchunks, st); break;
    case 4: launch_attn<DT, 4>(v, a, slices, nchunks, st); break;
    case 8: launch_attn<DT, 8>(v, a, slices, nchunks, st); break;
    default: return cudaErrorInvalidValue;
  }
  prof.end(st);
  return cudaGetLastError();
}

cudaError_t launch_decode_step(const CtxView &v, const StepArgs &a, cudaStream_t stream,
                               Prof &prof) {
  if (v.dtype == 1) return decode_t<1>(v, a, stream, prof);
  return decode_t<0>(v, a, stream, prof);
}

}  // namespace lkv
