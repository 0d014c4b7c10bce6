// decode.cu -- one decode step of LouisKV-style retrieval for a range of
// layers and all sequences [LouisKV notes, 方法详解 flowchart; 关键设计 1-3]:
//
//   k_step_boundary  r_t, trigger flag, segment close, local-buffer eviction,
//                    append of token t                      (1 CTA / (seq, layer))
//   k_score          s_u = qbar . c_u for every unit         (trigger steps only)
//   k_select         (score desc, id asc) budget prefix      (trigger steps only)
//   k_gather_offload selected rows host -> HBM staging (UVA; offload only)
//   k_attn           split-K softmax attention over selected units + local
//                    buffer, last CTA of each (seq, layer, kv head) combines
#include "lkv_internal.cuh"

namespace lkv {

constexpr int kMaxHeads = 128;

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

__device__ __forceinline__ int64_t slice_of(const CtxView &v, int l, int b, int h) {
  return ((int64_t)l * v.B + b) * v.Hkv + h;
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
  if (tid == 0) st = v.st[lb];
  __syncthreads();
  const int t = st.t;
  const int64_t qoff = ((int64_t)b * a.nl + li) * H * kHeadDim;
  const int64_t kvoff = ((int64_t)b * a.nl + li) * v.Hkv * kHeadDim;

  // 1. r_t = (1/H) sum_h cos(q_{t-1}^h, q_t^h) in fp32, fixed operation order
  if (t > 0) {
    if (tid < H) {
      float dot = 0.f, na = 0.f, nb = 0.f;
      for (int j0 = 0; j0 < kHeadDim; j0 += 16 / elem_bytes<DT>()) {
        float x[8], y[8];
        load16<DT>(v.q_prev, (lb * H + tid) * kHeadDim + j0, x);
        load16<DT>(a.q, qoff + (int64_t)tid * kHeadDim + j0, y);
#pragma unroll
        for (int e = 0; e < 16 / elem_bytes<DT>(); ++e) {
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
      for (int64_t k = tid; k < total; k += nth) {
        const int h = (int)(k / ((int64_t)seg_len * per_row));
        const int rem = (int)(k % ((int64_t)seg_len * per_row));
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
  {
    __shared__ int slow_any;
    if (tid == 0) slow_any = 0;
    __syncthreads();
    int slow = 0;
    for (int k = tid; k < v.Hkv * kHeadDim; k += nth) {
      const int h = k / kHeadDim, dim = k % kHeadDim;
      const int64_t gs = lb * v.Hkv + h;
      const int64_t di = (gs * v.dec_rows + t) * kHeadDim + dim;
      if constexpr (DT == 1) {
        const uint16_t kb = ((const uint16_t *)a.k_new)[kvoff + k];
        ((uint16_t *)v.dec_k)[di] = kb;
        ((uint16_t *)v.dec_v)[di] = ((const uint16_t *)a.v_new)[kvoff + k];
        v.segsum[gs * kHeadDim + dim] += bf16_fixed40(kb, &slow);
      } else {
        const float kf = ((const float *)a.k_new)[kvoff + k];
        ((float *)v.dec_k)[di] = kf;
        ((float *)v.dec_v)[di] = ((const float *)a.v_new)[kvoff + k];
        const double s = __longlong_as_double(v.segsum[gs * kHeadDim + dim]);
        v.segsum[gs * kHeadDim + dim] = __double_as_longlong(__dadd_rn(s, (double)kf));
      }
    }
    if (slow) atomicOr(&slow_any, 1);
    for (int k = tid; k < H * kHeadDim; k += nth) {
      if constexpr (DT == 1)
        ((uint16_t *)v.q_prev)[lb * H * kHeadDim + k] = ((const uint16_t *)a.q)[qoff + k];
      else
        ((float *)v.q_prev)[lb * H * kHeadDim + k] = ((const float *)a.q)[qoff + k];
    }
    __syncthreads();
    if (tid == 0) {
      if (slow_any) st.seg_slow = 1;
      st.t = t + 1;
      v.st[lb] = st;
      const int64_t o = (int64_t)b * a.nl + li;
      if (a.boundary) a.boundary[o] = (uint8_t)st.flag;
      if (a.r_out) a.r_out[o] = st.r;
    }
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
  __shared__ float qbar[kHeadDim];
  const int H = v.Hkv * v.G;
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * v.G) * kHeadDim;
  if (threadIdx.x < kHeadDim) {
    float acc = load_elem<DT>(a.q, qoff + threadIdx.x);
    for (int g = 1; g < v.G; ++g) acc = __fadd_rn(acc, load_elem<DT>(a.q, qoff + (int64_t)g * kHeadDim + threadIdx.x));
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
}

// ---------------------------------------------------------------- selection

__device__ __forceinline__ int32_t block_scan_excl(int32_t x, int32_t *wt, int32_t *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) wt[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int32_t w = lane < nw ? wt[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
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
// order while they fit. Output: ascending unit ids, their first rows and the
// exclusive token prefix of the ranges.
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
  __shared__ int32_t s_total, s_below, s_all;
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
      for (int k = tid; k < 32 * 256; k += nth) (&whist[0][0])[k] = 0;
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
      if (tid == 0) {
        int32_t run = s_below;
        int digit = 255;
        for (int bb = 0; bb < 256; ++bb) {
          if (run + whist[0][bb] > budget) { digit = bb; break; }
          run += whist[0][bb];
        }
        s_below = run;
        s_prefix = prefix | ((uint32_t)digit << shift);
        s_mask = mask | (255u << shift);
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
  __shared__ int32_t s_nsel, s_ntok;
  const int32_t cnt_ex = block_scan_excl(cnt, wt, &s_nsel);
  const int32_t tok_ex = block_scan_excl(toks, wt, &s_ntok);
  {
    int32_t run = tie_ex, k = cnt_ex, cum = tok_ex;
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
        sel_out[k] = u;
        row_out[k] = rows[u];
        cum_out[k] = cum;
        cum += ln[u];
        ++k;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    v.n_sel[gs] = s_nsel;
    v.n_tok[gs] = s_ntok;
    v.rng_cum[gs * (int64_t)(v.u_cap + 1) + s_nsel] = s_ntok;
    if (s_ntok > budget) set_err(v.err, kErrInternal);
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
}

// ---------------------------------------------------------------- attention

constexpr int kAttnWarps = 4;
constexpr int kTokPerWarp = kAttnChunk / kAttnWarps;  // 16

template <int DT, int G>
__global__ void __launch_bounds__(kAttnWarps * 32) k_attn(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const DecState st = v.st[lb];
  const int t_cur = st.t - 1, ws = st.win_start;
  const int nt = v.n_tok[gs], ns = v.n_sel[gs];
  const int total = nt + (t_cur - ws + 1);
  const int H = v.Hkv * G;
  const int nchunks = gridDim.y;
  const int chunk = blockIdx.y;

  __shared__ float qs[G][kHeadDim];
  __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
  __shared__ float wacc[kAttnWarps][G][kHeadDim];
  __shared__ int s_last;
  const float qscale = 1.4426950408889634f / sqrtf((float)kHeadDim);  // log2(e)/sqrt(d)
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
  for (int k = tid; k < G * kHeadDim; k += blockDim.x)
    qs[k / kHeadDim][k % kHeadDim] = load_elem<DT>(a.q, qoff + k) * qscale;
  __syncthreads();

  // this warp's tokens: f = chunk*64 + wid*16 + i
  const int fbase = chunk * kAttnChunk + wid * kTokPerWarp;
  constexpr int eb = elem_bytes<DT>();
  // lane i < 16 resolves the row of token fbase + i: base 0 = selected, 1 = buffer
  int64_t my_off = -1;
  if (lane < kTokPerWarp) {
    const int f = fbase + lane;
    if (f < total) {
      if (f < nt) {
        if (v.offload) {
          my_off = (gs * (int64_t)v.bud_cap + f) * kHeadDim;
        } else {
          const int32_t *cum = v.rng_cum + gs * (int64_t)(v.u_cap + 1);
          const int r = find_range(cum, ns, f);
          const int64_t row = v.rng_row[gs * v.u_cap + r] + (f - cum[r]);
          my_off = (gs * v.pool_rows + row) * kHeadDim;
        }
      } else {
        my_off = (((int64_t)1) << 62) | ((gs * v.dec_rows + ws + (f - nt)) * kHeadDim);
      }
    }
  }
  const void *selk = v.offload ? v.stage_k : v.pool_k;
  const void *selv = v.offload ? v.stage_v : v.pool_v;

  float qr[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) qr[g][e] = qs[g][lane * 4 + e];

  // K rows -> scores (all lanes end with every score)
  float sc[kTokPerWarp][G];
  float m[G];
#pragma unroll
  for (int g = 0; g < G; ++g) m[g] = -INFINITY;
  int64_t offs[kTokPerWarp];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) offs[i] = __shfl_sync(0xffffffffu, my_off, i);
  float kv[kTokPerWarp][4];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
    if (offs[i] >= 0) {
      const bool buf = (offs[i] >> 62) & 1;
      const int64_t o = offs[i] & ((((int64_t)1) << 62) - 1);
      const void *base = buf ? v.dec_k : selk;
      if constexpr (DT == 1) {
        const uint2 raw = __ldg((const uint2 *)((const char *)base + (o + lane * 4) * eb));
        kv[i][0] = __uint_as_float(raw.x << 16); kv[i][1] = __uint_as_float(raw.x & 0xffff0000u);
        kv[i][2] = __uint_as_float(raw.y << 16); kv[i][3] = __uint_as_float(raw.y & 0xffff0000u);
      } else {
        const float4 raw = __ldg((const float4 *)((const char *)base + (o + lane * 4) * eb));
        kv[i][0] = raw.x; kv[i][1] = raw.y; kv[i][2] = raw.z; kv[i][3] = raw.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) kv[i][e] = 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float p = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) p = fmaf(qr[g][e], kv[i][e], p);
#pragma unroll
      for (int o = 16; o; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      sc[i][g] = (offs[i] >= 0) ? p : -INFINITY;
      m[g] = fmaxf(m[g], sc[i][g]);
    }
  }
  // V rows
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
    if (offs[i] >= 0) {
      const bool buf = (offs[i] >> 62) & 1;
      const int64_t o = offs[i] & ((((int64_t)1) << 62) - 1);
      const void *base = buf ? v.dec_v : selv;
      if constexpr (DT == 1) {
        const uint2 raw = __ldg((const uint2 *)((const char *)base + (o + lane * 4) * eb));
        kv[i][0] = __uint_as_float(raw.x << 16); kv[i][1] = __uint_as_float(raw.x & 0xffff0000u);
        kv[i][2] = __uint_as_float(raw.y << 16); kv[i][3] = __uint_as_float(raw.y & 0xffff0000u);
      } else {
        const float4 raw = __ldg((const float4 *)((const char *)base + (o + lane * 4) * eb));
        kv[i][0] = raw.x; kv[i][1] = raw.y; kv[i][2] = raw.z; kv[i][3] = raw.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) kv[i][e] = 0.f;
    }
  }
  float lsum[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    lsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = (m[g] == -INFINITY) ? 0.f : exp2f(sc[i][g] - m[g]);
      lsum[g] += p;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] = fmaf(p, kv[i][e], acc[g][e]);
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int e = 0; e < 4; ++e) wacc[wid][g][lane * 4 + e] = acc[g][e];
    if (lane == 0) { wm[wid][g] = m[g]; wl[wid][g] = lsum[g]; }
  }
  __syncthreads();
  // merge the warps into the chunk partial
  const int64_t pbase = (gs * v.max_chunks + chunk) * G;
  for (int k = tid; k < G * kHeadDim; k += blockDim.x) {
    const int g = k / kHeadDim, dim = k % kHeadDim;
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
  const int64_t obase = (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
  for (int k = tid; k < G * kHeadDim; k += blockDim.x) {
    const int g = k / kHeadDim, dim = k % kHeadDim;
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
    a.out[obase + k] = o / z;
  }
  const int64_t so = ((int64_t)b * a.nl + li) * v.Hkv + h;
  if (a.selected_units) {
    const int32_t *sel = v.sel + gs * v.u_cap;
    for (int k = tid; k < ns; k += blockDim.x) a.selected_units[so * v.u_cap + k] = sel[k];
  }
  if (tid == 0) {
    if (a.n_selected) a.n_selected[so] = ns;
    v.attn_count[gs] = 0;
  }
}

// ---------------------------------------------------------------- host

template <int DT, int G>
static void launch_attn(const CtxView &v, const StepArgs &a, int slices, int nchunks,
                        cudaStream_t st) {
  k_attn<DT, G><<<dim3(slices, nchunks), kAttnWarps * 32, 0, st>>>(v, a);
}

template <int DT>
static cudaError_t decode_t(const CtxView &v, const StepArgs &a, cudaStream_t st) {
  const int slices = a.nl * v.B * v.Hkv;
  k_step_boundary<DT><<<a.nl * v.B, 1024, 0, st>>>(v, a);
  k_score<DT><<<dim3(slices, kScoreCtasPerHead), 256, 0, st>>>(v, a);
  k_select<<<slices, 1024, 0, st>>>(v, a);
  if (v.offload) k_gather_offload<DT><<<dim3(slices, 16), 256, 0, st>>>(v, a);
  const int nchunks = (a.budget + v.L + kAttnChunk - 1) / kAttnChunk;
  switch (v.G) {
    case 1: launch_attn<DT, 1>(v, a, slices, nchunks, st); break;
    case 2: launch_attn<DT, 2>(v, a, slices, nchunks, st); break;
    case 4: launch_attn<DT, 4>(v, a, slices, nchunks, st); break;
    case 8: launch_attn<DT, 8>(v, a, slices, nchunks, st); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_step(const CtxView &v, const StepArgs &a, cudaStream_t stream) {
  if (v.dtype == 1) return decode_t<1>(v, a, stream);
  return decode_t<0>(v, a, stream);
}

}  // namespace lkv
