// decode.cu -- decode steps of LouisKV-style retrieval for a range of layers
// and all sequences [LouisKV notes, 方法详解 flowchart; 关键设计 1-3]:
//
//   k_step_boundary  r_t, trigger flag, segment close, local-buffer eviction,
//                    append of token t, for a chunk of steps    (1 CTA / (seq, layer))
//   k_select         on retrieval steps: s_u = qbar . c_u for every unit, the
//                    (score desc, id asc) budget prefix, the pool row of every
//                    selected token; on every step the attention's descriptor
//                                                              (1 CTA / slice / step)
//   k_gather_offload selected rows host -> HBM staging (UVA; offload only)
//   k_attn_stream    tensor-core attention over (local buffer ++ selected rows)
//                    of every slice, rows split over warps by each slice's size;
//                    the last partial of a slice combines (k_attn: the scalar
//                    variant for fp32 rows or 1-2 query heads)
//
// Inputs/outputs of step k of a call live at base + k * stride (StepArgs).
#include <cstdlib>
#include <type_traits>

#include "lkv_internal.cuh"
#include "paris.cuh"

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

// Programmatic dependent launch: a kernel waits here for the previous kernel
// in the stream to complete (and its writes to be visible) before it touches
// any state; the next kernel may be scheduled as soon as this one signals.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ParisKV-style selector: the metadata of the keys the chunk's steps
// appended (a CTA per (sequence, layer) and step, a warp per KV head), after
// the boundary kernel and before the chunk's selections.
__global__ void __launch_bounds__(512) k_paris_append(CtxView v, StepArgs a) {
  const int li = blockIdx.x / v.B, b = blockIdx.x % v.B;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int wid = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  if (wid >= v.Hkv) return;
  const int t = v.aview[(int64_t)(a.slot + blockIdx.y) * v.n_lb + lb].x;
  const int64_t k = t - a.base_t;
  const uint16_t *kn = (const uint16_t *)a.k_new + k * a.stride_kv +
                       (((int64_t)b * a.nl + li) * v.Hkv + wid) * kHeadDim;
  const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(kn) + (threadIdx.x & 31));
  const uint16_t k4[4] = {(uint16_t)(raw.x & 0xffffu), (uint16_t)(raw.x >> 16), (uint16_t)(raw.y & 0xffffu),
                          (uint16_t)(raw.y >> 16)};
  const int64_t row = (lb * v.Hkv + wid) * v.pool_rows + v.n_cap + t;
  paris_encode_warp(k4, v.paris_sign, v.paris_thr, v.paris_lev, v.pk_bucket + row * kParisSub,
                    v.pk_code + row * 64, v.pk_w + row * kParisSub);
}

// 512 threads (64 registers each), the queries staged in their own dtype.
constexpr int kBoundaryThreads = 512;
constexpr int kQPitch = kHeadDim + 8;  // padded query rows in shared memory (elements)

// One staged query element as a float.
template <int DT>
__device__ __forceinline__ float qs_get(const void *qs, int i) {
  if constexpr (DT == 1) return __uint_as_float(((uint32_t)((const uint16_t *)qs)[i]) << 16);
  else return ((const float *)qs)[i];
}

// n_steps consecutive decode steps of one (sequence, layer) per CTA, step i
// in step slot a.slot + i. The state machine (segments, local buffer,
// evictions, plan slot) is sequential, but it depends only on the step
// inputs, never on a selection or an attention, so one launch runs a whole
// chunk of steps ahead of the selections and attentions that read its
// per-step views.
template <int DT>
__global__ void __launch_bounds__(kBoundaryThreads, 2) k_step_boundary(CtxView v, StepArgs a, int n_steps) {
  const int li = blockIdx.x / v.B, b = blockIdx.x % v.B;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int H = v.Hkv * v.G;
  const int tid = threadIdx.x, nth = blockDim.x;
  __shared__ DecState st;
  __shared__ float cosv[kMaxHeads];
  __shared__ int slow_any;
  // [2][H][kQPitch] elements of the dtype: previous and current queries
  extern __shared__ __align__(16) unsigned char qsm_raw[];
  using QT = typename std::conditional<DT == 1, uint16_t, float>::type;
  QT *qsm = reinterpret_cast<QT *>(qsm_raw);
  pdl_wait();
  pdl_trigger();
  if (tid == 0) st = v.st[lb];
  // loads that do not depend on the step go out with the state's: the
  // previous queries (16-byte vectors into padded shared rows) and this
  // thread's running sums of the open segment
  constexpr int per16 = 16 / elem_bytes<DT>();
  const int nvec = H * kHeadDim / per16;
  for (int y = tid; y < nvec; y += nth) {
    const int head = y / (kHeadDim / per16), j0 = (y % (kHeadDim / per16)) * per16;
    *(uint4 *)(qsm + (int64_t)head * kQPitch + j0) =
        __ldg((const uint4 *)((const QT *)v.q_prev + (lb * H + head) * kHeadDim + j0));
  }
  constexpr int kMaxPer = 16 * kHeadDim / kBoundaryThreads;  // Hkv * d <= 2048
  // the new key and value elements: one register a pair for bf16 (key in
  // the high half), two for fp32
  uint32_t kbits[kMaxPer], vbits[DT == 1 ? 1 : kMaxPer];
  int64_t ssum[kMaxPer];
#pragma unroll
  for (int r = 0; r < kMaxPer; ++r) {
    const int x = tid + r * nth;
    if (x < v.Hkv * kHeadDim) ssum[r] = v.segsum[(lb * v.Hkv + x / kHeadDim) * kHeadDim + x % kHeadDim];
  }
  __syncthreads();
  for (int i_step = 0; i_step < n_steps; ++i_step) {
  // queries of step t - 1 in buffer pb, of step t in cb
  const int pb = i_step & 1, cb = pb ^ 1;
  const int slot = a.slot + i_step;
  if (tid == 0) slow_any = 0;
  const int t = st.t;
  const int n_closed0 = st.n_closed;
  const int64_t k = t - a.base_t;
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  const void *k_new = (const char *)a.k_new + k * a.stride_kv * elem_bytes<DT>();
  const void *v_new = (const char *)a.v_new + k * a.stride_kv * elem_bytes<DT>();
  const int64_t qoff = ((int64_t)b * a.nl + li) * H * kHeadDim;
  const int64_t kvoff = ((int64_t)b * a.nl + li) * v.Hkv * kHeadDim;
  // then the step's inputs: the new key/value elements and the current queries
#pragma unroll
  for (int r = 0; r < kMaxPer; ++r) {
    const int x = tid + r * nth;
    if (x < v.Hkv * kHeadDim) {
      if constexpr (DT == 1) {
        kbits[r] = ((uint32_t)((const uint16_t *)k_new)[kvoff + x] << 16) |
                   (uint32_t)((const uint16_t *)v_new)[kvoff + x];
      } else {
        kbits[r] = __float_as_uint(((const float *)k_new)[kvoff + x]);
        vbits[DT == 1 ? 0 : r] = __float_as_uint(((const float *)v_new)[kvoff + x]);
      }
    }
  }
  for (int y = tid; y < nvec; y += nth) {
    const int head = y / (kHeadDim / per16), j0 = (y % (kHeadDim / per16)) * per16;
    *(uint4 *)(qsm + ((int64_t)cb * H + head) * kQPitch + j0) =
        __ldg((const uint4 *)((const QT *)q + qoff + (int64_t)head * kHeadDim + j0));
  }
  __syncthreads();

  // 1. r_t = (1/H) sum_h cos(q_{t-1}^h, q_t^h) in fp32, fixed operation order
  if (t > 0) {
    if (tid < H) {
      const QT *x = qsm + ((int64_t)pb * H + tid) * kQPitch;
      const QT *y = qsm + ((int64_t)cb * H + tid) * kQPitch;
      float dot = 0.f, na = 0.f, nb = 0.f;
#pragma unroll 8
      for (int j = 0; j < kHeadDim; ++j) {
        const float xv = qs_get<DT>(x, j), yv = qs_get<DT>(y, j);
        dot = __fmaf_rn(xv, yv, dot);
        na = __fmaf_rn(xv, xv, na);
        nb = __fmaf_rn(yv, yv, nb);
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
      // the policy's trigger (r_t is computed and reported under every one)
      st.flag = v.pol_trigger == kTrigEvery      ? 1
                : v.pol_trigger == kTrigInterval ? (t % v.pol_interval == 0 ? 1 : 0)
                                                 : (r < a.tau ? 1 : 0);
      if (st.flag) st.plan = (st.plan + 1) % v.plan_ring;  // a retrieval writes the next plan slot
    }
  } else if (tid == 0) {
    st.r = 0.f;
    st.flag = 1;
    st.plan = (st.plan + 1) % v.plan_ring;
  }
  __syncthreads();

  // 2. a boundary (with page units: a full page) closes the open segment;
  //    token t opens the next one
  const bool cut = v.pol_page > 0 ? t - st.open_start >= v.pol_page : st.flag != 0;
  if (cut && t > 0 && st.open_start < t) {
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
  //    (a segment closed during this step restarted the sum at zero)
  const bool restarted = st.n_closed != n_closed0;
  int slow = 0;
  // a segment spans at most L tokens: with every |key| below 2^(e_hi - 126)
  // its sum of magnitudes stays below 2^13, so the exact sum is also the
  // token-order double sum
  const uint32_t e_hi = min(131u, 139u - (32u - (uint32_t)__clz(max(v.L, 1) - 1)));
#pragma unroll
  for (int r = 0; r < kMaxPer; ++r) {
    const int x = tid + r * nth;
    if (x >= v.Hkv * kHeadDim) continue;
    const int h = x / kHeadDim, dim = x % kHeadDim;
    const int64_t gs = lb * v.Hkv + h;
    const int64_t di = (gs * v.dec_rows + t) * kHeadDim + dim;
    const int64_t prev = restarted ? 0 : ssum[r];
    if constexpr (DT == 1) {
      ((uint16_t *)v.dec_k)[di] = (uint16_t)(kbits[r] >> 16);
      ((uint16_t *)v.dec_v)[di] = (uint16_t)(kbits[r] & 0xffffu);
      ssum[r] = prev + bf16_fixed40((uint16_t)(kbits[r] >> 16), &slow, e_hi);
    } else {
      ((float *)v.dec_k)[di] = __uint_as_float(kbits[r]);
      ((float *)v.dec_v)[di] = __uint_as_float(vbits[DT == 1 ? 0 : r]);
      ssum[r] = __double_as_longlong(__dadd_rn(__longlong_as_double(prev), (double)__uint_as_float(kbits[r])));
    }
    v.segsum[gs * kHeadDim + dim] = ssum[r];
  }
  if (slow) atomicOr(&slow_any, 1);
  // the attention gets this step's queries pre-scaled by log2(e)/sqrt(d)
  // (its scores are in base 2)
  const float qscale = 1.4426950408889634f * rsqrtf((float)kHeadDim);
  for (int y = tid; y < nvec; y += nth) {
    const int head = y / (kHeadDim / per16), j0 = (y % (kHeadDim / per16)) * per16;
    const QT *src = qsm + ((int64_t)cb * H + head) * kQPitch + j0;
    float4 *qa = (float4 *)(v.q_attn + (((int64_t)slot * v.n_lb + lb) * H + head) * kHeadDim + j0);
#pragma unroll
    for (int i = 0; i < per16 / 4; ++i)
      qa[i] = make_float4(qs_get<DT>(src, 4 * i) * qscale, qs_get<DT>(src, 4 * i + 1) * qscale,
                          qs_get<DT>(src, 4 * i + 2) * qscale, qs_get<DT>(src, 4 * i + 3) * qscale);
    if (i_step == n_steps - 1)  // the last step's queries become the previous ones
      *(uint4 *)((QT *)v.q_prev + (lb * H + head) * kHeadDim + j0) = *(const uint4 *)src;
  }
  __syncthreads();
  if (tid == 0) {
    if (slow_any) st.seg_slow = 1;
    st.t = t + 1;
    // what this step's scoring, selection and attention need, in its slot
    v.aview[(int64_t)slot * v.n_lb + lb] = make_int4(t, st.win_start, st.plan, st.n_units * 2 + st.flag);
    const int64_t o = (int64_t)b * a.nl + li;
    if (a.boundary) a.boundary[k * a.stride_b + o] = (uint8_t)st.flag;
    if (a.r_out) a.r_out[k * a.stride_b + o] = st.r;
    if (i_step == n_steps - 1) v.st[lb] = st;
  }
  __syncthreads();
  }  // steps
}

// ---------------------------------------------------------------- scoring + selection

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

// The same for two values at once (one pass of barriers).
__device__ __forceinline__ int2 block_scan_excl2(int32_t x, int32_t y, int32_t *wt, int32_t *tx,
                                                 int32_t *ty) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t ix = x, iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t a = __shfl_up_sync(kFull, ix, o), b = __shfl_up_sync(kFull, iy, o);
    if (lane >= o) { ix += a; iy += b; }
  }
  if (lane == 31) { wt[wid] = ix; wt[32 + wid] = iy; }
  __syncthreads();
  if (wid == 0) {
    int32_t a = lane < nw ? wt[lane] : 0, b = lane < nw ? wt[32 + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t pa = __shfl_up_sync(kFull, a, o), pb = __shfl_up_sync(kFull, b, o);
      if (lane >= o) { a += pa; b += pb; }
    }
    if (lane < nw) { wt[lane] = a; wt[32 + lane] = b; }
    if (lane == nw - 1) { *tx = a; *ty = b; }
  }
  __syncthreads();
  const int2 r = make_int2(ix - x + (wid ? wt[wid - 1] : 0), iy - y + (wid ? wt[32 + wid - 1] : 0));
  __syncthreads();
  return r;
}

// threads of the scoring + selection kernel: with at most 85 registers each a
// CTA fits on an SM beside two attention CTAs
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;

// Budget selection of one (seq, layer, kv head) by the whole block: a
// length-weighted radix select of the cut K* (the smallest desc_key value
// with sum_{key <= K*} len > budget). Units with key < K* all precede the
// first unit that does not fit; units with key == K* are taken in id order
// while they fit. Output: ascending unit ids, their first rows, the exclusive
// token prefix, and the copy plan (selected rows cut at 64-token chunk
// boundaries).
constexpr int kSelSmemUnits = 4096;  // units whose keys, lengths and rows fit in shared memory
constexpr size_t kSelSmemBytes = (size_t)kSelSmemUnits * 12;

// Length-weighted radix select of the budget cut over the units' descending
// keys: cut->all when every unit fits; else cut->prefix = K*, the smallest
// key with sum_{key <= K*} len > budget, and cut->below = the length of the
// units with key < K*. Called by the whole block; whist and wt are scratch.
struct RadixCut {
  int32_t total, all, below;
  uint32_t prefix, mask;
};

template <typename KeyOf, typename LenOf>
__device__ void radix_cut(int U, int budget, KeyOf keyof, LenOf lenof, int32_t (*whist)[256], int32_t *wt,
                          RadixCut *cut) {
  const int tid = threadIdx.x, nth = blockDim.x, wid = tid >> 5;
  int32_t part = 0;
  for (int u = tid; u < U; u += nth) part += lenof(u);
  block_scan_excl(part, wt, &cut->total);
  if (tid == 0) {
    cut->all = cut->total <= budget;
    cut->prefix = 0;
    cut->mask = 0;
    cut->below = 0;
  }
  __syncthreads();
  if (!cut->all) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int x = tid; x < kScoreWarps * 256; x += nth) (&whist[0][0])[x] = 0;
      __syncthreads();
      const uint32_t prefix = cut->prefix, mask = cut->mask;
      for (int u = tid; u < U; u += nth) {
        const uint32_t key = keyof(u);
        if ((key & mask) == prefix) atomicAdd(&whist[wid][(key >> shift) & 255u], lenof(u));
      }
      __syncthreads();
      for (int bin = tid; bin < 256; bin += nth) {
        int32_t tot = 0;
        for (int w = 0; w < kScoreWarps; ++w) tot += whist[w][bin];
        whist[0][bin] = tot;
      }
      __syncthreads();
      if (tid < 32) {
        // warp scan over the 256 bins (8 per lane): the bin where the running
        // weight first exceeds the budget
        int32_t loc[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) { loc[e] = whist[0][tid * 8 + e]; sum += loc[e]; }
        int32_t inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(kFull, inc, o);
          if (tid >= o) inc += y;
        }
        int found = -1;
        int32_t run = cut->below + inc - sum;
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
          cut->below = below;
          cut->prefix = prefix | ((uint32_t)digit << shift);
          cut->mask = mask | (255u << shift);
        }
      }
      __syncthreads();
    }
  }
}

// Skip-and-continue budget fill on top of the stop-at-first-misfit prefix.
// Walking the selection order and taking every unit that still fits is the
// same as repeatedly taking the first unit in that order (smallest key, then
// smallest id) among the unmarked ones whose length fits what is left: a
// unit passed over earlier did not fit a larger remainder. Units of length 0
// always fit and are marked at once. Marks one bit per unit in `mark`.
template <typename Prefix, typename KeyOf, typename LenOf>
__device__ void skip_fill(int U, int budget, int u0, int u1, int32_t tie_ex, Prefix is_prefix,
                          KeyOf keyof, LenOf lenof, uint32_t *mark, int32_t *wt) {
  const int tid = threadIdx.x, nth = blockDim.x;
  __shared__ unsigned long long s_best;
  __shared__ int32_t s_left, s_tot;
  for (int w = tid; w < (U + 31) / 32; w += nth) mark[w] = 0;
  __syncthreads();
  int32_t run = tie_ex, toks = 0;
  for (int u = u0; u < u1; ++u)
    if (is_prefix(u, run)) {
      atomicOr(&mark[u >> 5], 1u << (u & 31));
      toks += lenof(u);
    }
  block_scan_excl(toks, wt, &s_tot);  // (its barriers also publish the marks)
  if (tid == 0) s_left = budget - s_tot;
  __syncthreads();
  for (int u = tid; u < U; u += nth)
    if (lenof(u) == 0 && !((mark[u >> 5] >> (u & 31)) & 1u)) atomicOr(&mark[u >> 5], 1u << (u & 31));
  __syncthreads();
  for (int it = 0; it < U; ++it) {
    const int32_t left = s_left;
    unsigned long long best = ~0ull;
    for (int u = tid; u < U; u += nth) {
      const int32_t len = lenof(u);
      if (len <= left && !((mark[u >> 5] >> (u & 31)) & 1u)) {
        const unsigned long long c = ((unsigned long long)keyof(u) << 32) | (uint32_t)u;
        best = c < best ? c : best;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(kFull, best, o);
      best = y < best ? y : best;
    }
    if (tid == 0) s_best = ~0ull;
    __syncthreads();
    if ((tid & 31) == 0 && best != ~0ull) atomicMin(&s_best, best);
    __syncthreads();
    const unsigned long long b = s_best;
    if (b == ~0ull) break;
    const int u = (int)(uint32_t)b;
    if (tid == 0) {
      mark[u >> 5] |= 1u << (u & 31);
      s_left = left - lenof(u);
    }
    __syncthreads();
  }
}

// Keys, lengths and first pool rows of the units go into shared memory in one
// round of loads (very large unit tables stay in global memory), unless the
// caller already put the keys there (keys_in_smem); scg: the step's scores.
__device__ void select_units(const CtxView &v, int64_t gs, int U, int budget, int ps, const float *scg,
                             bool keys_in_smem) {
  const int tid = threadIdx.x, nth = blockDim.x, wid = tid >> 5;
  extern __shared__ __align__(16) uint32_t sel_smem[];
  uint32_t *key_s = sel_smem;
  int32_t *len_s = (int32_t *)(sel_smem + kSelSmemUnits);
  int32_t *row_s = (int32_t *)(sel_smem + 2 * kSelSmemUnits);
  const int32_t *lng = v.unit_len + gs * v.u_cap;
  const int32_t *rwg = v.unit_row + gs * v.u_cap;
  const bool in_smem = U <= kSelSmemUnits;
  if (in_smem)
    for (int u = tid; u < U; u += nth) {
      if (!keys_in_smem) key_s[u] = desc_key(__ldcg(scg + u));
      len_s[u] = lng[u];
      row_s[u] = rwg[u];
    }
  __syncthreads();
  auto keyof = [&](int u) -> uint32_t { return in_smem ? key_s[u] : desc_key(__ldcg(scg + u)); };
  auto lenof = [&](int u) -> int32_t { return in_smem ? len_s[u] : lng[u]; };
  auto rowof = [&](int u) -> int32_t { return in_smem ? row_s[u] : rwg[u]; };
  __shared__ int32_t whist[kScoreWarps][256];
  __shared__ int32_t wt[64];
  __shared__ int32_t s_nsel, s_ntok, s_npieces;
  __shared__ RadixCut rc;
  radix_cut(U, budget, keyof, lenof, whist, wt, &rc);
  const bool all = rc.all != 0;
  const uint32_t kstar = rc.prefix;
  const int32_t below = rc.below;
  const int per = (U + nth - 1) / nth;
  const int u0 = tid * per, u1 = min(U, u0 + per);
  // skip-and-continue fill: the prefix below is extended unit by unit in
  // shared-memory marks (up to kSelSmemUnits units)
  __shared__ uint32_t s_mark[kSelSmemUnits / 32];
  const bool skip = v.pol_fill == kFillSkip && !all && in_smem;
  if (v.pol_fill == kFillSkip && !all && !in_smem && tid == 0) set_err(v.err, kErrCapacity);
  auto marked = [&](int u) -> bool { return (s_mark[u >> 5] >> (u & 31)) & 1u; };
  auto is_prefix = [&](int u, int32_t &run) -> bool {
    if (all) return true;
    const uint32_t key = keyof(u);
    if (key < kstar) return true;
    if (key == kstar) {
      run += lenof(u);
      return below + run <= budget;
    }
    return false;
  };
  auto is_sel = [&](int u, int32_t &run) -> bool { return skip ? marked(u) : is_prefix(u, run); };
  // exclusive id-order prefix of the tied units' lengths
  int32_t tl = 0;
  if (!all)
    for (int u = u0; u < u1; ++u)
      if (keyof(u) == kstar) tl += lenof(u);
  const int32_t tie_ex = block_scan_excl(tl, wt, nullptr);
  if (skip) skip_fill(U, budget, u0, u1, tie_ex, is_prefix, keyof, lenof, s_mark, wt);
  int32_t cnt = 0, toks = 0;
  {
    int32_t run = tie_ex;
    for (int u = u0; u < u1; ++u)
      if (is_sel(u, run)) { ++cnt; toks += lenof(u); }
  }
  const int2 ex = block_scan_excl2(cnt, toks, wt, &s_nsel, &s_ntok);
  const int32_t cnt_ex = ex.x, tok_ex = ex.y;
  int32_t npc = 0;  // copy pieces of this thread's selected units (when a reader needs them)
  // the selected units' first rows and token offsets, also kept in shared
  // memory (the radix histograms are free now) so that the pool row of every
  // selected token can be written by one thread per token
  constexpr int kSelStage = kScoreWarps * 256 / 2;
  int32_t *cum_sh = &whist[0][0], *row_sh = cum_sh + kSelStage;
  int32_t *tok_rows = v.offload ? nullptr : plan_sel_rows(v, ps, gs);
  const bool staged = s_nsel <= kSelStage;
  {
    int32_t run = tie_ex, kk = cnt_ex, cum = tok_ex;
    int32_t *sel_out = plan_sel(v, ps, gs);
    for (int u = u0; u < u1; ++u) {
      if (!is_sel(u, run)) continue;
      const int32_t len = lenof(u), row = rowof(u);
      sel_out[kk] = u;
      if (staged) {
        cum_sh[kk] = cum;
        row_sh[kk] = row;
      } else if (tok_rows) {
        for (int32_t j = 0; j < len && cum + j < v.sel_cap; ++j) tok_rows[cum + j] = row + j;
      }
      if (v.need_pieces && len > 0) npc += (cum + len - 1) / kAttnChunk - cum / kAttnChunk + 1;
      cum += len;
      ++kk;
    }
  }
  if (staged && tok_rows) {
    __syncthreads();
    // token x belongs to the last selected unit whose offset is <= x
    const int nsel = s_nsel, ntk = min(s_ntok, v.sel_cap);
    for (int x = tid; x < ntk; x += nth) {
      int lo = 0, hi = nsel - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum_sh[mid] <= x) lo = mid;
        else hi = mid - 1;
      }
      tok_rows[x] = row_sh[lo] + (x - cum_sh[lo]);
    }
  }
  if (tid == 0) s_npieces = 0;
  const int32_t pc_ex = v.need_pieces ? block_scan_excl(npc, wt, &s_npieces) : 0;
  if (v.need_pieces) {
    int32_t run = tie_ex, cum = tok_ex, p = pc_ex;
    int4 *pieces = v.pieces + gs * (int64_t)v.max_pieces;
    int32_t *cp = v.chunk_piece + gs * (int64_t)(v.max_chunks + 1);
    for (int u = u0; u < u1 && p - pc_ex < npc; ++u) {
      if (!is_sel(u, run)) continue;
      int32_t len = lenof(u), src = rowof(u), f = cum;
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
  const int nsc = (s_ntok + kAttnChunk - 1) / kAttnChunk;
  if (tid == 0) {
    *plan_nsel(v, ps, gs) = s_nsel;
    *plan_ntok(v, ps, gs) = s_ntok;
    atomicAdd((unsigned long long *)&v.counters[kCntSelUnits], (unsigned long long)s_nsel);
    atomicAdd((unsigned long long *)&v.counters[kCntSelTokens], (unsigned long long)s_ntok);
    if (v.need_pieces && nsc <= v.max_chunks) v.chunk_piece[gs * (int64_t)(v.max_chunks + 1) + nsc] = s_npieces;
    if (s_ntok > budget || s_ntok > v.sel_cap || s_npieces > v.max_pieces || nsc > v.max_chunks)
      set_err(v.err, kErrInternal);
  }
  __syncthreads();
  // the same pieces, grouped per chunk in fixed 64-slot blocks (a chunk of 64
  // rows has at most 64 pieces) so that the attention reads them in one go
  if (v.need_pieces && nsc <= v.max_chunks && s_npieces <= v.max_pieces) {
    const int32_t *cp = v.chunk_piece + gs * (int64_t)(v.max_chunks + 1);
    const int4 *pieces = v.pieces + gs * (int64_t)v.max_pieces;
    for (int p = tid; p < s_npieces; p += nth) {
      const int4 pc = pieces[p];
      const int c = pc.y / kAttnChunk;
      int4 q = pc;
      if (p == cp[c]) q.w = cp[c + 1] - cp[c];  // the chunk's piece count rides on its first piece
      plan_chunk_pieces(v, ps, gs)[c * kAttnChunk + (p - cp[c])] = q;
    }
    for (int c = tid; c < nsc; c += nth)
      plan_chunk_count(v, ps, gs)[c] = cp[c + 1] - cp[c];
  }
}

// Per-query-head selection, the baseline of the group-consistent one ("LouisKV
// ... Long Input-Output Sequences", 关键设计 3 其二 and 消融实验: selecting per
// head makes the heads of a group fetch overlapping sets). Each of the G
// query heads of the slice scores every unit with its own query, s_u = q_h .
// c_u (the fp32 FMA chain of the group score with q_h in place of the group
// sum), and takes its own budget selection (prefix or skip fill, radix cut
// as in select_units). The plan lists the union of the heads' units in id
// order with the mask of heads that chose each, the per-head counts, and the
// union's token rows with the mask in the top byte, from which the attention
// masks every head's scores to its own selection. Units in shared memory only
// (at most kSelSmemUnits; more is a capacity error). Shared memory: keys,
// lengths and rows (kSelSmemBytes), then head masks, skip marks and the
// radix histograms (kSelHeadSmemBytes in all).
constexpr size_t kSelHeadSmemBytes = kSelSmemBytes + kSelSmemUnits + kSelSmemUnits / 8 +
                                     (size_t)kScoreWarps * 256 * 4;

template <int DT>
__device__ __noinline__ void select_heads(const CtxView &v, int64_t gs, int U, int budget, int ps, const void *q,
                             int64_t qoff) {
  const int tid = threadIdx.x, nth = blockDim.x;
  extern __shared__ __align__(16) uint32_t sel_smem[];
  uint32_t *key_s = sel_smem;
  int32_t *len_s = (int32_t *)(sel_smem + kSelSmemUnits);
  int32_t *row_s = (int32_t *)(sel_smem + 2 * kSelSmemUnits);
  uint8_t *hm = (uint8_t *)(sel_smem + 3 * kSelSmemUnits);
  uint32_t *mark = sel_smem + 3 * kSelSmemUnits + kSelSmemUnits / 4;
  int32_t(*whist)[256] = reinterpret_cast<int32_t(*)[256]>(mark + kSelSmemUnits / 32);
  __shared__ int32_t wt[64];
  __shared__ RadixCut rc;
  __shared__ float qs[kHeadDim];
  __shared__ int32_t s_cnt, s_tok, s_nsel, s_ntok;
  int32_t *hn = plan_hsel_n(v, ps, gs), *ht = plan_hsel_tok(v, ps, gs);
  if (U > kSelSmemUnits) {
    if (tid == 0) {
      set_err(v.err, kErrCapacity);
      *plan_nsel(v, ps, gs) = 0;
      *plan_ntok(v, ps, gs) = 0;
      for (int g = 0; g < v.G; ++g) hn[g] = ht[g] = 0;
    }
    return;
  }
  const int32_t *lng = v.unit_len + gs * v.u_cap, *rwg = v.unit_row + gs * v.u_cap;
  for (int u = tid; u < U; u += nth) {
    len_s[u] = lng[u];
    row_s[u] = rwg[u];
    hm[u] = 0;
  }
  const int per = (U + nth - 1) / nth;
  const int u0 = tid * per, u1 = min(U, u0 + per);
  auto keyof = [&](int u) -> uint32_t { return key_s[u]; };
  auto lenof = [&](int u) -> int32_t { return len_s[u]; };
  constexpr int nvec = kHeadDim * elem_bytes<DT>() / 16;
  const uint4 *rows = (const uint4 *)((const char *)v.cent_op + gs * v.u_cap * kHeadDim * elem_bytes<DT>());
  for (int g = 0; g < v.G; ++g) {
    __syncthreads();  // the previous head is done with the keys and the query
    if (tid < kHeadDim) qs[tid] = load_elem<DT>(q, qoff + (int64_t)g * kHeadDim + tid);
    __syncthreads();
    for (int u = tid; u < U; u += nth) {
      float sc = 0.f;
#pragma unroll
      for (int j = 0; j < nvec; ++j) {
        const uint4 cur = __ldg(rows + (int64_t)u * nvec + j);
        const uint32_t w[4] = {cur.x, cur.y, cur.z, cur.w};
        if constexpr (DT == 1) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc = __fmaf_rn(qs[j * 8 + 2 * e], __uint_as_float(w[e] << 16), sc);
            sc = __fmaf_rn(qs[j * 8 + 2 * e + 1], __uint_as_float(w[e] & 0xffff0000u), sc);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) sc = __fmaf_rn(qs[j * 4 + e], __uint_as_float(w[e]), sc);
        }
      }
      key_s[u] = desc_key(sc);
    }
    __syncthreads();
    radix_cut(U, budget, keyof, lenof, whist, wt, &rc);
    const bool all = rc.all != 0;
    const uint32_t kstar = rc.prefix;
    const int32_t below = rc.below;
    auto is_prefix = [&](int u, int32_t &run) -> bool {
      if (all) return true;
      const uint32_t key = key_s[u];
      if (key < kstar) return true;
      if (key == kstar) {
        run += len_s[u];
        return below + run <= budget;
      }
      return false;
    };
    int32_t tl = 0;
    if (!all)
      for (int u = u0; u < u1; ++u)
        if (key_s[u] == kstar) tl += len_s[u];
    const int32_t tie_ex = block_scan_excl(tl, wt, nullptr);
    const bool skip = v.pol_fill == kFillSkip && !all;
    if (skip) skip_fill(U, budget, u0, u1, tie_ex, is_prefix, keyof, lenof, mark, wt);
    int32_t cnt = 0, toks = 0, run = tie_ex;
    for (int u = u0; u < u1; ++u) {
      const bool on = skip ? ((mark[u >> 5] >> (u & 31)) & 1u) != 0 : is_prefix(u, run);
      if (on) {
        hm[u] |= (uint8_t)(1u << g);
        ++cnt;
        toks += len_s[u];
      }
    }
    block_scan_excl2(cnt, toks, wt, &s_cnt, &s_tok);
    if (tid == 0) {
      hn[g] = s_cnt;
      ht[g] = s_tok;
      atomicAdd((unsigned long long *)&v.counters[kCntSelUnits], (unsigned long long)s_cnt);
      atomicAdd((unsigned long long *)&v.counters[kCntSelTokens], (unsigned long long)s_tok);
      if (s_tok > budget) set_err(v.err, kErrInternal);
    }
  }
  __syncthreads();
  // the union, in id order
  int32_t cnt = 0, toks = 0;
  for (int u = u0; u < u1; ++u)
    if (hm[u]) {
      ++cnt;
      toks += len_s[u];
    }
  const int2 ex = block_scan_excl2(cnt, toks, wt, &s_nsel, &s_ntok);
  int32_t *sel_out = plan_sel(v, ps, gs);
  uint8_t *msk_out = plan_sel_mask(v, ps, gs);
  int32_t *tok_rows = plan_sel_rows(v, ps, gs);
  int32_t kk = ex.x, cum = ex.y;
  for (int u = u0; u < u1; ++u) {
    const uint32_t m = hm[u];
    if (!m) continue;
    sel_out[kk] = u;
    msk_out[kk] = (uint8_t)m;
    const int32_t len = len_s[u], row = row_s[u];
    for (int32_t j = 0; j < len && cum + j < v.sel_cap; ++j) tok_rows[cum + j] = (row + j) | (int32_t)(m << kRowBits);
    cum += len;
    ++kk;
  }
  if (tid == 0) {
    *plan_nsel(v, ps, gs) = s_nsel;
    *plan_ntok(v, ps, gs) = s_ntok;
    if (s_ntok > v.sel_cap) set_err(v.err, kErrInternal);
  }
}

// ParisKV-style token selection of one (slice, step) (ParisKV technical
// summary, 核心算法创新 2: a coarse collision vote, then a rerank of the
// candidates on the compact codes). The region is every prefill token and
// every decode token that left the local buffer. The rotated group query
// qr = H D qbar is formed in single precision by the fast Hadamard
// butterfly; in each subspace the rho sign patterns p with the highest
// sim_p = sum_j +-qr_j (ties to the lower p) vote rho - r for the tokens in
// their bucket; the n_cand tokens with the highest vote sums (ties to the
// lower token) are reranked by est = sum_b w_b <v_b, qr_b>; the budget best
// by (est desc, token asc) are selected. The plan lists their pool rows in
// token order (as units and as per-token rows: every "unit" is one token).
// Shared memory: candidate keys, pattern similarities (later the radix
// histograms), candidate tokens, votes and the vote-sum histogram.
constexpr size_t kSelParisSmemBytes = kSelSmemBytes + kParisSub * 256 + 256 * 4;

template <int DT>
__device__ __noinline__ void select_paris(const CtxView &v, int64_t lb, int64_t gs, int budget, int ps, int slot,
                             const void *q, int64_t qoff, int win_start) {
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, wid = tid >> 5;
  extern __shared__ __align__(16) uint32_t sel_smem[];
  uint32_t *key_s = sel_smem;
  float *sim = reinterpret_cast<float *>(sel_smem + kSelSmemUnits);
  int32_t(*whist)[256] = reinterpret_cast<int32_t(*)[256]>(sel_smem + kSelSmemUnits);
  int32_t *cand = reinterpret_cast<int32_t *>(sel_smem + 2 * kSelSmemUnits);
  uint8_t *vote = reinterpret_cast<uint8_t *>(sel_smem + 3 * kSelSmemUnits);
  int32_t *hist = reinterpret_cast<int32_t *>(vote + kParisSub * 256);
  __shared__ float qr[kHeadDim], levs[8];
  __shared__ int32_t wt[64];
  __shared__ RadixCut rc;
  __shared__ int32_t s_cut, s_need, s_nc, s_nsel, s_dummy;
  const int64_t N = v.st[lb].n_prefill;  // constant since the build
  const int64_t R = N + win_start;
  const int rho = v.paris_rho;
  // 1. the rotated group query
  if (tid < kHeadDim) {
    float acc = load_elem<DT>(q, qoff + tid);
    for (int g = 1; g < v.G; ++g) acc = __fadd_rn(acc, load_elem<DT>(q, qoff + (int64_t)g * kHeadDim + tid));
    qr[tid] = ((v.paris_sign[tid >> 6] >> (tid & 63)) & 1ull) ? -acc : acc;
  }
  if (tid < 8) levs[tid] = v.paris_lev[tid];
  for (int x = tid; x < 256; x += nth) hist[x] = 0;
  __syncthreads();
  for (int h = 1; h < kHeadDim; h <<= 1) {
    if (tid < kHeadDim / 2) {
      const int j = (tid / h) * 2 * h + (tid % h);
      const float a = qr[j], b = qr[j + h];
      qr[j] = __fadd_rn(a, b);
      qr[j + h] = __fsub_rn(a, b);
    }
    __syncthreads();
  }
  // 2. similarities of the 256 sign patterns of every subspace, then the
  //    rho best of each (a warp per subspace, ties to the lower pattern)
  for (int x = tid; x < kParisSub * 256; x += nth) {
    const int b = x >> 8, p = x & 255;
    float sacc = 0.f;
#pragma unroll
    for (int j = 0; j < kParisDim; ++j) {
      const float xq = qr[b * kParisDim + j];
      sacc = __fadd_rn(sacc, ((p >> j) & 1) ? -xq : xq);
    }
    sim[x] = sacc;
    vote[x] = 0;
  }
  __syncthreads();
  for (int b = wid; b < kParisSub; b += nth / 32) {
    for (int r = 0; r < rho; ++r) {
      float bs = -INFINITY;
      int bp = 256;
      for (int k = 0; k < 8; ++k) {
        const int p = lane + 32 * k;
        const float sp = sim[b * 256 + p];
        if (!vote[b * 256 + p] && (sp > bs || (sp == bs && p < bp))) {
          bs = sp;
          bp = p;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float os = __shfl_xor_sync(kFull, bs, o);
        const int op = __shfl_xor_sync(kFull, bp, o);
        if (os > bs || (os == bs && op < bp)) {
          bs = os;
          bp = op;
        }
      }
      if (lane == 0) vote[b * 256 + bp] = (uint8_t)(rho - r);
      __syncwarp();
    }
  }
  __syncthreads();
  const uint8_t *bk = v.pk_bucket + gs * v.pool_rows * kParisSub;
  auto row_of = [&](int64_t r) -> int64_t { return r < N ? r : v.n_cap + (r - N); };
  auto coarse = [&](int64_t r) -> int {
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(bk + row_of(r) * kParisSub));
    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
    int c = 0;
#pragma unroll
    for (int b = 0; b < kParisSub; ++b) c += vote[b * 256 + ((w4[b >> 2] >> (8 * (b & 3))) & 255u)];
    return c;
  };
  // 3. every region token's vote sum, kept as a byte in the step slot's
  //    scratch; their histogram (per warp, then summed); the cut score and
  //    how many ties it takes
  uint8_t *sc = v.pk_score + ((int64_t)(slot % kChunk) * v.S_all + gs) * v.pk_pitch;
  for (int x = tid; x < kScoreWarps * 256; x += nth) (&whist[0][0])[x] = 0;
  __syncthreads();
  {
    constexpr int kU = 8;  // tokens in flight per thread
    for (int64_t r0_ = (int64_t)tid; r0_ < R; r0_ += (int64_t)kU * nth) {
      int c[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t r = r0_ + (int64_t)u * nth;
        c[u] = r < R ? coarse(r) : -1;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c[u] >= 0) {
          sc[r0_ + (int64_t)u * nth] = (uint8_t)c[u];
          atomicAdd(&whist[wid][c[u]], 1);
        }
    }
  }
  __syncthreads();
  for (int x = tid; x < 256; x += nth) {
    int32_t tot = 0;
    for (int w = 0; w < kScoreWarps; ++w) tot += whist[w][x];
    hist[x] = tot;
  }
  __syncthreads();
  if (tid == 0) {
    const int nc = v.paris_n_cand;
    int cut = 0, need = 1 << 30, above = 0;
    if (R > nc) {
      for (int x = 255; x >= 0; --x) {
        if (above + hist[x] >= nc) {
          cut = x;
          need = nc - above;
          break;
        }
        above += hist[x];
      }
    }
    s_cut = cut;
    s_need = need;
  }
  __syncthreads();
  // 4. the candidates in token order: every token above the cut, the first
  //    `need` at it
  //    (a thread's range is a whole number of 16-byte words of the vote
  //    bytes, read one word at a time; the scratch row pitch is a multiple
  //    of 16, so a word past R stays inside the row)
  const int64_t per = ((R + nth - 1) / nth + 15) / 16 * 16;
  const int64_t r0 = min(R, (int64_t)tid * per), r1 = min(R, r0 + per);
  const int cut = s_cut, need = s_need;
  auto vote_byte = [](const uint4 &x, int b) -> int {
    const uint32_t wv = b < 8 ? (b < 4 ? x.x : x.y) : (b < 12 ? x.z : x.w);
    return (int)((wv >> (8 * (b & 3))) & 255u);
  };
  int32_t n_gt = 0, n_eq = 0;
  for (int64_t r = r0; r < r1; r += 16) {
    const uint4 x = *reinterpret_cast<const uint4 *>(sc + r);
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const int c = vote_byte(x, b);
      const bool in = r + b < r1;
      n_gt += in && c > cut;
      n_eq += in && c == cut;
    }
  }
  const int2 ex = block_scan_excl2(n_gt, n_eq, wt, &s_dummy, &s_nc);
  const int32_t take_eq = max(0, min(n_eq, need - ex.y));
  const int32_t c_ex = block_scan_excl(n_gt + take_eq, wt, &s_nc);
  {
    int32_t k = c_ex, eq_seen = 0;
    for (int64_t r = r0; r < r1; r += 16) {
      const uint4 x = *reinterpret_cast<const uint4 *>(sc + r);
#pragma unroll
      for (int b = 0; b < 16; ++b) {
        const int c = vote_byte(x, b);
        if (r + b < r1 && (c > cut || (c == cut && eq_seen++ < take_eq))) cand[k++] = (int32_t)(r + b);
      }
    }
  }
  __syncthreads();
  const int nc = min(s_nc, kParisMaxCand);
  // 5. rerank on the codes: est = sum_b w_b dot_b, dot_b = sum_j v_j qr_j
  for (int c = tid; c < nc; c += nth) {
    const int64_t row = gs * v.pool_rows + row_of(cand[c]);
    const uint4 bx = __ldg(reinterpret_cast<const uint4 *>(v.pk_bucket + row * kParisSub));
    const uint32_t bw[4] = {bx.x, bx.y, bx.z, bx.w};
    const uint4 *cp = reinterpret_cast<const uint4 *>(v.pk_code + row * 64);
    const float4 *wp = reinterpret_cast<const float4 *>(v.pk_w + row * kParisSub);
    float est = 0.f;
#pragma unroll
    for (int b4 = 0; b4 < 4; ++b4) {
      const uint4 cx = __ldg(cp + b4);
      const float4 wx = __ldg(wp + b4);
      const uint32_t cw[4] = {cx.x, cx.y, cx.z, cx.w};
      const float ww[4] = {wx.x, wx.y, wx.z, wx.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int b = 4 * b4 + e;
        const uint32_t bits = (bw[b >> 2] >> (8 * (b & 3))) & 255u;
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < kParisDim; ++j) {
          const float lv = levs[(cw[e] >> (4 * j)) & 15u];
          dot = __fmaf_rn(((bits >> j) & 1u) ? -lv : lv, qr[b * kParisDim + j], dot);
        }
        est = __fmaf_rn(ww[e], dot, est);
      }
    }
    key_s[c] = desc_key(est);
  }
  __syncthreads();
  // 6. the budget best candidates (every candidate is one token)
  auto keyof = [&](int c) -> uint32_t { return key_s[c]; };
  auto one = [&](int) -> int32_t { return 1; };
  radix_cut(nc, budget, keyof, one, whist, wt, &rc);
  const bool all = rc.all != 0;
  const uint32_t kstar = rc.prefix;
  const int32_t below = rc.below;
  const int cper = (nc + nth - 1) / nth;
  const int c0 = tid * cper, c1 = min(nc, c0 + cper);
  int32_t tl = 0;
  if (!all)
    for (int c = c0; c < c1; ++c) tl += key_s[c] == kstar;
  const int32_t tie_ex = block_scan_excl(tl, wt, nullptr);
  auto chosen = [&](int c, int32_t &run) -> bool {
    if (all) return true;
    const uint32_t key = key_s[c];
    if (key < kstar) return true;
    if (key == kstar) return below + (++run) <= budget;
    return false;
  };
  int32_t cnt = 0;
  {
    int32_t run = tie_ex;
    for (int c = c0; c < c1; ++c) cnt += chosen(c, run);
  }
  const int32_t o_ex = block_scan_excl(cnt, wt, &s_nsel);
  {
    int32_t run = tie_ex, k = o_ex;
    int32_t *sel_out = plan_sel(v, ps, gs), *tok_rows = plan_sel_rows(v, ps, gs);
    for (int c = c0; c < c1; ++c)
      if (chosen(c, run)) {
        const int32_t row = (int32_t)row_of(cand[c]);
        if (k < v.u_cap) sel_out[k] = row;
        if (k < v.sel_cap) tok_rows[k] = row;
        ++k;
      }
  }
  if (tid == 0) {
    *plan_nsel(v, ps, gs) = s_nsel;
    *plan_ntok(v, ps, gs) = s_nsel;
    atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)R);
    atomicAdd((unsigned long long *)&v.counters[kCntSelUnits], (unsigned long long)s_nsel);
    atomicAdd((unsigned long long *)&v.counters[kCntSelTokens], (unsigned long long)s_nsel);
    if (s_nsel > budget || s_nsel > v.sel_cap || s_nsel > v.u_cap || s_nc > kParisMaxCand)
      set_err(v.err, kErrInternal);
  }
}

// kScoreSplit CTAs of kScoreThreads per (seq, layer, kv head) and step. On a
// step without retrieval the first only records the step's descriptor for
// the attention (the plan in force and its token count). On a retrieval step
// every CTA scores its share of the units, s_u = qbar . c_u (qbar the fp32
// sum of the group's queries in head order; the dot a sequential fp32 FMA
// chain in index order, a thread per unit), and the last CTA of the slice to
// finish takes the budget selection and writes the plan.
constexpr int kScoreSplit = 8;

template <int DT>
__global__ void __launch_bounds__(kScoreThreads, 3) k_select(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const int tid = threadIdx.x, nth = blockDim.x;
  pdl_wait();  // the step's view and every earlier selection's plan are complete and visible
  pdl_trigger();
  const int4 view = v.aview[(int64_t)a.slot * v.n_lb + lb];
  int4 *desc = v.adesc + (int64_t)a.slot * v.S_all + gs;
  if (!(view.w & 1)) {
    // no retrieval: the plan in force stays; the attention's descriptor
    // carries its token count
    if (blockIdx.y == 0 && tid == 0) *desc = make_int4(view.x, view.y, view.z, *plan_ntok(v, view.z, gs));
    return;
  }
  const int U = view.w >> 1;
  const int64_t k = view.x - a.base_t;
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  __shared__ float qbar[kHeadDim];
  __shared__ int s_last;
  const int H = v.Hkv * v.G;
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * v.G) * kHeadDim;
  if (v.paris) {  // one CTA runs the token pipeline of the slice
    if (blockIdx.y != 0) return;
    if constexpr (DT == 1) select_paris<DT>(v, lb, gs, a.budget, view.z, a.slot, q, qoff, view.y);
    if (tid == 0) *desc = make_int4(view.x, view.y, view.z, *plan_ntok(v, view.z, gs));
    return;
  }
  if (v.pol_per_head) {  // one CTA scores and selects for every head of the slice
    if (blockIdx.y != 0) return;
    if (tid == 0) atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)U * v.G);
    select_heads<DT>(v, gs, U, a.budget, view.z, q, qoff);
    if (tid == 0) *desc = make_int4(view.x, view.y, view.z, *plan_ntok(v, view.z, gs));
    return;
  }
  if (tid < kHeadDim) {
    float acc = load_elem<DT>(q, qoff + tid);
    for (int g = 1; g < v.G; ++g) acc = __fadd_rn(acc, load_elem<DT>(q, qoff + (int64_t)g * kHeadDim + tid));
    qbar[tid] = acc;
  }
  __syncthreads();
  constexpr int nvec = kHeadDim * elem_bytes<DT>() / 16;  // 16-byte vectors per centroid row
  const uint4 *rows = (const uint4 *)((const char *)v.cent_op + gs * v.u_cap * kHeadDim * elem_bytes<DT>());
  for (int u = blockIdx.y * nth + tid; u < U; u += gridDim.y * nth) {
    uint4 cur[nvec];
#pragma unroll
    for (int j = 0; j < nvec; ++j) cur[j] = __ldg(rows + (int64_t)u * nvec + j);
    float sc = 0.f;
#pragma unroll
    for (int j = 0; j < nvec; ++j) {
      const uint32_t w[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
      if constexpr (DT == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sc = __fmaf_rn(qbar[j * 8 + 2 * e], __uint_as_float(w[e] << 16), sc);
          sc = __fmaf_rn(qbar[j * 8 + 2 * e + 1], __uint_as_float(w[e] & 0xffff0000u), sc);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc = __fmaf_rn(qbar[j * 4 + e], __uint_as_float(w[e]), sc);
      }
    }
    v.scores[gs * v.u_cap + u] = sc;
  }
  // the last CTA of the slice to finish selects
  __threadfence();
  __syncthreads();
  int32_t *cnt = v.sel_count + (int64_t)(a.slot & (kRing - 1)) * v.S_all + gs;
  if (tid == 0) s_last = atomicAdd(cnt, 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) {
    *cnt = 0;
    atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)U);
  }
  select_units(v, gs, U, a.budget, view.z, v.scores + gs * v.u_cap, false);
  if (tid == 0) *desc = make_int4(view.x, view.y, view.z, *plan_ntok(v, view.z, gs));
}

// The selections of a whole chunk of steps in one launch (chunk selection):
// a CTA per (slice, step of the chunk). Given the boundary kernel's views,
// the retrievals of different steps are independent problems (each scores
// the units present at its step and writes its own plan slot), so they run
// side by side; a CTA of a step without retrieval leaves at once. Scores and
// selection as in k_select, the scores of a step in its own slot.
template <int DT>
__global__ void __launch_bounds__(kScoreThreads, 3) k_select_chunk(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const int tid = threadIdx.x, nth = blockDim.x;
  const int slot = a.slot + blockIdx.y;
  pdl_wait();  // the chunk's views are complete and visible
  pdl_trigger();
  const int4 view = v.aview[(int64_t)slot * v.n_lb + lb];
  if (!(view.w & 1)) return;
  const int U = view.w >> 1;
  const int64_t k = view.x - a.base_t;
  const void *q = (const char *)a.q + k * a.stride_q * elem_bytes<DT>();
  __shared__ float qbar[kHeadDim];
  const int H = v.Hkv * v.G;
  const int64_t qoff = (((int64_t)b * a.nl + li) * H + (int64_t)h * v.G) * kHeadDim;
  if (v.paris) {
    if constexpr (DT == 1) select_paris<DT>(v, lb, gs, a.budget, view.z, slot, q, qoff, view.y);
    return;
  }
  if (v.pol_per_head) {
    if (tid == 0) atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)U * v.G);
    select_heads<DT>(v, gs, U, a.budget, view.z, q, qoff);
    return;
  }
  if (tid < kHeadDim) {
    float acc = load_elem<DT>(q, qoff + tid);
    for (int g = 1; g < v.G; ++g) acc = __fadd_rn(acc, load_elem<DT>(q, qoff + (int64_t)g * kHeadDim + tid));
    qbar[tid] = acc;
  }
  __syncthreads();
  extern __shared__ __align__(16) uint32_t sel_smem[];
  const bool in_smem = U <= kSelSmemUnits;
  float *scg = v.scores + ((int64_t)(slot % kChunk) * v.S_all + gs) * v.u_cap;
  constexpr int nvec = kHeadDim * elem_bytes<DT>() / 16;
  const uint4 *rows = (const uint4 *)((const char *)v.cent_op + gs * v.u_cap * kHeadDim * elem_bytes<DT>());
  for (int u = tid; u < U; u += nth) {
    uint4 cur[nvec];
#pragma unroll
    for (int j = 0; j < nvec; ++j) cur[j] = __ldg(rows + (int64_t)u * nvec + j);
    float sc = 0.f;
#pragma unroll
    for (int j = 0; j < nvec; ++j) {
      const uint32_t w[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
      if constexpr (DT == 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sc = __fmaf_rn(qbar[j * 8 + 2 * e], __uint_as_float(w[e] << 16), sc);
          sc = __fmaf_rn(qbar[j * 8 + 2 * e + 1], __uint_as_float(w[e] & 0xffff0000u), sc);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc = __fmaf_rn(qbar[j * 4 + e], __uint_as_float(w[e]), sc);
      }
    }
    if (in_smem) sel_smem[u] = desc_key(sc);
    else scg[u] = sc;
  }
  if (tid == 0) atomicAdd((unsigned long long *)&v.counters[kCntScoreUnits], (unsigned long long)U);
  __syncthreads();
  select_units(v, gs, U, a.budget, view.z, scg, in_smem);
}

// ---------------------------------------------------------------- offload gather

// On a retrieval step, the selected rows go from the pinned host pool to this
// plan slot's HBM staging rows over UVA. A warp takes one copy piece of the
// selection (a contiguous run of <= 64 pool rows, from the selection's piece
// list) and moves its K and V rows in 16-byte vectors, eight loads in flight
// per lane, so the host link sees long contiguous reads.
constexpr int kGatherVec = 8;

template <int DT>
__global__ void __launch_bounds__(256) k_gather_offload(CtxView v, StepArgs a) {
  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  pdl_wait();
  pdl_trigger();
  const int4 view = v.aview[(int64_t)a.slot * v.n_lb + lb];
  if (!(view.w & 1)) return;
  const int ps = view.z;
  const int nt = *plan_ntok(v, ps, gs);
  const int nsc = (nt + kAttnChunk - 1) / kAttnChunk;
  if (nt == 0 || nsc > v.max_chunks) return;
  const int npieces = v.chunk_piece[gs * (int64_t)(v.max_chunks + 1) + nsc];
  const int4 *pieces = v.pieces + gs * (int64_t)v.max_pieces;
  constexpr int rb = kHeadDim * elem_bytes<DT>();
  constexpr int per_row = rb / 16;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.y * (blockDim.x / 32);
  const uint4 *src_k = (const uint4 *)((const char *)v.pool_k + gs * v.pool_rows * rb);
  const uint4 *src_v = (const uint4 *)((const char *)v.pool_v + gs * v.pool_rows * rb);
  uint4 *dst_k = (uint4 *)((char *)v.stage_k + ((int64_t)ps * v.S_all + gs) * v.bud_cap * rb);
  uint4 *dst_v = (uint4 *)((char *)v.stage_v + ((int64_t)ps * v.S_all + gs) * v.bud_cap * rb);
  for (int p = blockIdx.y * (blockDim.x / 32) + threadIdx.x / 32; p < npieces; p += warps) {
    const int4 pc = pieces[p];  // (first pool row, first selected token, rows)
    const int nvec = pc.z * per_row;
    const uint4 *sk = src_k + (int64_t)pc.x * per_row, *sv = src_v + (int64_t)pc.x * per_row;
    uint4 *dk = dst_k + (int64_t)pc.y * per_row, *dv = dst_v + (int64_t)pc.y * per_row;
    for (int x0 = 0; x0 < nvec; x0 += 32 * kGatherVec) {
      uint4 rk[kGatherVec], rv[kGatherVec];
#pragma unroll
      for (int e = 0; e < kGatherVec; ++e) {
        const int x = x0 + e * 32 + lane;
        if (x < nvec) {
          rk[e] = __ldcg(sk + x);
          rv[e] = __ldcg(sv + x);
        }
      }
#pragma unroll
      for (int e = 0; e < kGatherVec; ++e) {
        const int x = x0 + e * 32 + lane;
        if (x < nvec) {
          dk[x] = rk[e];
          dv[x] = rv[e];
        }
      }
    }
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    atomicAdd((unsigned long long *)&v.counters[kCntGatherRows], (unsigned long long)nt);
}

// ---------------------------------------------------------------- attention

// Two variants of the per-chunk arithmetic. The tensor-core one (bf16 rows,
// 4 or 8 query heads per KV head) runs 4 warps of 16 rows each; the scalar
// one (fp32 rows, or 1-2 query heads) 8 warps of 8 rows.
template <int DT, int G>
constexpr bool attn_tc() { return DT == 1 && (G == 4 || G == 8); }
template <int DT, int G>
constexpr int attn_warps() { return attn_tc<DT, G>() ? 4 : 8; }
template <int DT, int G>
constexpr int attn_threads() { return 32 * attn_warps<DT, G>(); }
constexpr int kRowsPerWarp = 8;  // scalar variant: rows of each chunk per warp
constexpr int kStages = 3;       // scalar variant: chunk stages per CTA
constexpr int kTcStages = 2;     // tensor-core variant: stages of each warp's ring
template <int DT, int G>
constexpr int attn_min_blocks() { return attn_tc<DT, G>() ? 3 : 2; }
constexpr int kPreChunks = 8;  // chunks whose copy plan a CTA prefetches
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // 2 s

union F2U {
  float2 f;
  unsigned long long u;
};
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  F2U x{a}, y{b}, z{c}, r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.u) : "l"(x.u), "l"(y.u), "l"(z.u));
  return r.f;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  F2U x{a}, y{b}, r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.u) : "l"(x.u), "l"(y.u));
  return r.f;
}

// d += A (16 x 16, row-major) * B (16 x 8, column-major), bf16 operands, fp32
// accumulation. Lane (g = lane / 4, t = lane % 4) holds A rows g and g + 8,
// columns 2t, 2t + 1, 2t + 8, 2t + 9 (a0: row g, a1: row g + 8, a2/a3 the
// same rows at columns + 8), B rows 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1)
// of column g, and D rows g (d0, d1) and g + 8 (d2, d3) at columns 2t, 2t + 1.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The bf16 parts of (x0, x1) (lo = false) or of their residuals x - bf16(x)
// (lo = true), packed low = x0: a value's two parts sum to it within 2^-17
// relative.
__device__ __forceinline__ uint32_t bf16_pair(float x0, float x1, bool lo) {
  // packed conversions: two values per instruction
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 r = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  const __nv_bfloat162 w = lo ? r : h;
  return *reinterpret_cast<const uint32_t *>(&w);
}
__device__ __forceinline__ uint32_t prmt(uint32_t x, uint32_t y, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(sel));
  return r;
}
// 16-byte asynchronous global -> shared copy; n < 16 source bytes are
// read and the rest zero-filled (n = 0: nothing is read).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t word(const uint4 &x, int j) {
  return j == 0 ? x.x : j == 1 ? x.y : j == 2 ? x.z : x.w;
}

// The 8 consecutive elements [8k, 8k + 8) of a row owned by lane k of a
// 16-lane group, as 4 float pairs (the group reads the row contiguously).
template <int DT>
__device__ __forceinline__ void row8(const unsigned char *row, int k, float2 (&o)[4]) {
  if constexpr (DT == 1) {
    const uint4 a = *(const uint4 *)(row + 16 * k);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int p = 0; p < 4; ++p)
      o[p] = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
  } else {
    const float4 a = *(const float4 *)(row + 32 * k);
    const float4 b = *(const float4 *)(row + 32 * k + 16);
    o[0] = make_float2(a.x, a.y); o[1] = make_float2(a.z, a.w);
    o[2] = make_float2(b.x, b.y); o[3] = make_float2(b.z, b.w);
  }
}

// Keep-or-send halving step of a butterfly reduce-scatter: lanes with `up`
// keep the upper half of x[0..2n), the others the lower half.
template <int N>
__device__ __forceinline__ void halve(float *x, bool up, int mask) {
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const float send = up ? x[j] : x[j + N], keep = up ? x[j + N] : x[j];
    x[j] = keep + __shfl_xor_sync(kFull, send, mask);
  }
}

// Reduce the per-lane partial dot products of the G heads of one row over
// its 16-lane group; on return lane k holds the full score of head
// head_of_lane<G>(k).
template <int G>
__device__ __forceinline__ float reduce_heads(float (&x)[G], int lane) {
  const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  if constexpr (G == 8) {
    halve<4>(x, b3, 8);
    halve<2>(x, b2, 4);
    halve<1>(x, b1, 2);
    return x[0] + __shfl_xor_sync(kFull, x[0], 1);
  } else if constexpr (G == 4) {
    halve<2>(x, b3, 8);
    halve<1>(x, b2, 4);
    float r = x[0] + __shfl_xor_sync(kFull, x[0], 2);
    return r + __shfl_xor_sync(kFull, r, 1);
  } else if constexpr (G == 2) {
    halve<1>(x, b3, 8);
    float r = x[0] + __shfl_xor_sync(kFull, x[0], 4);
    r += __shfl_xor_sync(kFull, r, 2);
    return r + __shfl_xor_sync(kFull, r, 1);
  } else {
    float r = x[0];
    r += __shfl_xor_sync(kFull, r, 8);
    r += __shfl_xor_sync(kFull, r, 4);
    r += __shfl_xor_sync(kFull, r, 2);
    return r + __shfl_xor_sync(kFull, r, 1);
  }
}

// The same reduction when lane k holds its partials in the permuted head
// order x[j] = head (head_of_lane(k) ^ j): the half a lane keeps is then
// always x[0..N) and the half it sends x[N..2N), so no selects are needed.
template <int G>
__device__ __forceinline__ float reduce_heads_perm(float (&x)[G]) {
  if constexpr (G >= 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] += __shfl_xor_sync(kFull, x[j + 4], 8);
  }
  if constexpr (G >= 4) {
    constexpr int m = G >= 8 ? 4 : 8;
#pragma unroll
    for (int j = 0; j < 2; ++j) x[j] += __shfl_xor_sync(kFull, x[j + 2], m);
  }
  if constexpr (G >= 2) {
    constexpr int m = G >= 8 ? 2 : (G >= 4 ? 4 : 8);
    x[0] += __shfl_xor_sync(kFull, x[1], m);
  }
  float r = x[0];
#pragma unroll
  for (int m = 16 / (2 * G); m >= 1; m >>= 1) r += __shfl_xor_sync(kFull, r, m);
  return r;
}

template <int G>
__device__ __forceinline__ int head_of_lane(int k) {
  if constexpr (G == 8) return ((k >> 3) & 1) * 4 + ((k >> 2) & 1) * 2 + ((k >> 1) & 1);
  else if constexpr (G == 4) return ((k >> 3) & 1) * 2 + ((k >> 2) & 1);
  else if constexpr (G == 2) return (k >> 3) & 1;
  else return 0;
}

template <int DT>
constexpr int stage_bytes() { return 2 * kAttnChunk * kHeadDim * elem_bytes<DT>(); }
// dynamic shared memory: the scalar variant's chunk ring, or the tensor-core
// variant's per-warp rings (each stage 16 rows of K and V)
template <int DT, int G>
constexpr size_t attn_smem() {
  return attn_tc<DT, G>() ? (size_t)attn_warps<DT, G>() * kTcStages * 2 * 16 * kHeadDim * elem_bytes<DT>()
                          : (size_t)kStages * stage_bytes<DT>();
}


// Split-K attention. CTA split of the nsplit CTAs of a (seq, layer, kv head)
// streams chunks [split * cpc, ...) of the slice's token list (selected rows,
// then the local buffer) through a 3-stage ring of shared-memory buffers
// filled by bulk copies. Per chunk each warp owns a block of rows: it scores
// them, updates its online softmax and adds p * V into its accumulators.
//  - tensor-core variant (bf16 rows, G = 4 or 8): 4 warps of 16 rows. Scores
//    and p * V are 16x8x16 bf16 products with fp32 accumulation; the queries
//    and the softmax weights enter as a bf16 high part plus a bf16 residual
//    (two columns per head), so both keep fp32 accuracy.
//  - scalar variant: 8 warps of 8 rows; pass 1 scores them (16 lanes per row,
//    2 rows per instruction), pass 2 adds p * V with packed fp32 FMAs.
// The CTAs' partial softmax states go to a per-step-slot scratch and the last
// CTA to finish combines them, so no CTA waits for another.
template <int DT, int G>
__global__ void __launch_bounds__(attn_threads<DT, G>(), attn_min_blocks<DT, G>())
    k_attn(CtxView v, StepArgs a, int cpc) {
  constexpr bool TC = attn_tc<DT, G>();
  constexpr int NW = attn_warps<DT, G>();
  constexpr int NTH = 32 * NW;
  constexpr int RB = kHeadDim * elem_bytes<DT>();
  constexpr int SB = stage_bytes<DT>();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bar[kStages];
  __shared__ float qs[G][kHeadDim];
  __shared__ __align__(16) float S[kAttnChunk][G];
  __shared__ float wm[NW][G], wl[NW][G];
  __shared__ __align__(16) int4 pcs[kPreChunks][kAttnChunk];  // copy plans, a ring of slots
  __shared__ int pcn[kPreChunks];
  __shared__ __align__(8) uint64_t pbar[kPreChunks];  // a plan slot's bulk load landed
  __shared__ int done_cnt[kStages];  // warps finished with the chunk in each stage
  // this CTA's partial: acc [G][d], then the maxima [G] and sums [G]
  __shared__ float part[G * kHeadDim + 2 * G];
  __shared__ int4 s_view;  // (t, win_start, plan slot, 0) of this step
  __shared__ int s_nt, s_ns, s_ok, s_last;

  const int per_l = v.B * v.Hkv;
  const int li = blockIdx.x / per_l, rem = blockIdx.x % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int l = a.l0 + li;
  const int64_t lb = (int64_t)l * v.B + b;
  const int64_t gs = lb * v.Hkv + h;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int grp = lane >> 4, kk = lane & 15;
  const int H = v.Hkv * G;
  const int nsplit = gridDim.y, split = blockIdx.y;
  const int c_begin = split * cpc;
  pdl_wait();
  pdl_trigger();

  // the step's view (window and plan slot) with the queries, then the plan:
  // its counts and the copy plan of this CTA's first chunks
  if (tid == 0) {
    s_view = v.aview[(int64_t)a.slot * v.n_lb + lb];
    s_ok = 1;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar[i], 1);
      done_cnt[i] = 0;
    }
    for (int i = 0; i < kPreChunks; ++i) mbar_init(&pbar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int x = tid; x < G * kHeadDim; x += NTH)
    qs[x / kHeadDim][x % kHeadDim] =
        v.q_attn[(((int64_t)a.slot * v.n_lb + lb) * H + (int64_t)h * G) * kHeadDim + x];
  __syncthreads();
  const int ps = s_view.z;
  // tensor-core variant: the token rows of this warp's first chunks go out
  // with the plan's counts (entries past the selected tokens are not used)
  int32_t pre_rows[kTcStages][8];
  if constexpr (TC) {
    const int32_t *tr = v.offload ? nullptr : plan_sel_rows(v, ps, gs);
#pragma unroll
    for (int i = 0; i < kTcStages; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int f = (c_begin + i) * kAttnChunk + 16 * wid + (lane >> 4) + 2 * k;
        pre_rows[i][k] = (tr && f < v.sel_cap) ? tr[f] : 0;
      }
  }
  const int4 *plan_pcs = plan_chunk_pieces(v, ps, gs);
  const int32_t *plan_pcn = plan_chunk_count(v, ps, gs);
  if (tid == 0) {
    s_nt = *plan_ntok(v, ps, gs);
    s_ns = *plan_nsel(v, ps, gs);
  }
  if (!TC && !v.offload)  // (the tensor-core variant reads the plan's token rows instead)
    for (int x = tid; x < kPreChunks * kAttnChunk; x += NTH) {
      const int i = x / kAttnChunk, c = c_begin + i;
      if (i < cpc && c < v.max_chunks) {
        pcs[i][x % kAttnChunk] = plan_pcs[c * kAttnChunk + x % kAttnChunk];
        if (x % kAttnChunk == 0) pcn[i] = plan_pcn[c];
      }
    }
  __syncthreads();
  const int t_cur = s_view.x, ws = s_view.y;
  const int64_t k = t_cur - a.base_t;
  const int nt = s_nt;
  const int total = nt + (t_cur - ws + 1);
  const int nch = (total + kAttnChunk - 1) / kAttnChunk;
  const int n_my = max(0, min(cpc, nch - c_begin));

  const unsigned char *selk, *selv;
  if (!v.offload) {
    selk = (const unsigned char *)v.pool_k + gs * v.pool_rows * RB;
    selv = (const unsigned char *)v.pool_v + gs * v.pool_rows * RB;
  } else {
    selk = (const unsigned char *)v.stage_k + ((int64_t)ps * v.S_all + gs) * v.bud_cap * RB;
    selv = (const unsigned char *)v.stage_v + ((int64_t)ps * v.S_all + gs) * v.bud_cap * RB;
  }
  // one warp fills stage (i % kStages) with chunk c_begin + i
  auto issue = [&](int i) {
    unsigned char *Ks = smem + (i % kStages) * SB;
    unsigned char *Vs = Ks + SB / 2;
    uint64_t *br = &bar[i % kStages];
    const int c = c_begin + i, f0 = c * kAttnChunk;
    const int nrow = min(kAttnChunk, total - f0);
    int np = 0, sel_direct = 0;
    const int4 *pieces = nullptr;
    const int slot = i % kPreChunks;
    if (f0 < nt) {
      if (!v.offload) {
        // chunks past the first kPreChunks: their plan was bulk-loaded into
        // this slot when the chunk kPreChunks earlier was issued
        if (i >= kPreChunks && !mbar_wait_bounded(&pbar[slot], ((i / kPreChunks) - 1) & 1, kWaitLimitNs))
          s_ok = 0;
        pieces = pcs[slot];
        np = i < kPreChunks ? pcn[slot] : pcs[slot][0].w;
      } else {
        sel_direct = min(f0 + kAttnChunk, nt) - f0;
      }
    }
    uint32_t bytes = 0;
    for (int p = lane; p < np; p += 32) bytes += 2u * (uint32_t)pieces[p].z * RB;
    const int win0 = max(f0, nt), win1 = f0 + nrow;
    if (lane == 0) bytes += 2u * (uint32_t)(max(win1 - win0, 0) + sel_direct) * RB;
#pragma unroll
    for (int o = 16; o; o >>= 1) bytes += __shfl_xor_sync(kFull, bytes, o);
    if (lane == 0) mbar_arrive_expect_tx(br, bytes);
    __syncwarp();
    for (int p = lane; p < np; p += 32) {
      const int4 pc = pieces[p];
      const int dr = pc.y - f0;
      bulk_g2s(Ks + dr * RB, selk + (int64_t)pc.x * RB, (uint32_t)pc.z * RB, br);
      bulk_g2s(Vs + dr * RB, selv + (int64_t)pc.x * RB, (uint32_t)pc.z * RB, br);
    }
    if (lane == 0) {
      if (sel_direct > 0) {
        bulk_g2s(Ks, selk + (int64_t)f0 * RB, (uint32_t)sel_direct * RB, br);
        bulk_g2s(Vs, selv + (int64_t)f0 * RB, (uint32_t)sel_direct * RB, br);
      }
      if (win1 > win0) {
        const int64_t r0 = gs * v.dec_rows + ws + (win0 - nt);
        bulk_g2s(Ks + (win0 - f0) * RB, (const unsigned char *)v.dec_k + r0 * RB,
                 (uint32_t)(win1 - win0) * RB, br);
        bulk_g2s(Vs + (win0 - f0) * RB, (const unsigned char *)v.dec_v + r0 * RB,
                 (uint32_t)(win1 - win0) * RB, br);
      }
    }
    // the slot's plan is consumed: bring in the plan of chunk i + kPreChunks
    // (1 KB, its piece count in the first piece) for that chunk's refill
    const int i2 = i + kPreChunks, c2 = c_begin + i2;
    if (!v.offload && i2 < n_my && c2 * kAttnChunk < nt && c2 < v.max_chunks) {
      __syncwarp();
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&pbar[slot], kAttnChunk * sizeof(int4));
        bulk_g2s(pcs[slot], plan_pcs + (int64_t)c2 * kAttnChunk, kAttnChunk * sizeof(int4), &pbar[slot]);
      }
    }
  };
  if (!TC && wid < min(n_my, kStages)) issue(wid);  // the first stages, one warp each

  auto wait_stage = [&](int i) {
    if (!mbar_wait_bounded(&bar[i % kStages], (i / kStages) & 1, kWaitLimitNs)) {
      // record the timeout, then give the copies one more bounded wait so
      // that none is still writing a buffer this block reuses
      s_ok = 0;
      mbar_wait_bounded(&bar[i % kStages], (i / kStages) & 1, kWaitLimitNs);
    }
  };
  // this warp is done with stage i; the last warp to finish refills it with
  // chunk i + kStages (no block-wide barrier: warps run ahead freely). The
  // warp's reads of the stage have returned (their values fed the arithmetic
  // before), and the refill orders itself after them with the proxy fence
  // below, so the count needs no memory fence.
  auto release_stage = [&](int i) {
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      last = atomicAdd(&done_cnt[i % kStages], 1) == NW - 1;
      if (last) done_cnt[i % kStages] = 0;
    }
    last = __shfl_sync(kFull, last, 0);
    if (last && i + kStages < n_my) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(i + kStages);
    }
  };
  // after the loop the pipeline buffers are free: the warp accumulators go there
  float(*wacc)[G][kHeadDim] = reinterpret_cast<float(*)[G][kHeadDim]>(smem);
  static_assert(NW * G * kHeadDim * sizeof(float) <= attn_smem<DT, G>(), "");

  if constexpr (TC) {
    // Column n of product nt_ (NT = G / 4 products per 16-row block) carries
    // head (G == 8 ? n : n % 4): its bf16 high part for nt_ == 0 (G == 8) or
    // n < 4 (G == 4), else the bf16 residual. Lane (g, t) ends with D columns
    // 2t, 2t + 1, i.e. heads hb and hb + 1.
    constexpr int NT = G / 4;
    const int gq = lane >> 2, tq = lane & 3;
    const int hb = G == 8 ? 2 * tq : 2 * (tq & 1);
    auto col_head = [](int n) { return G == 8 ? n : (n & 3); };
    auto col_lo = [](int nt, int n) { return G == 8 ? nt == 1 : n >= 4; };
    // B operand of the scores: k-steps 2P and 2P + 1 take dims
    // [32P + 8t, 32P + 8t + 8) (the same order as the K rows' A operand)
    uint32_t qb[4][NT][4];
#pragma unroll
    for (int P = 0; P < 4; ++P)
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_) {
        const float *qh = qs[col_head(gq)] + 32 * P + 8 * tq;
#pragma unroll
        for (int w = 0; w < 4; ++w) qb[P][nt_][w] = bf16_pair(qh[2 * w], qh[2 * w + 1], col_lo(nt_, gq));
      }
    float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};  // heads hb, hb + 1
    float o[NT][8][4];
#pragma unroll
    for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt_][m][e] = 0.f;

    const int r0 = 16 * wid;  // this warp's 16 rows of every chunk
    // This warp's ring: kTcStages stages of its 16 rows (K rows, then V rows),
    // filled by 16-byte asynchronous copies that the warp issues itself, so
    // no warp waits for another. Lane (rh = lane / 16, seg = lane % 16)
    // copies bytes [16 seg, 16 seg + 16) of rows rh, rh + 2, ..., rh + 14.
    constexpr int WB = 16 * RB;
    unsigned char *ring = smem + wid * kTcStages * 2 * WB;
    const int rh = lane >> 4, seg = lane & 15;
    const int32_t *tok_rows = v.offload ? nullptr : plan_sel_rows(v, ps, gs);
    const unsigned char *deck = (const unsigned char *)v.dec_k + gs * v.dec_rows * RB;
    const unsigned char *decv = (const unsigned char *)v.dec_v + gs * v.dec_rows * RB;
    // the pool rows of this lane's rows of chunk i (loaded a chunk ahead of
    // their copies; entries past the selected tokens are not used)
    auto fetch_rows = [&](int i, int32_t (&x)[8]) {
      const int f0 = (c_begin + i) * kAttnChunk + r0 + rh;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int f = f0 + 2 * k;
        x[k] = (tok_rows && i < n_my && f < nt && f < v.sel_cap) ? tok_rows[f] : 0;
      }
    };
    auto copy_rows = [&](int i, const int32_t (&x)[8]) {
      unsigned char *Kd = ring + (i % kTcStages) * 2 * WB;
      if (i < n_my) {
        const int f0 = (c_begin + i) * kAttnChunk + r0 + rh;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int f = f0 + 2 * k;
          // the source row: on the HBM pool every row is a pool row of the
          // slice (a selected token's from the plan, a local-buffer token's at
          // max_prefill + its position); offloaded, selected rows are staging
          // rows and local-buffer rows decode rows
          const unsigned char *ks = selk, *vs = selv;
          int64_t row = 0;
          uint32_t n = 16;
          if (f < nt) {
            row = tok_rows ? x[k] : f;
          } else if (f < total) {
            row = ws + f - nt;
            if (tok_rows) row += v.n_cap;
            else { ks = deck; vs = decv; }
          } else {
            n = 0;  // past the slice's last token: zero fill
          }
          ks += row * RB;
          vs += row * RB;
          const int r = rh + 2 * k;
          cp_async16(Kd + r * RB + 16 * seg, ks + 16 * seg, n);
          cp_async16(Kd + WB + r * RB + 16 * seg, vs + 16 * seg, n);
        }
      }
      cp_async_commit();  // (an empty group past this CTA's chunks)
    };
#pragma unroll
    for (int i = 0; i < kTcStages; ++i) copy_rows(i, pre_rows[i]);
    int32_t xn[8];
    fetch_rows(kTcStages, xn);
    for (int i = 0; i < n_my; ++i) {
      const unsigned char *Kw = ring + (i % kTcStages) * 2 * WB;
      const unsigned char *Vw = Kw + WB;
      cp_async_wait<kTcStages - 1>();  // this lane's copies of chunk i have landed
      __syncwarp();                  // and so have the other lanes'
      const int nrow = min(kAttnChunk, total - (c_begin + i) * kAttnChunk);
      const bool full = r0 + 16 <= nrow;  // (warp-uniform)
      // scores of rows g and g + 8, two accumulation chains
      float sc[NT][2][4];
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt_][0][e] = sc[nt_][1][e] = 0.f;
      const unsigned char *kr = Kw + gq * RB + 16 * tq;
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const uint4 x = *(const uint4 *)(kr + 64 * P);
        const uint4 y = *(const uint4 *)(kr + 8 * RB + 64 * P);
#pragma unroll
        for (int nt_ = 0; nt_ < NT; ++nt_) {
          mma_bf16(sc[nt_][0], x.x, y.x, x.y, y.y, qb[P][nt_][0], qb[P][nt_][1]);
          mma_bf16(sc[nt_][1], x.z, y.z, x.w, y.w, qb[P][nt_][2], qb[P][nt_][3]);
        }
      }
      // s[0], s[1]: row g, heads hb, hb + 1; s[2], s[3]: row g + 8
      float s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[e] = sc[0][0][e] + sc[0][1][e];
        if constexpr (NT == 2) s[e] += sc[1][0][e] + sc[1][1][e];
        else s[e] += __shfl_xor_sync(kFull, s[e], 2);  // high part + residual
      }
      if (!full) {  // rows past the chunk's end (a slice's last chunk) score -inf
        if (r0 + gq >= nrow) s[0] = s[1] = -INFINITY;
        if (r0 + gq + 8 >= nrow) s[2] = s[3] = -INFINITY;
      }
      // online softmax over the warp's rows; rescale only when a maximum moves
      float c[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(s[e], s[e + 2]);
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, msk));
        const float mn = fmaxf(mr[e], mx);
        c[e] = (mr[e] == -INFINITY) ? 0.f : exp2f(mr[e] - mn);
        mr[e] = mn;
      }
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = (s[e] == -INFINITY) ? 0.f : exp2f(s[e] - mr[e & 1]);
#pragma unroll
      for (int e = 0; e < 2; ++e) lr[e] = lr[e] * c[e] + p[e] + p[e + 2];
      if (__any_sync(kFull, c[0] != 1.f || c[1] != 1.f)) {
#pragma unroll
        for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
          for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt_][m][e] *= c[e & 1];
      }
      // p^T as the B operand of p * V (rows = tokens, columns as above),
      // through the warp's rows of S
      if (G == 8 || tq < 2) {
        *(float2 *)&S[r0 + gq][hb] = make_float2(p[0], p[1]);
        *(float2 *)&S[r0 + gq + 8][hb] = make_float2(p[2], p[3]);
      }
      __syncwarp();
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_) {
        const int h = col_head(gq);
        const bool lo = col_lo(nt_, gq);
        pb[nt_][0] = bf16_pair(S[r0 + 2 * tq][h], S[r0 + 2 * tq + 1][h], lo);
        pb[nt_][1] = bf16_pair(S[r0 + 2 * tq + 8][h], S[r0 + 2 * tq + 9][h], lo);
      }
      // p * V: product m = 4hf + j has output rows dim 64hf + 8g + 2j (row g)
      // and that dim + 1 (row g + 8); lane (g, t) reads tokens 2t, 2t + 1,
      // 2t + 8, 2t + 9 at dims [64hf + 8g, + 8) and pairs them up by token
      // (rows past the slice's end were zero-filled)
      const unsigned char *vr = Vw + (2 * tq) * RB + 16 * gq;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const uint4 v0 = *(const uint4 *)(vr + 128 * hf);
        const uint4 v1 = *(const uint4 *)(vr + RB + 128 * hf);
        const uint4 v2 = *(const uint4 *)(vr + 8 * RB + 128 * hf);
        const uint4 v3 = *(const uint4 *)(vr + 9 * RB + 128 * hf);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w0 = word(v0, j), w1 = word(v1, j), w2 = word(v2, j), w3 = word(v3, j);
          const uint32_t a0 = prmt(w0, w1, 0x5410u), a1 = prmt(w0, w1, 0x7632u);
          const uint32_t a2 = prmt(w2, w3, 0x5410u), a3 = prmt(w2, w3, 0x7632u);
#pragma unroll
          for (int nt_ = 0; nt_ < NT; ++nt_)
            mma_bf16(o[nt_][4 * hf + j], a0, a1, a2, a3, pb[nt_][0], pb[nt_][1]);
        }
      }
      // every lane's reads of this stage (and of S) are done: refill the
      // stage with chunk i + kTcStages, fetch the rows of the chunk after it
      __syncwarp();
      copy_rows(i + kTcStages, xn);
      fetch_rows(i + kTcStages + 1, xn);
    }
    cp_async_wait<0>();  // (only empty groups can remain)
    __syncthreads();
    // the warp's result: high part + residual, then heads hb, hb + 1 at dims
    // 64hf + 8g + [0, 8) from the lanes that hold the high parts
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (NT == 2) o[0][m][e] += o[NT - 1][m][e];
        else o[0][m][e] += __shfl_xor_sync(kFull, o[0][m][e], 2);
      }
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) lr[e] += __shfl_xor_sync(kFull, lr[e], msk);
    if (G == 8 || tq < 2) {
      if (gq == 0) {
        wm[wid][hb] = mr[0];
        wm[wid][hb + 1] = mr[1];
        wl[wid][hb] = lr[0];
        wl[wid][hb + 1] = lr[1];
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float *dst = &wacc[wid][hb + e][64 * hf + 8 * gq];
          *(float4 *)dst = make_float4(o[0][4 * hf][e], o[0][4 * hf][e + 2], o[0][4 * hf + 1][e],
                                       o[0][4 * hf + 1][e + 2]);
          *(float4 *)(dst + 4) = make_float4(o[0][4 * hf + 2][e], o[0][4 * hf + 2][e + 2],
                                             o[0][4 * hf + 3][e], o[0][4 * hf + 3][e + 2]);
        }
    }
  } else {
    const int hl = head_of_lane<G>(kk);  // head whose score this lane ends with
    // this lane's query slices in the permuted head order hl ^ j (see
    // reduce_heads_perm)
    float2 q2[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int p = 0; p < 4; ++p)
        q2[j][p] = make_float2(qs[hl ^ j][8 * kk + 2 * p], qs[hl ^ j][8 * kk + 2 * p + 1]);
    float m_run[G];
#pragma unroll
    for (int g = 0; g < G; ++g) m_run[g] = -INFINITY;
    float m_own = -INFINITY, l_own = 0.f;  // running max and sum of head lane % G
    float2 acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int p = 0; p < 4; ++p) acc[g][p] = make_float2(0.f, 0.f);

    const int r0 = wid * kRowsPerWarp;
    for (int i = 0; i < n_my; ++i) {
      const unsigned char *Ks = smem + (i % kStages) * SB;
      const unsigned char *Vs = Ks + SB / 2;
      wait_stage(i);
      const int nrow = min(kAttnChunk, total - (c_begin + i) * kAttnChunk);
      // pass 1: scores of this warp's 8 rows, 2 rows per instruction (rows past
      // the chunk's end, in a slice's last chunk only, score -inf)
      const bool full = r0 + kRowsPerWarp <= nrow;  // (warp-uniform)
      auto pass1 = [&](auto check) {
#pragma unroll
        for (int it = 0; it < kRowsPerWarp / 2; ++it) {
          const int r = r0 + it * 2 + grp;
          float2 kv[4];
          row8<DT>(Ks + r * RB, kk, kv);
          float part[G];
#pragma unroll
          for (int j = 0; j < G; ++j) {
            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < 4; ++p) s2 = ffma2(q2[j][p], kv[p], s2);
            part[j] = s2.x + s2.y;
          }
          float s = reduce_heads_perm<G>(part);
          if (decltype(check)::value && r >= nrow) s = -INFINITY;
          if ((kk & (16 / G - 1)) == 0) S[r][hl] = s;
        }
      };
      if (full) pass1(std::false_type{});
      else pass1(std::true_type{});
      __syncwarp();
      // chunk maximum per head over the warp's rows, softmax weights in place
      float mx = -INFINITY;
      for (int x = lane; x < kRowsPerWarp * G; x += 32) mx = fmaxf(mx, S[r0 + x / G][x % G]);
#pragma unroll
      for (int msk = G; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, msk));
      float corr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mc = __shfl_sync(kFull, mx, g);
        const float mn = fmaxf(m_run[g], mc);
        corr[g] = (m_run[g] == -INFINITY) ? 0.f : exp2f(m_run[g] - mn);
        m_run[g] = mn;
      }
      // mx already holds the chunk maximum of head lane % G
      const float m_own_new = fmaxf(m_own, mx);
      const float corr_own = (m_own == -INFINITY) ? 0.f : exp2f(m_own - m_own_new);
      m_own = m_own_new;
      float psum = 0.f;
      for (int x = lane; x < kRowsPerWarp * G; x += 32) {
        const float sv = S[r0 + x / G][x % G];
        const float p = (sv == -INFINITY) ? 0.f : exp2f(sv - m_own_new);
        S[r0 + x / G][x % G] = p;
        psum += p;
      }
      l_own = l_own * corr_own + psum;
      __syncwarp();
      // pass 2: acc = corr * acc + sum_r p_r v_r
      bool rescale = false;  // (warp-uniform: the chunk maxima come from shuffles)
#pragma unroll
      for (int g = 0; g < G; ++g) rescale |= corr[g] != 1.f;
      if (rescale) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 c2 = make_float2(corr[g], corr[g]);
#pragma unroll
          for (int p = 0; p < 4; ++p) acc[g][p] = fmul2(acc[g][p], c2);
        }
      }
      auto pass2 = [&](auto check) {
#pragma unroll
        for (int it = 0; it < kRowsPerWarp / 2; ++it) {
          const int r = r0 + it * 2 + grp;
          float2 vv[4];
          row8<DT>(Vs + r * RB, kk, vv);
          if (decltype(check)::value && r >= nrow) {
#pragma unroll
            for (int p = 0; p < 4; ++p) vv[p] = make_float2(0.f, 0.f);  // unwritten shared memory
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pg = S[r][g];
            const float2 p2 = make_float2(pg, pg);
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[g][p] = ffma2(p2, vv[p], acc[g][p]);
          }
        }
      };
      if (full) pass2(std::false_type{});
      else pass2(std::true_type{});
      release_stage(i);
    }
    __syncthreads();
    // sum the two row groups of each warp; per-head totals of l
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        acc[g][p].x += __shfl_xor_sync(kFull, acc[g][p].x, 16);
        acc[g][p].y += __shfl_xor_sync(kFull, acc[g][p].y, 16);
      }
#pragma unroll
    for (int msk = G; msk < 32; msk <<= 1) l_own += __shfl_xor_sync(kFull, l_own, msk);
    if (lane < G) {  // lane g < G keeps the books of head g
      wm[wid][lane] = m_own;
      wl[wid][lane] = l_own;
    }
    if (grp == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          wacc[wid][g][8 * kk + 2 * p] = acc[g][p].x;
          wacc[wid][g][8 * kk + 2 * p + 1] = acc[g][p].y;
        }
    }
  }
  __syncthreads();
  if (!s_ok && tid == 0) set_err(v.err, kErrTimeout);
  // merge the warps into this CTA's partial: straight to the per-step-slot
  // scratch when the slice is split over several CTAs, else to shared memory
  const int64_t so = ((int64_t)b * a.nl + li) * v.Hkv + h;
  constexpr int kPart = G * kHeadDim + 2 * G;  // acc [G][d], maxima [G], sums [G]
  const int scr = a.slot & (kRing - 1);  // attention scratch slot
  const int64_t slot_part = ((int64_t)scr * v.S_all + gs) * kAttnMaxSplit * kPart;
  float *mine = nsplit > 1 ? v.attn_part + slot_part + (int64_t)split * kPart : part;
  for (int x = tid; x < G * kHeadDim; x += NTH) {
    const int g = x / kHeadDim, dim = x % kHeadDim;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mm = fmaxf(mm, wm[w][g]);
    float o = 0.f, z = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sw = (wm[w][g] == -INFINITY) ? 0.f : exp2f(wm[w][g] - mm);
      o = fmaf(sw, wacc[w][g][dim], o);
      z = fmaf(sw, wl[w][g], z);
    }
    mine[g * kHeadDim + dim] = o;
    if (dim == 0) {
      mine[G * kHeadDim + g] = mm;
      mine[G * kHeadDim + G + g] = z;
    }
  }
  // the last CTA of the slice to finish combines every CTA's partial; the
  // others leave at once
  const float *parts = part;
  if (nsplit > 1) {
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&v.attn_count[(int64_t)scr * v.S_all + gs], 1) == nsplit - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // all partials into shared memory (the ring is free) in one round of
    // coalesced loads
    float *staged = reinterpret_cast<float *>(smem);
    static_assert((size_t)kAttnMaxSplit * kPart * sizeof(float) <= attn_smem<DT, G>(), "");
    if constexpr (kPart % 4 == 0) {
      const float4 *src = reinterpret_cast<const float4 *>(v.attn_part + slot_part);
      for (int x = tid; x < nsplit * kPart / 4; x += NTH) reinterpret_cast<float4 *>(staged)[x] = __ldcg(src + x);
    } else {
      for (int x = tid; x < nsplit * kPart; x += NTH) staged[x] = __ldcg(v.attn_part + slot_part + x);
    }
    parts = staged;
  }
  __syncthreads();
  {
    float *out = a.out + k * a.stride_out;
    const int64_t obase = (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
    for (int x = tid; x < G * kHeadDim; x += NTH) {
      const int g = x / kHeadDim;
      float mc[kAttnMaxSplit];
      float mm = -INFINITY;
#pragma unroll
      for (int c = 0; c < kAttnMaxSplit; ++c) {
        mc[c] = (c < nsplit) ? parts[c * kPart + G * kHeadDim + g] : -INFINITY;
        mm = fmaxf(mm, mc[c]);
      }
      float o = 0.f, z = 0.f;
#pragma unroll
      for (int c = 0; c < kAttnMaxSplit; ++c) {
        if (c >= nsplit || mc[c] == -INFINITY) continue;
        const float sw = exp2f(mc[c] - mm);
        o = fmaf(sw, parts[c * kPart + x], o);
        z = fmaf(sw, parts[c * kPart + G * kHeadDim + G + g], z);
      }
      out[obase + x] = o / z;
    }
    const int ns = s_ns;
    if (a.selected_units) {
      const int32_t *sel = plan_sel(v, ps, gs);
      int32_t *dst = a.selected_units + k * a.stride_sel + so * v.u_cap;
      for (int x = tid; x < ns; x += NTH) dst[x] = sel[x];
    }
    if (tid == 0) {
      if (nsplit > 1) v.attn_count[(int64_t)scr * v.S_all + gs] = 0;
      if (a.n_selected) a.n_selected[k * a.stride_nsel + so] = ns;
      atomicAdd((unsigned long long *)&v.counters[kCntAttnRows], (unsigned long long)total);
      atomicAdd((unsigned long long *)&v.counters[kCntAttnSlices], 1ull);
    }
  }
}


// ---------------------------------------------------------------- streaming attention

// Tensor-core attention (bf16 rows, 4 or 8 query heads per KV head) that
// splits the step's rows over warps in proportion to each slice's actual
// size. Every slice of the call has total_s = (local-buffer rows) +
// (selected tokens) rows, known only on the device; warp w of the W warps
// of the launch serves exactly one slice:
//   w0(s) = floor((W - S) * pre(s) / R) + s,   pre(s) = sum of the totals of
//   slices before s, R = all rows,
// so slice s gets w0(s + 1) - w0(s) >= 1 warps and every warp about R / W
// rows, whatever the mix of slice sizes. A slice's rows are ordered local
// buffer first (their pool rows follow from the window start alone), then
// the selected tokens (pool row from the plan's per-token row table, or the
// offload staging row). A warp streams its rows in 16-row tiles through its
// own ring of NS stages of 16-byte cp.async copies (no warp waits for
// another), computes scores and p * V with mma.sync bf16 products (queries
// and softmax weights split into a bf16 high part and a bf16 residual, so
// both keep fp32 accuracy), writes its partial softmax state, and the last
// warp of the slice to finish combines the slice's partials.
constexpr int kStreamRowsPerWarp = 64;  // fewest rows a warp is given at the largest budget

template <int NS>
constexpr size_t stream_ring_bytes(int nw) { return (size_t)nw * NS * 2 * 16 * kHeadDim * 2; }
// dynamic shared memory: the rings, then per slice the row prefix (S + 1
// entries), the window start, the selected-token count, t and the plan slot
template <int NS>
constexpr size_t stream_smem(int nw, int S) { return stream_ring_bytes<NS>(nw) + (size_t)(5 * S + 1) * 4; }

int stream_warp_cap(int sms) { return sms * 16 > kStreamMaxSlices ? sms * 16 : kStreamMaxSlices; }

constexpr int kStreamIdxWin = 256;  // selected-token row entries a warp keeps in shared memory

__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t *p, int32_t x) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(x) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

template <int G, int NW, int NS, int MINB>
__global__ void __launch_bounds__(32 * NW, MINB) k_attn_stream(CtxView v, StepArgs a, int S, int W) {
  constexpr int RB = kHeadDim * 2;  // bytes of a bf16 row
  constexpr int WB = 16 * RB;       // a stage: 16 K rows, then 16 V rows
  constexpr int NT = G / 4;         // products per 16-row block
  constexpr int kPart = G * kHeadDim + 2 * G;
  static_assert(kPart * 4 <= NS * 2 * WB, "a warp's state must fit in its ring");
  extern __shared__ __align__(128) unsigned char smem[];
  int32_t *pre = reinterpret_cast<int32_t *>(smem + stream_ring_bytes<NS>(NW));  // [S + 1]
  int32_t *ws_s = pre + S + 1, *nt_s = ws_s + S, *t_s = nt_s + S, *pl_s = t_s + S;
  __shared__ int32_t wt[64];
  __shared__ int32_t s_total;
  __shared__ int32_t sl_w[NW];                   // slice of each warp (-1: no work)
  __shared__ int32_t idx_w[NW][kStreamIdxWin];   // each warp's window of the token-row table
  __shared__ __align__(16) float S_w[NW][16][G];  // each warp's softmax weights of a tile
  __shared__ __align__(8) uint64_t full_w[NW][NS];  // a stage's copies have landed
  __shared__ uint8_t hmask_w[NW][NS][16];  // per-query-head selection: heads that take each row
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int w = blockIdx.x * NW + wid;
  const int per_l = v.B * v.Hkv;
  const int64_t gs0 = (int64_t)a.l0 * per_l;
  if (lane < NS) {
    mbar_init(&full_w[wid][lane], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();

  // 1. the call's slice descriptors (t, window start, plan slot, selected
  //    tokens), their row totals and the exclusive prefix; with chunk
  //    selection from the step view and the plan in force
  {
    const int4 *desc = v.adesc + (int64_t)a.slot * v.S_all + gs0;
    const int per = (S + 32 * NW - 1) / (32 * NW);
    const int s0 = tid * per, s1 = min(S, s0 + per);
    int32_t part = 0;
    for (int s = s0; s < s1; ++s) {
      int4 d;
      if (v.chunk_sel) {
        const int64_t lb_s = (int64_t)(a.l0 + s / per_l) * v.B + (s % per_l) / v.Hkv;
        const int4 vw = v.aview[(int64_t)a.slot * v.n_lb + lb_s];
        d = make_int4(vw.x, vw.y, vw.z, *plan_ntok(v, vw.z, gs0 + s));
      } else {
        d = desc[s];
      }
      ws_s[s] = d.y;
      nt_s[s] = d.w;
      t_s[s] = d.x;
      pl_s[s] = d.z;
      part += d.w + (d.x - d.y + 1);
    }
    int32_t run = block_scan_excl(part, wt, &s_total);
    for (int s = s0; s < s1; ++s) {
      pre[s] = run;
      run += nt_s[s] + (t_s[s] - ws_s[s] + 1);
    }
    if (tid == 0) pre[S] = s_total;
    __syncthreads();
  }
  const int64_t R = pre[S];
  const bool active = w < W;
  // 2. this warp's slice (largest s with w0(s) <= w) and its shares of the
  //    slice's local-buffer rows and selected tokens
  auto w0 = [&](int s) -> int { return (int)((int64_t)(W - S) * pre[s] / R) + s; };
  int sl = 0;
  {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (w0(mid) <= w) lo = mid;
      else hi = mid - 1;
    }
    sl = lo;
  }
  const int wf = w0(sl), nw_s = w0(sl + 1) - wf;
  if (lane == 0) sl_w[wid] = active ? sl : -1;
  const int li = sl / per_l, rem = sl % per_l;
  const int b = rem / v.Hkv, h = rem % v.Hkv;
  const int64_t lb = (int64_t)(a.l0 + li) * v.B + b;
  const int64_t gs = gs0 + sl;
  const int win = t_s[sl] - ws_s[sl] + 1, ntok = nt_s[sl], ws = ws_s[sl], ps = pl_s[sl];
  const int kw = w - wf;
  const int wa = active ? (int)((int64_t)win * kw / nw_s) : 0;
  const int wb = active ? (int)((int64_t)win * (kw + 1) / nw_s) : 0;
  const int ja = active ? (int)((int64_t)ntok * kw / nw_s) : 0;
  const int jb = active ? (int)((int64_t)ntok * (kw + 1) / nw_s) : 0;
  const int n_wt = (wb - wa + 15) / 16;            // local-buffer tiles, first
  const int n_tiles = n_wt + (jb - ja + 15) / 16;  // then selected-token tiles
  const int64_t so = ((int64_t)b * a.nl + li) * v.Hkv + h;
  const int64_t k_out = t_s[sl] - a.base_t;
  // the slice's first warp reports the selection in force (it does not
  // depend on the attention)
  const bool per_head = v.pol_per_head != 0;
  if (active && kw == 0) {
    const int ns = *plan_nsel(v, ps, gs);
    const int32_t *sel = plan_sel(v, ps, gs);
    if (!per_head) {
      if (a.selected_units) {
        int32_t *dst = a.selected_units + k_out * a.stride_sel + so * v.u_cap;
        for (int x = lane; x < ns; x += 32) dst[x] = sel[x];
      }
      if (lane == 0 && a.n_selected) a.n_selected[k_out * a.stride_nsel + so] = ns;
    } else {
      // each query head's own selection: the union entries carrying its bit
      const uint8_t *mk = plan_sel_mask(v, ps, gs);
      const int32_t *hn = plan_hsel_n(v, ps, gs);
      for (int g = 0; g < G; ++g) {
        if (a.selected_units) {
          int32_t *dst = a.selected_units + k_out * a.stride_sel + (so * G + g) * v.u_cap;
          int base = 0;
          for (int x0 = 0; x0 < ns; x0 += 32) {
            const int x = x0 + lane;
            const bool on = x < ns && ((mk[x] >> g) & 1);
            const unsigned bal = __ballot_sync(kFull, on);
            if (on) dst[base + __popc(bal & ((1u << lane) - 1))] = sel[x];
            base += __popc(bal);
          }
        }
        if (lane == 0 && a.n_selected) a.n_selected[k_out * a.stride_nsel + so * G + g] = hn[g];
      }
    }
  }

  // row sources: local-buffer row f and selected token j
  const unsigned char *win_k, *win_v, *sel_k, *sel_v;
  const int32_t *tok_rows = nullptr;
  if (!v.offload) {
    win_k = (const unsigned char *)v.pool_k + (gs * v.pool_rows + v.n_cap + ws) * RB;
    win_v = (const unsigned char *)v.pool_v + (gs * v.pool_rows + v.n_cap + ws) * RB;
    sel_k = (const unsigned char *)v.pool_k + gs * v.pool_rows * RB;
    sel_v = (const unsigned char *)v.pool_v + gs * v.pool_rows * RB;
    tok_rows = plan_sel_rows(v, ps, gs);
  } else {
    win_k = (const unsigned char *)v.dec_k + (gs * v.dec_rows + ws) * RB;
    win_v = (const unsigned char *)v.dec_v + (gs * v.dec_rows + ws) * RB;
    sel_k = (const unsigned char *)v.stage_k + ((int64_t)ps * v.S_all + gs) * v.bud_cap * RB;
    sel_v = (const unsigned char *)v.stage_v + ((int64_t)ps * v.S_all + gs) * v.bud_cap * RB;
  }
  // a window of the selected tokens' table entries (pool rows) in shared
  // memory, filled with one round of loads
  int32_t *idx = idx_w[wid];
  int jwin = ja;
  int32_t e_idx[kStreamIdxWin / 32];  // the first window, loaded now, stored when first needed
  auto load_idx = [&](int j0) {
    jwin = j0;
#pragma unroll
    for (int r = 0; r < kStreamIdxWin / 32; ++r) {
      const int j = j0 + lane + 32 * r;
      e_idx[r] = j < jb ? tok_rows[j] : 0;
    }
  };
  auto store_idx = [&]() {
#pragma unroll
    for (int r = 0; r < kStreamIdxWin / 32; ++r) idx[lane + 32 * r] = e_idx[r];
    __syncwarp();
  };
  auto fill_idx = [&](int j0) {
    load_idx(j0);
    store_idx();
  };
  bool idx_ready = tok_rows == nullptr || jb == ja;
  if (!idx_ready) load_idx(ja);
  unsigned char *ring = smem + (size_t)wid * NS * 2 * WB;
  // Tile i goes to stage i % NS as bulk copies of its runs of consecutive
  // pool rows (lane r < 16 looks at row r; a run starts where the rows stop
  // being consecutive), completing on the stage's barrier. Rows past the
  // tile's end are zeroed so that their zero softmax weights meet finite
  // values.
  int n_issued = 0;
  auto issue = [&](int i) {
    if (i >= n_tiles) return;
    n_issued = i + 1;
    const bool wt_ = i < n_wt;
    const int base = wt_ ? wa + 16 * i : ja + 16 * (i - n_wt);
    const int nrow = wt_ ? min(16, wb - base) : min(16, jb - base);
    if (!wt_ && !idx_ready) {
      store_idx();
      idx_ready = true;
    }
    if (!wt_ && tok_rows && base + nrow > jwin + kStreamIdxWin) fill_idx(base);
    unsigned char *Kd = ring + (i % NS) * 2 * WB;
    uint64_t *bar = &full_w[wid][i % NS];
    int32_t row = 0;
    if (lane < nrow) row = (wt_ || !tok_rows) ? base + lane : idx[base + lane - jwin];
    if (per_head && lane < 16) {  // the heads of each selected row (all heads for the buffer)
      hmask_w[wid][i % NS][lane] = wt_ ? 0xffu : (uint8_t)((uint32_t)row >> kRowBits);
      row &= kRowMask;
    }
    const int32_t prev = __shfl_up_sync(kFull, row, 1);
    const unsigned starts = __ballot_sync(kFull, lane < nrow && (lane == 0 || row != prev + 1));
    if (nrow < 16) {  // zero the rows past the tile's end (generic proxy)
      for (int x = lane; x < (16 - nrow) * RB / 16; x += 32) {
        reinterpret_cast<uint4 *>(Kd + nrow * RB)[x] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(Kd + WB + nrow * RB)[x] = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nrow * 2 * RB);
    __syncwarp();
    if ((starts >> lane) & 1) {
      const unsigned after = starts & ~((2u << lane) - 1);  // later run starts
      const int end = after ? __ffs(after) - 1 : nrow;
      const uint32_t bytes = (uint32_t)(end - lane) * RB;
      const unsigned char *ks = (wt_ ? win_k : sel_k) + (int64_t)row * RB;
      const unsigned char *vs = (wt_ ? win_v : sel_v) + (int64_t)row * RB;
      bulk_g2s(Kd + lane * RB, ks, bytes, bar);
      bulk_g2s(Kd + WB + lane * RB, vs, bytes, bar);
    }
  };
  // the first stages: the local-buffer tiles (no table entries needed); the
  // selected-token tiles follow in the loop, by when their entries are in
  for (int i = 0; i < NS && i < (idx_ready ? n_tiles : n_wt); ++i) issue(i);

  // the queries (pre-scaled by log2(e)/sqrt(d)): column n of product nt_
  // carries head (G == 8 ? n : n % 4), its bf16 high part for nt_ == 0
  // (G == 8) or n < 4 (G == 4), else the bf16 residual; lane (g, t) ends
  // with D columns 2t, 2t + 1, i.e. heads hb and hb + 1
  const int gq = lane >> 2, tq = lane & 3;
  const int hb = G == 8 ? 2 * tq : 2 * (tq & 1);
  auto col_head = [](int n) { return G == 8 ? n : (n & 3); };
  auto col_lo = [](int nt, int n) { return G == 8 ? nt == 1 : n >= 4; };
  const int H = v.Hkv * G;
  uint32_t qb[4][NT][4];
  if (active) {
    const float *qh = v.q_attn + (((int64_t)a.slot * v.n_lb + lb) * H + (int64_t)h * G + col_head(gq)) * kHeadDim +
                      8 * tq;
    float qf[4][8];
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const float4 u0 = __ldg((const float4 *)(qh + 32 * P));
      const float4 u1 = __ldg((const float4 *)(qh + 32 * P + 4));
      qf[P][0] = u0.x; qf[P][1] = u0.y; qf[P][2] = u0.z; qf[P][3] = u0.w;
      qf[P][4] = u1.x; qf[P][5] = u1.y; qf[P][6] = u1.z; qf[P][7] = u1.w;
    }
#pragma unroll
    for (int P = 0; P < 4; ++P)
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
        for (int q = 0; q < 4; ++q) qb[P][nt_][q] = bf16_pair(qf[P][2 * q], qf[P][2 * q + 1], col_lo(nt_, gq));
  }
  float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};  // heads hb, hb + 1
  float o[NT][8][4];
#pragma unroll
  for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt_][m][e] = 0.f;
  bool ok = true;

  for (int i = 0; i < n_tiles; ++i) {
    const unsigned char *Kw = ring + (i % NS) * 2 * WB;
    const unsigned char *Vw = Kw + WB;
    while (n_issued <= i) issue(n_issued);  // (a warp whose first tile is a selected one)
    if (!mbar_wait_bounded(&full_w[wid][i % NS], (i / NS) & 1, kWaitLimitNs)) {
      ok = false;  // record it; the drain below waits once more for the copies
      break;
    }
    const bool wt_ = i < n_wt;
    const int nrow = wt_ ? min(16, wb - (wa + 16 * i)) : min(16, jb - (ja + 16 * (i - n_wt)));
    // scores of rows g and g + 8, two accumulation chains
    float sc[NT][2][4];
#pragma unroll
    for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt_][0][e] = sc[nt_][1][e] = 0.f;
    const unsigned char *kr = Kw + gq * RB + 16 * tq;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const uint4 x = *(const uint4 *)(kr + 64 * P);
      const uint4 y = *(const uint4 *)(kr + 8 * RB + 64 * P);
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_) {
        mma_bf16(sc[nt_][0], x.x, y.x, x.y, y.y, qb[P][nt_][0], qb[P][nt_][1]);
        mma_bf16(sc[nt_][1], x.z, y.z, x.w, y.w, qb[P][nt_][2], qb[P][nt_][3]);
      }
    }
    // s[0], s[1]: row g, heads hb, hb + 1; s[2], s[3]: row g + 8
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[e] = sc[0][0][e] + sc[0][1][e];
      if constexpr (NT == 2) s[e] += sc[1][0][e] + sc[1][1][e];
      else s[e] += __shfl_xor_sync(kFull, s[e], 2);  // high part + residual
    }
    if (nrow < 16) {  // rows past the tile's end score -inf
      if (gq >= nrow) s[0] = s[1] = -INFINITY;
      if (gq + 8 >= nrow) s[2] = s[3] = -INFINITY;
    }
    if (per_head) {  // a head sees only the rows of its own selection (and the buffer)
      const uint32_t m0 = hmask_w[wid][i % NS][gq], m1 = hmask_w[wid][i % NS][gq + 8];
      if (!((m0 >> hb) & 1u)) s[0] = -INFINITY;
      if (!((m0 >> (hb + 1)) & 1u)) s[1] = -INFINITY;
      if (!((m1 >> hb) & 1u)) s[2] = -INFINITY;
      if (!((m1 >> (hb + 1)) & 1u)) s[3] = -INFINITY;
    }
    // online softmax; rescale only when a maximum moves
    float c[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(s[e], s[e + 2]);
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, msk));
      const float mn = fmaxf(mr[e], mx);
      c[e] = (mr[e] == -INFINITY) ? 0.f : exp2f(mr[e] - mn);
      mr[e] = mn;
    }
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = (s[e] == -INFINITY) ? 0.f : exp2f(s[e] - mr[e & 1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) lr[e] = lr[e] * c[e] + p[e] + p[e + 2];
    if (__any_sync(kFull, c[0] != 1.f || c[1] != 1.f)) {
#pragma unroll
      for (int nt_ = 0; nt_ < NT; ++nt_)
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt_][m][e] *= c[e & 1];
    }
    // p^T as the B operand of p * V (rows = tokens), through shared memory
    float(*Sw)[G] = S_w[wid];
    if (G == 8 || tq < 2) {
      *(float2 *)&Sw[gq][hb] = make_float2(p[0], p[1]);
      *(float2 *)&Sw[gq + 8][hb] = make_float2(p[2], p[3]);
    }
    __syncwarp();
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt_ = 0; nt_ < NT; ++nt_) {
      const int hh = col_head(gq);
      const bool lo_ = col_lo(nt_, gq);
      pb[nt_][0] = bf16_pair(Sw[2 * tq][hh], Sw[2 * tq + 1][hh], lo_);
      pb[nt_][1] = bf16_pair(Sw[2 * tq + 8][hh], Sw[2 * tq + 9][hh], lo_);
    }
    // p * V: product m = 4 hf + j has output rows dim 64 hf + 8 g + 2 j (row
    // g) and that dim + 1 (row g + 8); lane (g, t) reads tokens 2t, 2t + 1,
    // 2t + 8, 2t + 9 at dims [64 hf + 8 g, + 8) and pairs them up by token
    const unsigned char *vr = Vw + (2 * tq) * RB + 16 * gq;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint4 v0 = *(const uint4 *)(vr + 128 * hf);
      const uint4 v1 = *(const uint4 *)(vr + RB + 128 * hf);
      const uint4 v2 = *(const uint4 *)(vr + 8 * RB + 128 * hf);
      const uint4 v3 = *(const uint4 *)(vr + 9 * RB + 128 * hf);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w0_ = word(v0, j), w1_ = word(v1, j), w2_ = word(v2, j), w3_ = word(v3, j);
        const uint32_t a0 = prmt(w0_, w1_, 0x5410u), a1 = prmt(w0_, w1_, 0x7632u);
        const uint32_t a2 = prmt(w2_, w3_, 0x5410u), a3 = prmt(w2_, w3_, 0x7632u);
#pragma unroll
        for (int nt_ = 0; nt_ < NT; ++nt_) mma_bf16(o[nt_][4 * hf + j], a0, a1, a2, a3, pb[nt_][0], pb[nt_][1]);
      }
    }
    // every lane's reads of this stage (and of the weights) are done: keep
    // NS tiles in flight
    __syncwarp();
    while (n_issued < n_tiles && n_issued < i + 1 + NS) issue(n_issued);
  }
  if (!ok) {
    // a copy never completed: record it, and let every copy this warp issued
    // land (one more bounded wait per stage) before the block's memory goes
    if (lane == 0) set_err(v.err, kErrTimeout);
    for (int i2 = max(0, n_issued - NS); i2 < n_issued; ++i2)
      mbar_wait_bounded(&full_w[wid][i2 % NS], (i2 / NS) & 1, kWaitLimitNs);
  }
  __syncwarp();

  // 3. this warp's state (high part + residual, per-head maxima and sums)
  //    into its ring, which is free now
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if constexpr (NT == 2) o[0][m][e] += o[NT - 1][m][e];
      else o[0][m][e] += __shfl_xor_sync(kFull, o[0][m][e], 2);
    }
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) lr[e] += __shfl_xor_sync(kFull, lr[e], msk);
  float *mine = reinterpret_cast<float *>(ring);
  if (G == 8 || tq < 2) {
    if (gq == 0) {
      mine[G * kHeadDim + hb] = mr[0];
      mine[G * kHeadDim + hb + 1] = mr[1];
      mine[G * kHeadDim + G + hb] = lr[0];
      mine[G * kHeadDim + G + hb + 1] = lr[1];
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float *dst = mine + (hb + e) * kHeadDim + 64 * hf + 8 * gq;
        *(float4 *)dst = make_float4(o[0][4 * hf][e], o[0][4 * hf][e + 2], o[0][4 * hf + 1][e],
                                     o[0][4 * hf + 1][e + 2]);
        *(float4 *)(dst + 4) = make_float4(o[0][4 * hf + 2][e], o[0][4 * hf + 2][e + 2],
                                           o[0][4 * hf + 3][e], o[0][4 * hf + 3][e + 2]);
      }
  }
  __syncthreads();

  // 4. the first warp of each slice in this CTA merges the CTA's warps of
  //    that slice into one partial (stored at the index of that first warp);
  //    the last partial of the slice to arrive combines them all
  if (!active || (wid > 0 && sl_w[wid - 1] == sl)) return;
  int n_mine = 1;
  while (wid + n_mine < NW && sl_w[wid + n_mine] == sl) ++n_mine;
  constexpr int kVec = G * kHeadDim / 4 / 32;  // float4s per lane (= G; float4 lane + 32 j lies in head j)
  static_assert(kVec == G, "");
  float4 acc[kVec];
  float M[G], Z[G];
  {
    const float *st0 = reinterpret_cast<const float *>(smem + (size_t)wid * NS * 2 * WB);
    constexpr size_t kStride = (size_t)NS * 2 * WB / 4;  // floats between consecutive warps' states
#pragma unroll
    for (int g = 0; g < G; ++g) {
      M[g] = -INFINITY;
      for (int u = 0; u < n_mine; ++u) M[g] = fmaxf(M[g], st0[u * kStride + G * kHeadDim + g]);
      Z[g] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int u = 0; u < n_mine; ++u) {
      const float *st = st0 + u * kStride;
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const float m = st[G * kHeadDim + j];
        const float f = (m == -INFINITY) ? 0.f : exp2f(m - M[j]);
        const float4 x = *reinterpret_cast<const float4 *>(st + 4 * (lane + 32 * j));
        acc[j].x = fmaf(f, x.x, acc[j].x);
        acc[j].y = fmaf(f, x.y, acc[j].y);
        acc[j].z = fmaf(f, x.z, acc[j].z);
        acc[j].w = fmaf(f, x.w, acc[j].w);
        Z[j] = fmaf(f, st[G * kHeadDim + G + j], Z[j]);
      }
    }
  }
  // partial ids of the slice: its first warp, then the first warp of every
  // later CTA that serves it
  const int n_parts = 1 + (w0(sl + 1) - 1) / NW - wf / NW;
  float *pbase = v.attn_wpart + (int64_t)(a.slot & (kRing - 1)) * v.w_cap * kPart;
  int32_t *cnt = v.attn_count + (int64_t)(a.slot & (kRing - 1)) * v.S_all + gs;
  if (n_parts > 1) {
    float *dst = pbase + (int64_t)w * kPart;
#pragma unroll
    for (int j = 0; j < kVec; ++j) *reinterpret_cast<float4 *>(dst + 4 * (lane + 32 * j)) = acc[j];
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        dst[G * kHeadDim + g] = M[g];
        dst[G * kHeadDim + G + g] = Z[g];
      }
    // publish (every lane's release fence) and count; the last partial's
    // warp acquires the others' before reading them
    fence_acq_rel_gpu();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atom_add_acq_rel_gpu(cnt, 1) == n_parts - 1;
    last = __shfl_sync(kFull, last, 0);
    if (!last) return;
    fence_acq_rel_gpu();
    // every partial's maxima, sums and accumulators, loaded together in
    // groups of four
    float Mx[G];
#pragma unroll
    for (int g = 0; g < G; ++g) Mx[g] = -INFINITY;
    for (int c0 = 0; c0 < n_parts; c0 += 32) {
      const int cc = c0 + lane;
      const int pid = cc == 0 ? wf : (wf / NW + cc) * NW;
#pragma unroll
      for (int g = 0; g < G; ++g)
        Mx[g] = fmaxf(Mx[g], cc < n_parts ? __ldcg(pbase + (int64_t)pid * kPart + G * kHeadDim + g) : -INFINITY);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int msk = 16; msk; msk >>= 1) Mx[g] = fmaxf(Mx[g], __shfl_xor_sync(kFull, Mx[g], msk));
      M[g] = Mx[g];
      Z[g] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n_parts; c0 += 4) {
      float4 x[4][kVec];
      float mm[4][G], ll[4][G];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cc = c0 + u;
        const int pid = cc == 0 ? wf : (wf / NW + cc) * NW;
        const float *src = pbase + (int64_t)(cc < n_parts ? pid : wf) * kPart;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mm[u][g] = __ldcg(src + G * kHeadDim + g);
          ll[u][g] = __ldcg(src + G * kHeadDim + G + g);
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) x[u][j] = __ldcg(reinterpret_cast<const float4 *>(src) + lane + 32 * j);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + u >= n_parts) break;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          const float f = (mm[u][j] == -INFINITY) ? 0.f : exp2f(mm[u][j] - M[j]);
          Z[j] = fmaf(f, ll[u][j], Z[j]);
          acc[j].x = fmaf(f, x[u][j].x, acc[j].x);
          acc[j].y = fmaf(f, x[u][j].y, acc[j].y);
          acc[j].z = fmaf(f, x[u][j].z, acc[j].z);
          acc[j].w = fmaf(f, x[u][j].w, acc[j].w);
        }
      }
    }
  }
  float *out = a.out + k_out * a.stride_out + (((int64_t)b * a.nl + li) * H + (int64_t)h * G) * kHeadDim;
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const float z = Z[j];
    reinterpret_cast<float4 *>(out)[lane + 32 * j] =
        make_float4(acc[j].x / z, acc[j].y / z, acc[j].z / z, acc[j].w / z);
  }
  if (lane == 0) {
    if (n_parts > 1) *cnt = 0;
    atomicAdd((unsigned long long *)&v.counters[kCntAttnRows], (unsigned long long)(win + ntok));
    atomicAdd((unsigned long long *)&v.counters[kCntAttnSlices], 1ull);
  }
}

// ---------------------------------------------------------------- host-link ceiling

// Plain streaming read of pinned, mapped host memory into device memory:
// every thread moves 16-byte vectors, eight loads in flight, over a grid
// that fills the GPU. It does what the offload gather does minus the
// selection (one contiguous run), so its rate is the ceiling that gather is
// measured against on the same link.
__global__ void __launch_bounds__(256) k_uva_read(const uint4 *src, uint4 *dst, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = __ldcg(src + i + e * stride);
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[i + e * stride] = r[e];
  }
  for (; i < n16; i += stride) dst[i] = __ldcg(src + i);
}

cudaError_t launch_uva_read(const void *host_src, void *dev_dst, int64_t bytes, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  k_uva_read<<<sms * 8, 256, 0, st>>>((const uint4 *)host_src, (uint4 *)dev_dst, bytes / 16);
  return cudaGetLastError();
}

// Single-launch read ceiling of device memory: the same grid and load
// pattern as k_uva_read, reads only (each thread folds its loads into one
// word, stored only when it matches a value no input of the measurement
// gives, so the loads cannot be dropped). A decode step's attention reads
// its rows in one launch; this kernel reads the same number of bytes
// contiguously, so its event-timed rate bounds what one launch of that size
// reaches.
__device__ uint32_t g_read_sink;

__global__ void __launch_bounds__(256) k_read_ceiling(const uint4 *src, int64_t n16) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = __ldcg(src + i + e * stride);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc ^= r[e].x ^ r[e].y ^ r[e].z ^ r[e].w;
  }
  for (; i < n16; i += stride) {
    const uint4 r = __ldcg(src + i);
    acc ^= r.x ^ r.y ^ r.z ^ r.w;
  }
  if (acc == 0x9e3779b9u) g_read_sink = acc;
}

cudaError_t launch_read_ceiling(const void *src, int64_t bytes, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  k_read_ceiling<<<sms * 8, 256, 0, st>>>((const uint4 *)src, bytes / 16);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- failure-path check

// One CTA waits on an mbarrier that nothing completes. The wait gives up
// after limit_ns, records the timeout bit exactly as a kernel whose bounded
// wait ran out does, and the CTA returns.
__global__ void k_diag_wait(CtxView v, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  __syncthreads();
  if (!ok && threadIdx.x == 0) set_err(v.err, kErrTimeout);
}

cudaError_t launch_diag_wait(const CtxView &v, uint64_t limit_ns, cudaStream_t st) {
  k_diag_wait<<<1, 32, 0, st>>>(v, limit_ns);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor drains and waits for it in pdl_wait().
// Scheduling priorities: the serial boundary/selection chain of the decode
// steps goes first, so that a pending attention grid does not hold back the
// next step's chain when SM resources free up.
static int g_prio_chain = 0, g_prio_attn = 0;

template <typename... KArgs, typename... Args>
static void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = g_prio_chain;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, kern, args...);
}



static int g_attn_slots = 2 * 152;  // resident attention CTAs on the device
static int g_attn_split = 0;        // CTAs per slice forced by LKV_ATTN_CTAS_PER_SLICE (0: auto)
constexpr int kAttnConcurrent = 3;  // pipelined attention grids sized to run this many at once

// Split of a slice's chunks over at most kAttnMaxSplit CTAs:
// `concurrent` grids (consecutive steps of a pipelined graph, else 1) are
// resident at once where possible.
static void attn_split(int slices, int nch, int concurrent, int *nsplit, int *cpc) {
  int want = g_attn_split > 0 ? g_attn_split : g_attn_slots / (slices * concurrent);
  if (want < 1) want = 1;
  if (want > kAttnMaxSplit) want = kAttnMaxSplit;
  if (want > nch) want = nch;
  *cpc = (nch + want - 1) / want;
  *nsplit = (nch + *cpc - 1) / *cpc;
}

template <int DT, int G>
static void launch_attn(const CtxView &v, const StepArgs &a, int slices, int nch, int concurrent,
                        cudaStream_t st) {
  int nsplit = 1, cpc = 1;
  attn_split(slices, nch, concurrent, &nsplit, &cpc);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(slices, nsplit);
  cfg.blockDim = dim3(attn_threads<DT, G>());
  cfg.dynamicSmemBytes = attn_smem<DT, G>();
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = g_prio_attn;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, k_attn<DT, G>, v, a, cpc);
}

// Streaming attention launch configurations: (warps per CTA, ring stages
// per warp). A single-step launch has the GPU to itself and takes one CTA of
// 8 warps with 3-stage rings per SM; inside a pipelined decode graph three
// attention launches share the GPU with the boundary and selection kernels,
// so CTAs are smaller.
struct StreamCfg {
  int nw, ns, minb;  // warps per CTA, ring stages per warp, CTAs per SM the registers must allow
};
constexpr StreamCfg kStreamCfgs[] = {{8, 3, 1}, {4, 2, 3}, {4, 3, 2}, {8, 2, 1}};
static int g_stream_single = 0, g_stream_pipe = 1;
static int g_stream_pipe_div = 6;  // a pipelined launch takes 1 / this of the resident warps
static int g_stream_blocks[4] = {1, 1, 1, 1};  // resident CTAs per SM of each configuration
static int g_sms = 152;

template <int G, int C>
static auto stream_kernel() {
  constexpr StreamCfg cf = kStreamCfgs[C];
  return k_attn_stream<G, cf.nw, cf.ns, cf.minb>;
}

template <int G, int C>
static cudaError_t prep_stream() {
  constexpr StreamCfg cf = kStreamCfgs[C];
  const size_t smem = stream_smem<cf.ns>(cf.nw, kStreamMaxSlices);
  cudaError_t e = cudaFuncSetAttribute(stream_kernel<G, C>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel<G, C>(), 32 * cf.nw,
                                                    stream_ring_bytes<cf.ns>(cf.nw) + 8 * 1024);
  if (e != cudaSuccess) return e;
  g_stream_blocks[C] = per_sm > 0 ? per_sm : 1;
  return cudaSuccess;
}

template <int G>
static cudaError_t prep_stream_all() {
  cudaError_t e = prep_stream<G, 0>();
  if (e == cudaSuccess) e = prep_stream<G, 1>();
  if (e == cudaSuccess) e = prep_stream<G, 2>();
  if (e == cudaSuccess) e = prep_stream<G, 3>();
  if (e != cudaSuccess) return e;
  if (const char *env = getenv("LKV_ATTN_STREAM_PIPE")) {
    const int x = atoi(env);
    if (x >= 0 && x < 4) g_stream_pipe = x;
  }
  if (const char *env = getenv("LKV_ATTN_STREAM_DIV")) {
    const int x = atoi(env);
    if (x >= 1 && x <= 16) g_stream_pipe_div = x;
  }
  if (const char *env = getenv("LKV_ATTN_STREAM_SINGLE")) {
    const int x = atoi(env);
    if (x >= 0 && x < 4) g_stream_single = x;
  }
  return cudaSuccess;
}

template <int G, int C>
static void launch_stream_c(const CtxView &v, const StepArgs &a, int slices, int concurrent,
                            cudaStream_t st) {
  constexpr StreamCfg cf = kStreamCfgs[C];
  int64_t W = (int64_t)g_stream_blocks[C] * g_sms * cf.nw / (concurrent > 1 ? g_stream_pipe_div : 1);
  const int64_t sel_max = (int64_t)(v.pol_per_head ? v.G : 1) * a.budget;  // a per-head union: up to G budgets
  const int64_t rows_cap = (int64_t)slices * ((sel_max + v.L + kStreamRowsPerWarp - 1) / kStreamRowsPerWarp);
  if (W > rows_cap) W = rows_cap;
  if (W < slices) W = slices;
  if (W > v.w_cap) W = v.w_cap;
  const int P = (int)((W + cf.nw - 1) / cf.nw);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P);
  cfg.blockDim = dim3(32 * cf.nw);
  cfg.dynamicSmemBytes = stream_smem<cf.ns>(cf.nw, slices);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = g_prio_attn;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, stream_kernel<G, C>(), v, a, slices, (int)W);
}

template <int G>
static void launch_stream(const CtxView &v, const StepArgs &a, int slices, int concurrent,
                          cudaStream_t st) {
  switch (concurrent > 1 ? g_stream_pipe : g_stream_single) {
    case 0: launch_stream_c<G, 0>(v, a, slices, concurrent, st); break;
    case 1: launch_stream_c<G, 1>(v, a, slices, concurrent, st); break;
    case 2: launch_stream_c<G, 2>(v, a, slices, concurrent, st); break;
    default: launch_stream_c<G, 3>(v, a, slices, concurrent, st); break;
  }
}

template <int DT, int G>
static cudaError_t prep_attn() {
  cudaError_t e = cudaFuncSetAttribute(k_attn<DT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)attn_smem<DT, G>());
  if (e != cudaSuccess) return e;
  int per_sm = 0, dev = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_attn<DT, G>, attn_threads<DT, G>(),
                                                    attn_smem<DT, G>());
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (per_sm > 0 && sms > 0) g_attn_slots = per_sm * sms;
  if (sms > 0) g_sms = sms;
  if constexpr (DT == 1 && (G == 4 || G == 8)) {
    e = prep_stream_all<G>();
    if (e != cudaSuccess) return e;
  }
  int least = 0, greatest = 0;  // numerically: least >= greatest; greatest is the highest priority
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess) {
    g_prio_chain = greatest;
    g_prio_attn = least;
  }
  if (const char *env = getenv("LKV_ATTN_CTAS_PER_SLICE")) {
    const int x = atoi(env);
    g_attn_split = (x >= 1 && x <= kAttnMaxSplit) ? x : 0;
  }
  e = cudaFuncSetAttribute(k_select<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelHeadSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_select_chunk<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSelHeadSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_step_boundary<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(2 * kMaxHeads * kQPitch * elem_bytes<DT>()));
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
static cudaError_t decode_t(const CtxView &v, const StepArgs &a, int n_steps, cudaStream_t st, Prof &prof,
                            const Pipe *pipe) {
  const int slices = a.nl * v.B * v.Hkv;
  const int H = v.Hkv * v.G;
  cudaError_t e = cudaSuccess;
  // the boundary tests and state of all n_steps steps, step i in slot a.slot + i
  prof.begin(kPBoundary, st);
  launch_pdl(k_step_boundary<DT>, dim3(a.nl * v.B), dim3(kBoundaryThreads),
             (size_t)2 * H * kQPitch * elem_bytes<DT>(), st, v, a, n_steps);
  if (v.paris) launch_pdl(k_paris_append, dim3(a.nl * v.B, n_steps), dim3(32 * v.Hkv), 0, st, v, a);
  prof.end(st);
  // pipelined: the selection lane follows the boundary kernel, each step's
  // attention follows its selection on a side stream
  cudaStream_t ss = st;
  if (pipe) {
    ss = pipe->sel;
    e = cudaEventRecord(pipe->b_done, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, pipe->b_done, 0);
    if (e != cudaSuccess) return e;
  }
  const int nch = (a.budget + v.L + kAttnChunk - 1) / kAttnChunk;
  const int conc = pipe ? kAttnConcurrent : 1;
  if (v.chunk_sel) {
    // chunk selection: every retrieval of the n_steps steps in one launch,
    // then the steps' attentions (step i's on attn[i % kAttnStreams], so it
    // follows step i - kAttnStreams's, whose scratch slot it may share)
    const int chunk = pipe ? pipe->step / kChunk : 0;
    if (pipe && chunk >= 2) {  // chunk - 2's attentions are done (plan ring, see Pipe)
      e = cudaStreamWaitEvent(ss, pipe->chunk_done[(chunk - 2) % 3], 0);
      if (e != cudaSuccess) return e;
    }
    prof.begin(kPSelect, ss);
    launch_pdl(k_select_chunk<DT>, dim3(slices, n_steps), dim3(kScoreThreads),
               v.pol_per_head ? kSelHeadSmemBytes : v.paris ? kSelParisSmemBytes : kSelSmemBytes, ss, v, a);
    prof.end(ss);
    if (pipe) {
      e = cudaEventRecord(pipe->sel_done, ss);
      if (e != cudaSuccess) return e;
    }
    for (int i = 0; i < n_steps; ++i) {
      StepArgs ai = a;
      ai.slot = a.slot + i;
      const int step = pipe ? pipe->step + i : 0;
      cudaStream_t as = ss;
      if (pipe) {
        as = pipe->attn[step % kAttnStreams];
        e = cudaStreamWaitEvent(as, pipe->sel_done, 0);
        if (e != cudaSuccess) return e;
      }
      prof.begin(kPAttn, as);
      if (v.G == 4) launch_stream<4>(v, ai, slices, conc, as);
      else launch_stream<8>(v, ai, slices, conc, as);
      prof.end(as);
      if (pipe) {
        e = cudaEventRecord(pipe->attn_done[step % kAttnStreams], as);
        if (e != cudaSuccess) return e;
      }
    }
    if (pipe) {  // every attention of this chunk, joined
      for (int s = 0; s < kAttnStreams && s < n_steps && e == cudaSuccess; ++s)
        e = cudaStreamWaitEvent(pipe->join, pipe->attn_done[(pipe->step + n_steps - 1 - s) % kAttnStreams], 0);
      if (e == cudaSuccess) e = cudaEventRecord(pipe->chunk_done[chunk % 3], pipe->join);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  for (int i = 0; i < n_steps; ++i) {
    StepArgs ai = a;
    ai.slot = a.slot + i;
    const int step = pipe ? pipe->step + i : 0;
    // bound the attentions in flight (see Pipe): every kSelWaitStride-th
    // selection waits for the attention kAttnStreams steps before it
    if (pipe && step >= kAttnStreams && step % kSelWaitStride == 0) {
      e = cudaStreamWaitEvent(ss, pipe->attn_done[step % kAttnStreams], 0);
      if (e != cudaSuccess) return e;
    }
    prof.begin(kPSelect, ss);
    launch_pdl(k_select<DT>, dim3(slices, kScoreSplit), dim3(kScoreThreads),
               v.pol_per_head ? kSelHeadSmemBytes : v.paris ? kSelParisSmemBytes : kSelSmemBytes, ss, v, ai);
    prof.end(ss);
    if (v.offload) {
      prof.begin(kPGather, ss);
      launch_pdl(k_gather_offload<DT>, dim3(slices, 64), dim3(256), 0, ss, v, ai);
      prof.end(ss);
    }
    cudaStream_t as = ss;
    if (pipe) {
      as = pipe->attn[step % kAttnStreams];
      e = cudaEventRecord(pipe->sel_done, ss);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(as, pipe->sel_done, 0);
      if (e != cudaSuccess) return e;
    }
    prof.begin(kPAttn, as);
    const bool stream = DT == 1 && (v.G == 4 || v.G == 8) && slices <= kStreamMaxSlices;
    if (stream && v.G == 4) {
      launch_stream<4>(v, ai, slices, conc, as);
    } else if (stream) {
      launch_stream<8>(v, ai, slices, conc, as);
    } else {
      switch (v.G) {
        case 1: launch_attn<DT, 1>(v, ai, slices, nch, conc, as); break;
        case 2: launch_attn<DT, 2>(v, ai, slices, nch, conc, as); break;
        case 4: launch_attn<DT, 4>(v, ai, slices, nch, conc, as); break;
        case 8: launch_attn<DT, 8>(v, ai, slices, nch, conc, as); break;
        default: return cudaErrorInvalidValue;
      }
    }
    prof.end(as);
    if (pipe) {
      e = cudaEventRecord(pipe->attn_done[step % kAttnStreams], as);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_steps(const CtxView &v, const StepArgs &a, int n_steps, cudaStream_t stream,
                                Prof &prof, const Pipe *pipe) {
  if (v.dtype == 1) return decode_t<1>(v, a, n_steps, stream, prof, pipe);
  return decode_t<0>(v, a, n_steps, stream, prof, pipe);
}

}  // namespace lkv
