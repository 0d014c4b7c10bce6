// kmeans.cu -- prefill index build: K-means over each (sequence, KV head)'s
// keys, then the cluster-grouped K/V pool and the unit table
// [LouisKV notes, 关键设计 2: cluster the input keys with K-means; centroid =
// mean of the cluster's keys; it is the retrieval index of the cluster].
//
// Lloyd round = assign (argmin squared distance to the scoring operand of the
// current centroids) + update (member mean).
//
// Assignment is decided on the double-precision squared distance
//   D(k, c) = sum_j (k_j - c_j)^2   (index order, separate sub/mul/add),
// ties to the lowest cluster id. A fast single-precision distance e_j =
// |c_j|^2 - 2 k.c_j (equal to D - |k|^2 up to rounding) filters: with a proven
// bound beta on |e_j - (D_j - |k|^2)|, a key whose two smallest e differ by
// more than 2 beta has a certain argmin; otherwise the key goes on a list and
// is settled by evaluating D in double precision for the two candidates (or
// for every cluster when a third one is also within 2 beta).
//
// Update: members are grouped by a stable counting sort (token order within a
// cluster); the member sum of bf16 keys is formed exactly in fixed point
// (2^-35, else 2^-40), which equals the token-order double sum whenever no
// partial sum can round; otherwise, and always for fp32 keys, it is the
// double-precision token-order sum itself; centroid = float(sum / count) in
// double.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <mutex>
#include <string>

#include "../../include/lkv.h"
#include "lkv_internal.cuh"

namespace lkv {

// ---------------------------------------------------------------- init

template <int DT>
__global__ void k_init_cent(const void *keys, int64_t n, int32_t c,
                            const int64_t *idx, float *cent32, int64_t gs0,
                            int32_t u_cap) {
  const int s = blockIdx.y, j = blockIdx.x, t = threadIdx.x;  // 128 threads
  const int64_t row = idx[(int64_t)s * c + j];
  const float v = load_elem<DT>(keys, ((int64_t)s * n + row) * kHeadDim + t);
  cent32[((gs0 + s) * u_cap + j) * kHeadDim + t] = v;
}

template <int DT>
__global__ void k_key_norms(const void *keys, int64_t n, int64_t n_cap, float *knorm) {
  const int s = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (i >= n) return;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float x = load_elem<DT>(keys, ((int64_t)s * n + i) * kHeadDim + lane * 4 + e);
    acc = fmaf(x, x, acc);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) knorm[(int64_t)s * n_cap + i] = sqrtf(acc);
}

// Scoring/assignment operand of the current centroids (bf16-rounded for bf16
// keys), its squared norm in fp32, and per-slice maxima of |c| and |c|^2.
// A CTA covers 64 centroids (a warp per centroid, lane per 4 dimensions) and
// folds its maxima into the slice's two words with one atomic each.
constexpr int kPrepPerCta = 64;

template <int DT>
__global__ void __launch_bounds__(256)
k_prepare_operand(const float *cent32, void *cent_op, int32_t c, int32_t c_pad, int32_t c2_pitch,
                  int32_t u_cap, int64_t gs0, float *c2, float *cstat, uint16_t *c2b) {
  __shared__ float wmax[8][2];
  const int s = blockIdx.y;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float cmax = 0.f, c2max = 0.f;
  for (int t = 0; t < kPrepPerCta / 8; ++t) {
    const int j = blockIdx.x * kPrepPerCta + t * 8 + wid;
    if (j >= c_pad) break;
    const int64_t base = ((gs0 + s) * u_cap + j) * kHeadDim + lane * 4;
    if (j >= c) {
      // padding up to c_pad for the tensor-core filter: |c|^2 = FLT_MAX (a
      // finite value no distance reaches) and zero operand rows, so the
      // padded columns of a chunk stay finite and never win
      if (lane == 0) c2[(int64_t)s * c2_pitch + j] = FLT_MAX;
      // the tensor-core filter's -|c|^2 / 2 row: a value no filter value reaches
      if (c2b && lane < 8)
        reinterpret_cast<uint32_t *>(c2b + ((int64_t)s * c2_pitch + j) * 16)[lane] = lane == 0 ? 0xf1800000u >> 16 : 0u;
      if (j < u_cap) {
        if constexpr (DT == 1) *(uint2 *)((uint16_t *)cent_op + base) = make_uint2(0u, 0u);
        else *(float4 *)((float *)cent_op + base) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      continue;
    }
    const float4 x4 = *(const float4 *)(cent32 + base);
    float x[4] = {x4.x, x4.y, x4.z, x4.w};
    if constexpr (DT == 1) {
      uint16_t b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        b[e] = f32_to_bf16_bits(x[e]);
        x[e] = bf16_bits_to_f32(b[e]);
      }
      *(uint2 *)((uint16_t *)cent_op + base) =
          make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16), (uint32_t)b[2] | ((uint32_t)b[3] << 16));
    } else {
      *(float4 *)((float *)cent_op + base) = x4;
    }
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc = fmaf(x[e], x[e], acc);
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) c2[(int64_t)s * c2_pitch + j] = acc;
    if (c2b && lane < 8) {
      // -|c|^2 / 2 as a bf16 pair (high part and rounded remainder) for the
      // tensor-core filter's extra product with a row of ones
      const float hv = -0.5f * acc;
      const uint16_t hi = f32_to_bf16_bits(hv);
      const uint16_t lo = f32_to_bf16_bits(hv - bf16_bits_to_f32(hi));
      reinterpret_cast<uint32_t *>(c2b + ((int64_t)s * c2_pitch + j) * 16)[lane] =
          lane == 0 ? (uint32_t)hi | ((uint32_t)lo << 16) : 0u;
    }
    cmax = fmaxf(cmax, sqrtf(acc));
    c2max = fmaxf(c2max, acc);
  }
  if (lane == 0) { wmax[wid][0] = cmax; wmax[wid][1] = c2max; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) { cmax = fmaxf(cmax, wmax[w][0]); c2max = fmaxf(c2max, wmax[w][1]); }
    // non-negative floats order like their bit patterns
    atomicMax((unsigned *)&cstat[2 * s], __float_as_uint(cmax));
    atomicMax((unsigned *)&cstat[2 * s + 1], __float_as_uint(c2max));
  }
}

template <int DT>
static void launch_prepare(const CtxView &v, int32_t c, int32_t c_pad, int32_t c2_pitch, int64_t gs0,
                           int S, float *c2, float *cstat, cudaStream_t st, uint16_t *c2b = nullptr) {
  k_prepare_operand<DT><<<dim3((c_pad + kPrepPerCta - 1) / kPrepPerCta, S), 256, 0, st>>>(
      v.cent32, v.cent_op, c, c_pad, c2_pitch, v.u_cap, gs0, c2, cstat, c2b);
}

// ---------------------------------------------------------------- assignment

// Running three smallest (value, index) pairs, lexicographic order; only the
// value of the third is kept.
struct Top3 {
  float v1, v2, v3;
  int32_t j1, j2;
};

__device__ __forceinline__ bool lex_less(float a, int32_t ia, float b, int32_t ib) {
  return a < b || (a == b && ia < ib);
}

__device__ __forceinline__ void top3_push(Top3 &t, float v, int32_t j) {
  // callers push indices in increasing order, so a strict value compare
  // keeps the lowest index among equal values
  if (v < t.v3) {
    if (v < t.v2) {
      t.v3 = t.v2;
      if (v < t.v1) {
        t.v2 = t.v1; t.j2 = t.j1;
        t.v1 = v; t.j1 = j;
      } else {
        t.v2 = v; t.j2 = j;
      }
    } else {
      t.v3 = v;
    }
  }
}

__device__ __forceinline__ Top3 top3_merge(const Top3 &a, const Top3 &b) {
  // merge two lexicographically sorted top-3 lists
  float v[6] = {a.v1, a.v2, a.v3, b.v1, b.v2, b.v3};
  int32_t j[6] = {a.j1, a.j2, 0x7fffffff, b.j1, b.j2, 0x7fffffff};
  int ia = 0, ib = 3;
  float ov[3];
  int32_t oj[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    bool take_a = (ib >= 6) || (ia < 3 && lex_less(v[ia], j[ia], v[ib], j[ib]));
    if (take_a) { ov[k] = v[ia]; oj[k] = j[ia]; ++ia; }
    else { ov[k] = v[ib]; oj[k] = j[ib]; ++ib; }
  }
  Top3 r;
  r.v1 = ov[0]; r.j1 = oj[0]; r.v2 = ov[1]; r.j2 = oj[1]; r.v3 = ov[2];
  return r;
}

__device__ __forceinline__ Top3 top3_shfl(const Top3 &t, int lanemask) {
  Top3 o;
  o.v1 = __shfl_xor_sync(0xffffffffu, t.v1, lanemask);
  o.v2 = __shfl_xor_sync(0xffffffffu, t.v2, lanemask);
  o.v3 = __shfl_xor_sync(0xffffffffu, t.v3, lanemask);
  o.j1 = __shfl_xor_sync(0xffffffffu, t.j1, lanemask);
  o.j2 = __shfl_xor_sync(0xffffffffu, t.j2, lanemask);
  return o;
}

// Decision for one key from its filtered top-3: write the certain argmin, or
// queue the key for the exact double-precision comparison. Keys with two
// candidates fill the queue from the front (amb_count), keys with three or
// more from the back (amb_crowd); each key queues at most once and the queue
// holds one entry per key, so the two ends never meet.
__device__ __forceinline__ void assign_decide(const Top3 &t, int32_t c, float kn,
                                              float cmax, float c2max, float eps,
                                              int32_t s, int64_t row, int32_t *assign_row,
                                              int4 *amb, int32_t *amb_count,
                                              int32_t *amb_crowd, int32_t amb_cap,
                                              int32_t *err) {
  const float beta2 = 2.f * eps * (kn * cmax + c2max);
  // (non-finite keys or centroids leave the filter without a candidate: the
  // id written stays in range and the key goes to the full exact scan)
  const bool valid = t.j1 < c && (c == 1 || t.j2 < c);
  *assign_row = t.j1 < c ? t.j1 : 0;
  if (c == 1 || (valid && t.v2 - t.v1 > beta2)) return;
  // (the tensor-core filter's indices can name another cell only where two
  // values lie within 2^-20 relative of each other, far inside 2^-6 beta)
  const bool crowded = !valid || ((c > 2) && !(t.v3 - t.v1 > beta2 * (1.f + 0x1p-6f)));
  const int slot = atomicAdd(crowded ? amb_crowd : amb_count, 1);
  if (slot < amb_cap)
    amb[crowded ? amb_cap - 1 - slot : slot] = make_int4(s, (int)row, t.j1, t.j2);
  else
    set_err(err, kErrCapacity);
}

// SIMT fp32 filter: CTA = 64 keys x all centroids, 64-centroid tiles.
// Thread (ty, tx) owns keys 4ty..4ty+3 x centroids 4tx..4tx+3 of a tile.
constexpr int kAsTile = 64;
constexpr int kAsThreads = 256;
constexpr int kEsPitch = kAsTile + 1;
constexpr size_t kAsSmem = sizeof(float) * (2 * kHeadDim * kAsTile + kAsTile * kEsPitch + kAsTile + kAsTile);

template <int DT>
__global__ void __launch_bounds__(kAsThreads)
k_assign_simt(const void *keys, int64_t n, int32_t c, const void *cent_op,
              int32_t u_cap, const float *c2, int32_t c_cap, const float *knorm,
              int64_t n_cap, const float *cstat, float eps, int32_t *assign,
              int64_t gs0, int4 *amb, int32_t *amb_count, int32_t *amb_crowd, int32_t amb_cap,
              int32_t *err) {
  extern __shared__ float sm[];
  float *Ks = sm;                               // [128][64] key tile, transposed
  float *Cs = Ks + kHeadDim * kAsTile;          // [128][64] centroid tile, transposed
  float *Es = Cs + kHeadDim * kAsTile;          // [64][65] filtered distances
  float *c2s = Es + kAsTile * kEsPitch;         // [64]
  float *kns = c2s + kAsTile;                   // [64]
  const int s = blockIdx.y;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  const int64_t row0 = (int64_t)blockIdx.x * kAsTile;
  const int64_t gs = gs0 + s;
  const int eb = elem_bytes<DT>();
  // key tile: chunk (col = id % 64, part = id / 64) of 16 bytes
  {
    const int per_row = kHeadDim * eb / 16;  // 16 (bf16) or 32 (fp32) chunks
    for (int id = tid; id < kAsTile * per_row; id += kAsThreads) {
      const int r = id % kAsTile, part = id / kAsTile;
      const int64_t i = row0 + r;
      float vals[8];
      const int ne = 16 / eb;
      if (i < n) {
        const char *src = (const char *)keys + (((int64_t)s * n + i) * kHeadDim) * eb + part * 16;
        uint4 raw = *(const uint4 *)src;
        if constexpr (DT == 1) {
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            vals[2 * e] = __uint_as_float(w[e] << 16);
            vals[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        } else {
          vals[0] = __uint_as_float(raw.x); vals[1] = __uint_as_float(raw.y);
          vals[2] = __uint_as_float(raw.z); vals[3] = __uint_as_float(raw.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) vals[e] = 0.f;
      }
      for (int e = 0; e < ne; ++e) Ks[(part * ne + e) * kAsTile + r] = vals[e];
    }
    if (tid < kAsTile) {
      const int64_t i = row0 + tid;
      kns[tid] = (i < n) ? knorm[(int64_t)s * n_cap + i] : 0.f;
    }
  }
  Top3 top;
  top.v1 = top.v2 = top.v3 = INFINITY;
  top.j1 = top.j2 = 0x7fffffff;
  const int my_r = tid / 4, my_p = tid % 4;  // scan role: key my_r, 16 columns
  const void *cbase = (const char *)cent_op + (gs * u_cap) * (int64_t)kHeadDim * eb;
  for (int j0 = 0; j0 < c; j0 += kAsTile) {
    __syncthreads();
    const int per_row = kHeadDim * eb / 16;
    for (int id = tid; id < kAsTile * per_row; id += kAsThreads) {
      const int r = id % kAsTile, part = id / kAsTile;
      const int j = j0 + r;
      float vals[8];
      const int ne = 16 / eb;
      if (j < c) {
        const char *src = (const char *)cbase + ((int64_t)j * kHeadDim) * eb + part * 16;
        uint4 raw = *(const uint4 *)src;
        if constexpr (DT == 1) {
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            vals[2 * e] = __uint_as_float(w[e] << 16);
            vals[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        } else {
          vals[0] = __uint_as_float(raw.x); vals[1] = __uint_as_float(raw.y);
          vals[2] = __uint_as_float(raw.z); vals[3] = __uint_as_float(raw.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) vals[e] = 0.f;
      }
      for (int e = 0; e < ne; ++e) Cs[(part * ne + e) * kAsTile + r] = vals[e];
    }
    if (tid < kAsTile) c2s[tid] = (j0 + tid < c) ? c2[(int64_t)s * c_cap + j0 + tid] : 0.f;
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int k = 0; k < kHeadDim; ++k) {
      const float4 ka = *(const float4 *)&Ks[k * kAsTile + 4 * ty];
      const float4 cb = *(const float4 *)&Cs[k * kAsTile + 4 * tx];
      const float av[4] = {ka.x, ka.y, ka.z, ka.w};
      const float bv[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        Es[(4 * ty + a) * kEsPitch + 4 * tx + b] = fmaf(-2.f, acc[a][b], c2s[4 * tx + b]);
    __syncthreads();
#pragma unroll 4
    for (int q = 0; q < 16; ++q) {
      const int col = my_p * 16 + q;
      const int j = j0 + col;
      if (j < c) top3_push(top, Es[my_r * kEsPitch + col], j);
    }
  }
  // merge the four column slices of each key (lanes 4r..4r+3 of one warp)
  top = top3_merge(top, top3_shfl(top, 1));
  top = top3_merge(top, top3_shfl(top, 2));
  const int64_t i = row0 + my_r;
  if (my_p == 0 && i < n) {
    assign_decide(top, c, kns[my_r], cstat[2 * s], cstat[2 * s + 1], eps, s, i,
                  &assign[gs * n_cap + i], amb, amb_count, amb_crowd, amb_cap, err);
  }
}

// ---------------------------------------------------------------- tcgen05 distance filter

// Tensor-core filter for bf16 keys: a persistent CTA takes 128-key tiles; per
// tile it streams the centroid operand in 256-row chunks and computes
// k . c~ for all 128 x 256 pairs with tcgen05.mma (bf16 x bf16 -> fp32 in
// TMEM, two accumulators so MMAs of chunk n+1 overlap the epilogue of chunk
// n). Warp 0 issues the TMA loads (128B-swizzled K-major tiles), warp 1 the
// MMAs and owns the tensor memory, warps 2..17 read the accumulators (four
// warps per TMEM lane quadrant, one per 64-column quarter of a chunk), keep
// the two best per 64-column block and fold them, as e_j - |k|^2, into each
// key's best three; the same certified decision as the SIMT filter follows
// (eps covers the tensor-core fp32 accumulation error with a wide margin).
constexpr int kTcM = 128;
constexpr int kTcN = 256;
constexpr int kTcEpiWarps = 16;
constexpr int kTcWarps = 2 + kTcEpiWarps;
constexpr int kTcThreads = kTcWarps * 32;
constexpr uint32_t kTcABytes = kTcM * kHeadDim * 2;  // 32 KB: two 64-column halves of 16 KB
constexpr uint32_t kTcBBytes = kTcN * kHeadDim * 2;  // 64 KB: two halves of 32 KB
// The extra K block of each chunk: a 16-column bf16 tile of ones (A) against
// each centroid's -|c~|^2 / 2 split into a bf16 high part and remainder (B),
// rows of 32 bytes in the 32-byte swizzle
constexpr uint32_t kTcB1Bytes = kTcN * 32;           // 8 KB
constexpr uint32_t kTcA1Bytes = kTcM * 32;           // 4 KB
constexpr size_t kTcSmem = 2 * kTcABytes + 2 * kTcBBytes + 2 * kTcB1Bytes + kTcA1Bytes + 1024;
constexpr uint32_t kTcIdesc = (1u << 4)            // fp32 accumulator
                              | (1u << 7)          // A bf16
                              | (1u << 10)         // B bf16
                              | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
constexpr uint64_t kTcWaitNs = 2000000000ull;
// Filter margin: 2^-13 bounds the tensor-core fp32 accumulation error of a
// 128-term bf16 dot product with a wide safety factor; 2^-15 covers the
// row or column index carried in the low mantissa bits of the maxima
// (2^-20) and the bf16 pair that stands for |c~|^2 / 2 (2^-17 of it).
constexpr float kTcEps = 0x1p-13f + 0x1p-15f;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tc_mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tc_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool tc_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
               : "=r"(ok) : "r"(smem_addr(bar)), "r"(phase) : "memory");
  return ok != 0;
}
// Bounded wait; on timeout it raises the block's abort flag and returns false.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t phase, volatile int *abort) {
  if (tc_try_wait(bar, phase)) return true;
  const uint64_t t0 = gtimer();
  while (!tc_try_wait(bar, phase)) {
    if (*abort || gtimer() - t0 > kTcWaitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)) : "memory");
}
// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 bytes
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}
// The same for the 32-byte-row tiles of the extra K block (32-byte swizzle:
// rows of 32 bytes, 8-row groups 256 bytes apart).
__device__ __forceinline__ uint64_t sw32_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;           // leading byte offset (unused for this layout)
  d |= (uint64_t)(256 >> 4) << 32;  // stride byte offset: 8 rows x 32 bytes
  d |= (uint64_t)1 << 46;           // descriptor version
  d |= (uint64_t)6 << 61;           // 32-byte swizzle
  return d;
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               ::"r"(d_tmem), "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Two IEEE single-precision fused multiply-adds in one instruction.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Index tracking for the tensor-core filter. A row or column maximum of a
// chunk's 8 x 8 grid of values carries its row or column index in the low
// three mantissa bits (a relative change below 2^-20, covered by the filter's
// margin), so the top-2 network keeps the indices without separate
// bookkeeping. The bits are formed with integer multiplies,
// (e >> 3) * 8 + local, with the multipliers 2^29 and 8 passed in at run
// time: the min/max network loads the ALU pipe, and multiplies issue on the
// FMA pipe (measured faster than a single logic operation on the ALU).
__device__ __forceinline__ float pack3_mul(float e, uint32_t local, uint32_t m29, uint32_t m8) {
  return __uint_as_float(__umulhi(__float_as_uint(e), m29) * m8 + local);
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// The two smallest values of a block (c1 <= c2) absorb the pair {q, r}. With
// (m, M) = (min, max)(q, r), the k-th smallest of the union of two sorted
// lists is the minimum over i + j = k of max(a_i, b_j): the smallest is
// min(c1, m) and the second min(c2, max(c1, m), M). Five min/max operations
// per two values.
__device__ __forceinline__ void top2_pair(float &c1, float &c2, float q, float r) {
  const float m = fminf(q, r), M = fmaxf(q, r);
  c2 = min3f(c2, fmaxf(c1, m), M);
  c1 = fminf(c1, m);
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// The mirror image: the two largest values (c1 >= c2) absorb {q, r}.
__device__ __forceinline__ void top2max_pair(float &c1, float &c2, float q, float r) {
  const float M = fmaxf(q, r), m = fminf(q, r);
  c2 = max3f(c2, fminf(c1, M), m);
  c1 = fmaxf(c1, M);
}
// Merge of two candidate lists with explicit column ids. The first two
// entries of each list are exact; the third may be a lower bound of the
// list's third smallest value, and the merged third is then a lower bound
// too (it is a non-decreasing function of the inputs).
__device__ __forceinline__ Top3 top3_union(const Top3 &a, const Top3 &b) {
  Top3 r;
  const bool bw = b.v1 < a.v1;
  r.v1 = bw ? b.v1 : a.v1;
  r.j1 = bw ? b.j1 : a.j1;
  float x = bw ? a.v1 : b.v1;
  int32_t jx = bw ? a.j1 : b.j1;
  if (a.v2 < x) { x = a.v2; jx = a.j2; }
  if (b.v2 < x) { x = b.v2; jx = b.j2; }
  r.v2 = x;
  r.j2 = jx;
  r.v3 = min3f(a.v3, b.v3, fminf(fmaxf(a.v1, b.v2), fmaxf(a.v2, b.v1)));
  return r;
}

// 16 columns of the thread's TMEM lane, without waiting for them: the
// registers are valid after tc_wait_ld16 on the same array, which names them
// as read-write operands so that the compiler cannot use them earlier.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_assign_tc(const __grid_constant__ CUtensorMap keys_map, const __grid_constant__ CUtensorMap cent_map,
            const __grid_constant__ CUtensorMap c2b_map, int64_t n, int32_t c, int32_t u_cap, const float *knorm,
            int64_t n_cap, const float *cstat, float eps, int32_t *assign, int64_t gs0, int n_slices,
            int4 *amb, int32_t *amb_count, int32_t *amb_crowd, int32_t amb_cap, int32_t *err,
            uint32_t m29, uint32_t m8) {
  extern __shared__ unsigned char tc_smem_raw[];
  __shared__ __align__(8) uint64_t a_full[2], a_empty[2], b_full[2], b_empty[2], acc_full[2], acc_empty[2];
  __shared__ __align__(8) uint64_t mma_done;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ float xv[3][kTcM][3];
  __shared__ int32_t xj[3][kTcM][2];
  const uint32_t base = (smem_addr(tc_smem_raw) + 1023u) & ~1023u;
  const uint32_t A0 = base, B0 = base + 2 * kTcABytes;
  const uint32_t B1 = B0 + 2 * kTcBBytes, A1 = B1 + 2 * kTcB1Bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (int)((n + kTcM - 1) / kTcM);
  const int n_items = n_slices * tiles;
  const int nch = (c + kTcN - 1) / kTcN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc_mbar_init(&a_full[i], 1);
      tc_mbar_init(&a_empty[i], 1);
      tc_mbar_init(&b_full[i], 1);
      tc_mbar_init(&b_empty[i], 1);
      tc_mbar_init(&acc_full[i], 1);
      tc_mbar_init(&acc_empty[i], kTcEpiWarps);
    }
    tc_mbar_init(&mma_done, 1);
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the ones of the extra K block (every element 1.0 in bf16; the layout
  // does not matter), made visible to the tensor cores' async proxy
  {
    uint32_t *a1 = reinterpret_cast<uint32_t *>(tc_smem_raw + (A1 - smem_addr(tc_smem_raw)));
    for (int x = threadIdx.x; x < (int)(kTcA1Bytes / 4); x += blockDim.x) a1[x] = 0x3f803f80u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // tensor memory: two 128 x 256 fp32 accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(&tmem_base_s)), "r"(2 * kTcN) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int it = 0, gc = 0;
      int a_last[2] = {-1, -1}, b_last[2] = {-1, -1};  // last fill count issued per stage
      for (int item = blockIdx.x; item < n_items && !abort_s; item += gridDim.x, ++it) {
        const int sl = item / tiles;
        const int64_t m0 = (int64_t)(item % tiles) * kTcM;
        const int ai = it & 1;
        if (!tc_wait(&a_empty[ai], ((it >> 1) & 1) ^ 1, &abort_s)) break;
        tc_expect_tx(&a_full[ai], kTcABytes);
        const int ya = (int)(sl * n + m0);
        tma_load_2d(A0 + ai * kTcABytes, &keys_map, 0, ya, &a_full[ai]);
        tma_load_2d(A0 + ai * kTcABytes + kTcABytes / 2, &keys_map, 64, ya, &a_full[ai]);
        a_last[ai] = it;
        for (int ch = 0; ch < nch; ++ch, ++gc) {
          const int bi = gc & 1;
          if (!tc_wait(&b_empty[bi], ((gc >> 1) & 1) ^ 1, &abort_s)) break;
          tc_expect_tx(&b_full[bi], kTcBBytes + kTcB1Bytes);
          // rows past the slice's table read as zeros
          const int zb = (int)(gs0 + sl);
          tma_load_3d(B0 + bi * kTcBBytes, &cent_map, 0, ch * kTcN, zb, &b_full[bi]);
          tma_load_3d(B0 + bi * kTcBBytes + kTcBBytes / 2, &cent_map, 64, ch * kTcN, zb, &b_full[bi]);
          tma_load_3d(B1 + bi * kTcB1Bytes, &c2b_map, 0, ch * kTcN, sl, &b_full[bi]);
          b_last[bi] = gc;
        }
      }
      if (abort_s) {  // let the copies still in flight land before the block exits
        const uint64_t t0 = gtimer();
        for (int i = 0; i < 2; ++i) {
          while (a_last[i] >= 0 && !tc_try_wait(&a_full[i], (a_last[i] >> 1) & 1) && gtimer() - t0 < kTcWaitNs) {}
          while (b_last[i] >= 0 && !tc_try_wait(&b_full[i], (b_last[i] >> 1) & 1) && gtimer() - t0 < kTcWaitNs) {}
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int it = 0, gc = 0;
      for (int item = blockIdx.x; item < n_items && !abort_s; item += gridDim.x, ++it) {
        const int ai = it & 1;
        if (!tc_wait(&a_full[ai], (it >> 1) & 1, &abort_s)) break;
        tc_fence_after();
        for (int ch = 0; ch < nch; ++ch, ++gc) {
          const int bi = gc & 1, ti = gc & 1;
          if (!tc_wait(&b_full[bi], (gc >> 1) & 1, &abort_s)) break;
          if (!tc_wait(&acc_empty[ti], ((gc >> 1) & 1) ^ 1, &abort_s)) break;
          tc_fence_after();
          const uint32_t d = tmem + ti * kTcN;
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t ao = A0 + ai * kTcABytes + (k >> 2) * (kTcABytes / 2) + (k & 3) * 32;
            const uint32_t bo = B0 + bi * kTcBBytes + (k >> 2) * (kTcBBytes / 2) + (k & 3) * 32;
            tc_mma(d, sw128_desc(ao), sw128_desc(bo), k > 0 ? 1u : 0u);
          }
          // + ones . (-|c~|^2 / 2): the accumulator holds k.c~ - |c~|^2 / 2,
          // which is (|k|^2 - e) / 2 for the squared distance e
          tc_mma(d, sw32_desc(A1), sw32_desc(B1 + bi * kTcB1Bytes), 1u);
          tc_commit(&b_empty[bi]);
          tc_commit(&acc_full[ti]);
        }
        tc_commit(&a_empty[ai]);
      }
      // every MMA of this block has completed before the tensor memory is freed
      tc_commit(&mma_done);
      const uint64_t t0 = gtimer();
      while (!tc_try_wait(&mma_done, 0) && gtimer() - t0 < kTcWaitNs) {}
    }
  } else {  // epilogue: warps 2..17
    const int quad = warp & 3, qtr = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + qtr * 64;
    int gc = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int sl = item / tiles;
      const int64_t i = (int64_t)(item % tiles) * kTcM + row;
      const float kn = (i < n) ? knorm[(int64_t)sl * n_cap + i] : 0.f;
      Top3 top;
      top.v1 = top.v2 = top.v3 = INFINITY;
      top.j1 = top.j2 = 0x7fffffff;
      for (int ch = 0; ch < nch; ++ch, ++gc) {
        const int ti = gc & 1;
        // the two largest of this chunk's 64 values k.c~ - |c~|^2 / 2. The
        // values form an 8 x 8 grid (row = 8 consecutive columns) with row
        // maxima R and column maxima Cm, taken on the raw values. The largest
        // value M is max R, at (row of max R, column of max Cm). The second
        // largest x2 is exactly max(second of R, second of Cm): in another
        // row than M it is that row's maximum and sits in M's column unless
        // it is also its own column's maximum; in M's row it is its column's
        // maximum. Only the 16 maxima carry their row or column index (low
        // three mantissa bits, a relative change below 2^-20, inside the
        // filter's margin). Where two values of the chunk lie within that
        // change of each other the indices may name another cell; such a
        // key's two best values are then within the margin, so it is not
        // certified, and its chunk's second value, standing in for the
        // third, sends it to the full exact scan. The columns come in four
        // groups of 16 (two grid rows), the TMEM load of the next group in
        // flight while the current one is reduced.
        float R[8], Cm[8];
        uint32_t ra[16], rb[16];
        if (!abort_s) tc_wait(&acc_full[ti], (gc >> 1) & 1, &abort_s);
        __syncwarp();
        tc_fence_after();
        const uint32_t tacc = tbase + ti * kTcN;
        tmem_ld16_async(tacc, ra);
        auto group = [&](const uint32_t(&r)[16], int g) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float a0 = __uint_as_float(r[c]), a1 = __uint_as_float(r[8 + c]);
            Cm[c] = g == 0 ? fmaxf(a0, a1) : max3f(Cm[c], a0, a1);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t *y = r + 8 * h;
            R[2 * g + h] = max3f(max3f(__uint_as_float(y[0]), __uint_as_float(y[1]), __uint_as_float(y[2])),
                                 max3f(__uint_as_float(y[3]), __uint_as_float(y[4]), __uint_as_float(y[5])),
                                 fmaxf(__uint_as_float(y[6]), __uint_as_float(y[7])));
          }
        };
        tc_wait_ld16(ra);
        tmem_ld16_async(tacc + 16, rb);
        group(ra, 0);
        tc_wait_ld16(rb);
        tmem_ld16_async(tacc + 32, ra);
        group(rb, 1);
        tc_wait_ld16(ra);
        tmem_ld16_async(tacc + 48, rb);
        group(ra, 2);
        tc_wait_ld16(rb);
        group(rb, 3);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) tc_arrive(&acc_empty[ti]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          R[k] = pack3_mul(R[k], k, m29, m8);
          Cm[k] = pack3_mul(Cm[k], k, m29, m8);
        }
        // the two largest of R and of Cm (pairwise: the first pair seeds the
        // list, each further pair is merged into it)
        float r1 = fmaxf(R[0], R[1]), r2 = fminf(R[0], R[1]);
        float c1 = fmaxf(Cm[0], Cm[1]), c2 = fminf(Cm[0], Cm[1]);
#pragma unroll
        for (int k = 2; k < 8; k += 2) {
          top2max_pair(r1, r2, R[k], R[k + 1]);
          top2max_pair(c1, c2, Cm[k], Cm[k + 1]);
        }
        const float q1 = r1, q2 = fmaxf(r2, c2);
        const uint32_t i1 = __float_as_uint(r1) & 7u, k1 = __float_as_uint(c1) & 7u;
        const uint32_t i2r = __float_as_uint(r2) & 7u, k2c = __float_as_uint(c2) & 7u;
        const uint32_t hr = __float_as_uint(r2) >> 3, hc = __float_as_uint(c2) >> 3;
        // x2's cell: (its row, M's column), (M's row, its column), or, when
        // it is both a row and a column maximum, (its row, its column)
        const uint32_t cell2 = hr == hc ? 8u * i2r + k2c : (r2 > c2 ? 8u * i2r + k1 : 8u * i1 + k2c);
        // fold the chunk's two into the running list with column ids, as
        // e - |k|^2 = -2 (k.c~ - |c~|^2 / 2) (exact scaling); the chunk's
        // third smallest is at least p2, so p2 stands in as a lower bound
        // for it (a key is certified to have at most two candidates only
        // when that bound clears the margin)
        const float p1 = -2.f * q1, p2 = -2.f * q2;
        const int jb = ch * kTcN + qtr * 64;
        Top3 cur;
        cur.v1 = p1; cur.v2 = p2; cur.v3 = p2;
        cur.j1 = q1 > -INFINITY ? jb + (int)(8u * i1 + k1) : 0x7fffffff;
        cur.j2 = q2 > -INFINITY ? jb + (int)cell2 : 0x7fffffff;
        top = top3_union(top, cur);
      }
      // merge the four column quarters of each key, then decide
      if (qtr > 0) {
        xv[qtr - 1][row][0] = top.v1; xv[qtr - 1][row][1] = top.v2; xv[qtr - 1][row][2] = top.v3;
        xj[qtr - 1][row][0] = top.j1; xj[qtr - 1][row][1] = top.j2;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kTcEpiWarps * 32) : "memory");
      if (qtr == 0 && i < n) {
        Top3 m = top;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          Top3 o;
          o.v1 = xv[q][row][0]; o.v2 = xv[q][row][1]; o.v3 = xv[q][row][2];
          o.j1 = xj[q][row][0]; o.j2 = xj[q][row][1];
          m = top3_union(m, o);
        }
        assign_decide(m, c, kn, cstat[2 * sl], cstat[2 * sl + 1], eps, sl, i,
                      &assign[(gs0 + sl) * n_cap + i], amb, amb_count, amb_crowd, amb_cap, err);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kTcEpiWarps * 32) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kTcN) : "memory");
  }
  if (threadIdx.x == 0 && abort_s) set_err(err, kErrTimeout);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

// bf16 tensor map over `slices` tables of `rows` rows of 128 elements
// (slices == 0: one 2-D table), boxes of 64 x box_rows with 128-byte swizzle;
// rows outside a table read as zeros.
static bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows,
                     uint64_t slices = 0) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows, (cuuint64_t)slices};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)kHeadDim * 2 * rows};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, slices ? 3 : 2, const_cast<void *>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor map over the filter's -|c~|^2 / 2 rows: `slices` tables of
// `rows` rows of 16 elements, boxes of 16 x 256 with 32-byte swizzle.
static bool make_c2b_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t slices) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {16, (cuuint64_t)rows, (cuuint64_t)slices};
  const cuuint64_t strides[2] = {32, 32 * rows};
  const cuuint32_t box[3] = {16, (cuuint32_t)kTcN, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Exact settlement of the queued keys: warp per entry.
template <int DT>
__device__ __forceinline__ double sqdist64(const void *key_row, const void *cent_row) {
  double acc = 0.0;
  for (int j = 0; j < kHeadDim; ++j) {
    const double diff = __dsub_rn((double)load_elem<DT>(key_row, j),
                                  (double)load_elem<DT>(cent_row, j));
    acc = __dadd_rn(acc, __dmul_rn(diff, diff));
  }
  return acc;
}

// Single-precision squared distances of one key to centroids j0..j0+31 by a
// warp: lane l holds key dimensions 4l..4l+3, forms its partial sums for all
// 32 centroids, and a butterfly transpose-reduction leaves centroid j0 + l's
// total in lane l (+inf past the last centroid).
template <int DT>
__device__ __forceinline__ float scan32(const float (&k4)[4], const char *cb, int j0, int c,
                                        int lane) {
  constexpr int eb = DT == 1 ? 2 : 4;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int j = j0 + i;
    if (j < c) {
      const char *row = cb + ((int64_t)j * kHeadDim + lane * 4) * eb;
      float cv[4];
      if constexpr (DT == 1) {
        const uint2 u = __ldg((const uint2 *)row);
        cv[0] = __uint_as_float(u.x << 16); cv[1] = __uint_as_float(u.x & 0xffff0000u);
        cv[2] = __uint_as_float(u.y << 16); cv[3] = __uint_as_float(u.y & 0xffff0000u);
      } else {
        const float4 f = __ldg((const float4 *)row);
        cv[0] = f.x; cv[1] = f.y; cv[2] = f.z; cv[3] = f.w;
      }
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float d = k4[t] - cv[t];
        acc = fmaf(d, d, acc);
      }
      v[i] = acc;
    } else {
      v[i] = INFINITY;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = lane & off;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Keys with two candidates: a lane pair per queue entry, 16 entries per warp;
// the two exact distances are computed by the pair's two lanes (each
// sequentially over the dimensions, the oracle's order), the smaller wins,
// the lower id on a tie. (The double-precision unit runs a warp instruction
// at a time whatever its active lanes, so every lane carries a distance.)
template <int DT>
__global__ void k_refine_pairs(const void *keys, int64_t n, const void *cent_op, int32_t u_cap,
                               int32_t *assign, int64_t n_cap, int64_t gs0, const int4 *amb,
                               const int32_t *amb_count, int32_t amb_cap, int64_t *n_refined) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int total = min(*amb_count, amb_cap);
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd((unsigned long long *)n_refined, (unsigned long long)total);
  const int eb = elem_bytes<DT>();
  for (int64_t w = w0; w * 16 < total; w += warps) {
    const int64_t q = w * 16 + (lane >> 1);
    const bool on = q < total;
    double best = INFINITY;
    int32_t bj = 0x7fffffff;
    int64_t gs = 0, row = 0;
    if (on) {
      const int4 e = amb[q];
      gs = gs0 + e.x;
      row = e.y;
      const char *key_row = (const char *)keys + ((int64_t)e.x * n + row) * kHeadDim * eb;
      const char *cb = (const char *)cent_op + gs * u_cap * (int64_t)kHeadDim * eb;
      bj = (lane & 1) ? e.w : e.z;
      best = sqdist64<DT>(key_row, cb + (int64_t)bj * kHeadDim * eb);
    }
    const double ob = __shfl_xor_sync(0xffffffffu, best, 1);
    const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, 1);
    if (ob < best || (ob == best && oj < bj)) bj = oj;
    if (on && (lane & 1) == 0) assign[gs * n_cap + row] = bj;
  }
}

// Keys with three or more candidates within the filter's margin: a CTA per
// queue entry. A single-precision pass over all centroids (each warp a
// stripe of 32-centroid blocks) bounds every squared distance D_j: each term
// (k_i - c_i)^2 takes one rounding of the difference and one FMA, and a sum
// of 128 non-negative terms in any order lies within 2^-16 * D_j of the true
// value. The true argmin is therefore among the centroids whose
// single-precision distance is within a factor 1 + 2^-13 of the smallest one
// (plus 2^-100 for underflowing terms); only those get the exact distance.
constexpr int kCrowdThreads = 256;
constexpr int kCrowdCand = 1024;  // candidates compacted per entry (more: the per-thread scan)

template <int DT>
__global__ void __launch_bounds__(kCrowdThreads)
k_refine_crowded(const void *keys, int64_t n, int32_t c, const void *cent_op, int32_t u_cap,
                 int32_t *assign, int64_t n_cap, int64_t gs0, const int4 *amb,
                 const int32_t *amb_crowd, int32_t amb_cap, int64_t *n_refined) {
  extern __shared__ float d32[];  // [c]
  __shared__ int32_t cand[kCrowdCand];
  __shared__ int s_nc;
  __shared__ float wmin[kCrowdThreads / 32];
  __shared__ double wbest[kCrowdThreads / 32];
  __shared__ int32_t wj[kCrowdThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int nw = kCrowdThreads / 32;
  const int total = min(*amb_crowd, amb_cap);
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd((unsigned long long *)n_refined, (unsigned long long)total);
  const int eb = elem_bytes<DT>();
  for (int q = blockIdx.x; q < total; q += gridDim.x) {
    const int4 e = amb[amb_cap - 1 - q];
    const int64_t gs = gs0 + e.x;
    const int64_t row = e.y;
    const char *key_row = (const char *)keys + ((int64_t)e.x * n + row) * kHeadDim * eb;
    const char *cb = (const char *)cent_op + gs * u_cap * (int64_t)kHeadDim * eb;
    float k4[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) k4[t] = load_elem<DT>(key_row, lane * 4 + t);
    float m = INFINITY;
    for (int j0 = wid * 32; j0 < c; j0 += nw * 32) {
      const float dj = scan32<DT>(k4, cb, j0, c, lane);
      if (j0 + lane < c) d32[j0 + lane] = dj;
      m = fminf(m, dj);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) wmin[wid] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < nw; ++w) m = fminf(m, wmin[w]);
    const float thr = fmaf(m, 0x1p-13f, m) + 0x1p-100f;
    // the candidates, compacted into adjacent threads (the double-precision
    // unit runs a warp instruction at a time whatever its active lanes)
    if (threadIdx.x == 0) s_nc = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < c; j += kCrowdThreads)
      if (d32[j] <= thr) {
        const int k = atomicAdd(&s_nc, 1);
        if (k < kCrowdCand) cand[k] = j;
      }
    __syncthreads();
    const int nc = s_nc;
    double best = INFINITY;
    int32_t bj = 0x7fffffff;
    if (nc <= kCrowdCand) {
      for (int i = threadIdx.x; i < nc; i += kCrowdThreads) {
        const int j = cand[i];
        const double d64 = sqdist64<DT>(key_row, cb + (int64_t)j * kHeadDim * eb);
        if (d64 < best || (d64 == best && j < bj)) { best = d64; bj = j; }
      }
    } else {
      for (int j = threadIdx.x; j < c; j += kCrowdThreads) {
        if (d32[j] <= thr) {
          const double d64 = sqdist64<DT>(key_row, cb + (int64_t)j * kHeadDim * eb);
          if (d64 < best) { best = d64; bj = j; }  // ascending j: keeps lowest on ties
        }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, o);
      if (ob < best || (ob == best && oj < bj)) { best = ob; bj = oj; }
    }
    if (lane == 0) { wbest[wid] = best; wj[wid] = bj; }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < nw; ++w)
        if (wbest[w] < best || (wbest[w] == best && wj[w] < bj)) { best = wbest[w]; bj = wj[w]; }
      assign[gs * n_cap + row] = bj < c ? bj : 0;  // (no finite distance: stays in range)
    }
    __syncthreads();
  }
}

// Both settlement kernels for one filter pass.
template <int DT>
static void launch_refine(const void *keys, int64_t n, int32_t c, const void *cent_op,
                          int32_t u_cap, int32_t *assign, int64_t n_cap, int64_t gs0,
                          const int4 *amb, const int32_t *amb_count, const int32_t *amb_crowd,
                          int32_t amb_cap, int64_t *n_refined, cudaStream_t st) {
  k_refine_pairs<DT><<<304, 256, 0, st>>>(keys, n, cent_op, u_cap, assign, n_cap, gs0, amb,
                                          amb_count, amb_cap, n_refined);
  k_refine_crowded<DT><<<608, kCrowdThreads, (size_t)c * sizeof(float), st>>>(
      keys, n, c, cent_op, u_cap, assign, n_cap, gs0, amb, amb_crowd, amb_cap, n_refined);
}

// ---------------------------------------------------------------- stable counting sort

__global__ void k_count_parts(const int32_t *assign, int64_t n, int64_t n_cap,
                              int32_t c, int32_t c_cap, int parts, int64_t gs0,
                              int32_t *cnt_part) {
  extern __shared__ int32_t hist[];
  const int s = blockIdx.y, p = blockIdx.x;
  for (int j = threadIdx.x; j < c; j += blockDim.x) hist[j] = 0;
  __syncthreads();
  const int64_t lo = n * p / parts, hi = n * (p + 1) / parts;
  const int32_t *a = assign + (gs0 + s) * n_cap;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) atomicAdd(&hist[a[i]], 1);
  __syncthreads();
  int32_t *out = cnt_part + ((int64_t)s * kMaxParts + p) * c_cap;
  for (int j = threadIdx.x; j < c; j += blockDim.x) out[j] = hist[j];
}

// Block-wide exclusive scan of one int per thread (blockDim <= 1024).
__device__ __forceinline__ int32_t block_excl_scan(int32_t x, int32_t *warp_tot, int32_t *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int32_t w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) warp_tot[lane] = w;  // inclusive warp prefix
    if (lane == nw - 1 && total) *total = w;
  }
  __syncthreads();
  const int32_t r = inc - x + (wid ? warp_tot[wid - 1] : 0);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024)
k_scan_parts(int32_t c, int32_t c_cap, int parts, int32_t *cnt_part,
             int32_t *count, int32_t *offs) {
  __shared__ int32_t warp_tot[32];
  const int s = blockIdx.x;
  int32_t *cp = cnt_part + (int64_t)s * kMaxParts * c_cap;
  const int per = (c + blockDim.x - 1) / blockDim.x;
  const int j0 = threadIdx.x * per;
  int32_t local = 0;
  for (int k = 0; k < per; ++k) {
    const int j = j0 + k;
    if (j < c) {
      int32_t tot = 0;
      for (int p = 0; p < parts; ++p) tot += cp[(int64_t)p * c_cap + j];
      count[(int64_t)s * c_cap + j] = tot;
      local += tot;
    }
  }
  int32_t run = block_excl_scan(local, warp_tot, nullptr);
  for (int k = 0; k < per; ++k) {
    const int j = j0 + k;
    if (j < c) {
      offs[(int64_t)s * c_cap + j] = run;
      int32_t r2 = run;
      for (int p = 0; p < parts; ++p) {
        const int32_t x = cp[(int64_t)p * c_cap + j];
        cp[(int64_t)p * c_cap + j] = r2;
        r2 += x;
      }
      run = r2;
    }
  }
}

// Each part's tokens are placed by one warp, 32 at a time, in token order:
// equal clusters within a group of 32 are ranked by lane; the part's running
// per-cluster offsets live in shared memory.
__global__ void k_scatter(const int32_t *assign, int64_t n, int64_t n_cap, int32_t c,
                          int32_t c_cap, int parts, int64_t gs0, const int32_t *cnt_part,
                          int32_t *perm) {
  extern __shared__ int32_t off[];
  const int s = blockIdx.y, p = blockIdx.x;
  const int32_t *src = cnt_part + ((int64_t)s * kMaxParts + p) * c_cap;
  for (int j = threadIdx.x; j < c; j += blockDim.x) off[j] = src[j];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int64_t lo = n * p / parts, hi = n * (p + 1) / parts;
  const int32_t *a = assign + (gs0 + s) * n_cap;
  int32_t *pm = perm + (gs0 + s) * n_cap;
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const bool valid = i < hi;
    const int32_t key = valid ? a[i] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(peers) - 1;
    const int rank = __popc(peers & lt);
    int32_t pb = (valid && lane == leader) ? off[key] : 0;
    pb = __shfl_sync(0xffffffffu, pb, leader);
    if (valid) pm[pb + rank] = (int32_t)i;
    __syncwarp();
    if (valid && lane == leader) off[key] = pb + __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------- update

// Warp per cluster, lane per 4 dimensions, members in token order. Members
// are fetched eight at a time (indices first, then the eight key rows) so
// the loads overlap; the sums still take the members in token order. A
// persistent grid whose warps take clusters in turn keeps a long cluster from
// holding up others.
//
// bf16 member sums are formed exactly in 2^-40 fixed point. That is the
// token-order double sum too while every partial sum fits 53 bits. Every
// partial sum is a multiple of 2^(e_min - 134), e_min the smallest biased
// exponent among the nonzero members, and at most the sum of magnitudes A:
// it fits when A < 2^(e_min - 81). A cluster of at most 256 members (each
// below 32, e_min >= 94) always qualifies; a larger one is checked with its
// e_min and a float sum of magnitudes. Any other cluster is summed in
// double precision in token order.
//
// The mean is sum / count rounded to double, then to float. It is formed
// without a double division: with y = RN(1/count), q = RN(sum * y) is
// within an ulp of the quotient, and q + (sum - count q) y rounded once
// (two FMAs, the remainder exact) is the correctly rounded quotient
// (Markstein's theorem on division by a correctly rounded reciprocal).
constexpr int kUpdBatch = 8;
constexpr int kUpdThreads = 256;
constexpr int32_t kUpdExactCount = 256;

template <int DT>
__device__ __forceinline__ void load4(const void *keys, int64_t row, int lane, float (&x)[4],
                                      uint2 &raw) {
  if constexpr (DT == 1) {
    raw = __ldg((const uint2 *)((const uint16_t *)keys + row * kHeadDim + lane * 4));
  } else {
    const float4 f = __ldg((const float4 *)((const float *)keys + row * kHeadDim + lane * 4));
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
  }
}

// RN(1/count) for the counts of the fast path, rounded once by the compiler's
// IEEE division at compile time (a warp-uniform constant-memory read instead
// of a double-precision reciprocal per cluster)
struct RcpTable {
  double v[kUpdExactCount + 1];
  constexpr RcpTable() : v() {
    for (int i = 1; i <= kUpdExactCount; ++i) v[i] = 1.0 / i;
  }
};
__constant__ RcpTable c_rcp = RcpTable();

__device__ __forceinline__ float mean_rn(double sum, double cnt, double y) {
  const double q = __dmul_rn(sum, y);
  const double r = __fma_rn(-q, cnt, sum);
  return __double2float_rn(__fma_rn(r, y, q));
}

// Fast exact accumulation of one bf16 value (the low 16 bits of b) in 2^-35
// fixed point: v * 2^35 = +-(128 + m) << (e - 99) for biased exponents
// 99..131 (2^-28 <= |v| < 32), a shift of at most 32, so the 64-bit value
// is one 32-bit shift (lo) and one funnel shift (hi, the sign-extended
// mantissa's upper word). A nonzero value outside that range sets *oor
// (the caller then takes the 2^-40 path) and adds nothing.
__device__ __forceinline__ void fixed35_add(uint32_t b, int64_t &acc, int &oor) {
  const uint32_t e = (b >> 7) & 0xffu;
  const uint32_t sh = e - 99u;
  const bool in = sh <= 32u;
  if (!in && (b & 0x7fffu) != 0u) oor = 1;
  const int32_t m = in ? (int32_t)((b & 0x7fu) | 0x80u) : 0;
  const int32_t ms = (b & 0x8000u) ? -m : m;
  const uint32_t sx = (uint32_t)(ms >> 31);
  uint32_t lo, hi;
  asm("shl.b32 %0, %1, %2;" : "=r"(lo) : "r"((uint32_t)ms), "r"(sh));
  asm("shf.l.clamp.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"((uint32_t)ms), "r"(sx), "r"(sh));
  acc += (int64_t)(((uint64_t)hi << 32) | lo);
}

// fixed35_add over a cluster of at most kUpdExactCount members
__device__ __forceinline__ void fixed35_sums(const void *keys, const int32_t *pm, int32_t cnt, int64_t row0,
                                             int lane, int64_t (&acc)[4], int &oor) {
  int32_t mine = lane < min(kUpdBatch, cnt) ? __ldg(pm + lane) : 0;
  for (int32_t m0 = 0; m0 < cnt; m0 += kUpdBatch) {
    const int nb = min(kUpdBatch, cnt - m0);
    uint2 raw[kUpdBatch];
    float unused[4];
#pragma unroll
    for (int b = 0; b < kUpdBatch; ++b) {
      const int32_t i = __shfl_sync(0xffffffffu, mine, b);
      if (b < nb) load4<1>(keys, row0 + i, lane, unused, raw[b]);
    }
    // the next batch: its member ids now, its rows into L2 while this batch
    // is summed (lane b takes both 128-byte halves of row b)
    const int nb1 = min(kUpdBatch, cnt - m0 - kUpdBatch);
    const int32_t next = lane < nb1 ? __ldg(pm + m0 + kUpdBatch + lane) : 0;
    if (lane < nb1) {
      const char *p = (const char *)keys + (row0 + next) * (int64_t)(kHeadDim * 2);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128));
    }
#pragma unroll
    for (int b = 0; b < kUpdBatch; ++b) {
      if (b < nb) {
        fixed35_add(raw[b].x & 0xffffu, acc[0], oor);
        fixed35_add(raw[b].x >> 16, acc[1], oor);
        fixed35_add(raw[b].y & 0xffffu, acc[2], oor);
        fixed35_add(raw[b].y >> 16, acc[3], oor);
      }
    }
    mine = next;
  }
}

__device__ __forceinline__ uint32_t bf16_exp_nz(uint32_t bits16) {
  const uint32_t e = (bits16 >> 7) & 0xffu;
  return (bits16 & 0x7fffu) ? e : 255u;  // zeros do not set the grid
}

// Exact fixed-point sums of a cluster's bf16 members (this lane's four
// dimensions); big (warp-uniform): also the smallest biased exponent of the
// nonzero members and the float sum of magnitudes.
__device__ __noinline__ void fixed_sums(const void *keys, const int32_t *pm, int32_t cnt, int64_t row0,
                                           int lane, bool big, int64_t (&acc)[4], int &oor, uint32_t &e_min,
                                           float &asum) {
  for (int32_t m0 = 0; m0 < cnt; m0 += kUpdBatch) {
    const int nb = min(kUpdBatch, cnt - m0);
    const int32_t mine = lane < nb ? __ldg(pm + m0 + lane) : 0;
    uint2 raw[kUpdBatch];
    float unused[4];
#pragma unroll
    for (int b = 0; b < kUpdBatch; ++b) {
      const int32_t i = __shfl_sync(0xffffffffu, mine, b);
      if (b < nb) load4<1>(keys, row0 + i, lane, unused, raw[b]);
    }
#pragma unroll
    for (int b = 0; b < kUpdBatch; ++b) {
      if (b < nb) {
        acc[0] += bf16_fixed40((uint16_t)(raw[b].x & 0xffffu), &oor);
        acc[1] += bf16_fixed40((uint16_t)(raw[b].x >> 16), &oor);
        acc[2] += bf16_fixed40((uint16_t)(raw[b].y & 0xffffu), &oor);
        acc[3] += bf16_fixed40((uint16_t)(raw[b].y >> 16), &oor);
        if (big) {
          e_min = min(e_min, min(min(bf16_exp_nz(raw[b].x), bf16_exp_nz(raw[b].x >> 16)),
                                 min(bf16_exp_nz(raw[b].y), bf16_exp_nz(raw[b].y >> 16))));
          asum += (__uint_as_float((raw[b].x & 0x7fffu) << 16) + __uint_as_float((raw[b].x >> 16 & 0x7fffu) << 16)) +
                  (__uint_as_float((raw[b].y & 0x7fffu) << 16) + __uint_as_float((raw[b].y >> 16 & 0x7fffu) << 16));
        }
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kUpdThreads, 2) k_update(const void *keys, int64_t n, int64_t n_cap, int32_t c,
                         int32_t c_cap, int32_t u_cap, int64_t gs0, const int32_t *perm,
                         const int32_t *count, const int32_t *offs, float *cent32,
                         int64_t *n_inexact, int n_slices) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w < (int64_t)n_slices * c;
       w += nwarps) {
  const int s = (int)(w / c), j = (int)(w % c);
  const int32_t cnt = count[(int64_t)s * c_cap + j];
  if (cnt == 0) continue;  // empty cluster keeps its centroid
  const int32_t base = offs[(int64_t)s * c_cap + j];
  const int64_t gs = gs0 + s;
  const int32_t *pm = perm + gs * n_cap + base;
  const int64_t row0 = (int64_t)s * n;
  const double cd = (double)cnt, y = cnt <= kUpdExactCount ? c_rcp.v[cnt] : __drcp_rn(cd);
  double sum[4] = {0.0, 0.0, 0.0, 0.0};
  bool slow = (DT == 0);
  if constexpr (DT == 1) {
    int64_t acc[4] = {0, 0, 0, 0};
    int oor = 0;
    uint32_t e_min = 255u;
    float asum = 0.f;
    const bool big = cnt > kUpdExactCount;
    // small clusters: the 2^-35 path first, the 2^-40 path if a member lies
    // below its range
    bool done = false;
    if (!big) {
      int oor35 = 0;
      fixed35_sums(keys, pm, cnt, row0, lane, acc, oor35);
      done = __any_sync(0xffffffffu, oor35) == 0;
      if (done) {
        // the mean of the 2^-35 sum with the scale folded into the
        // reciprocal and the count (both exact): q = RN(S y 2^-35), then
        // q + (S - count 2^35 q) y 2^-35, the same correctly rounded value
        const double y35 = y * 0x1p-35, c35 = cd * 0x1p35;
        float mf[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const double sd = __ll2double_rn(acc[e]);
          const double q = __dmul_rn(sd, y35);
          mf[e] = __double2float_rn(__fma_rn(__fma_rn(-q, c35, sd), y35, q));
        }
        *(float4 *)(cent32 + (gs * u_cap + j) * kHeadDim + lane * 4) = make_float4(mf[0], mf[1], mf[2], mf[3]);
        continue;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = 0;
      }
    }
    if (!done) fixed_sums(keys, pm, cnt, row0, lane, big, acc, oor, e_min, asum);
    if (!done && big && e_min < 255u) {
      // the float sum of 4 cnt magnitudes is at least (1 - 4 cnt 2^-24) A,
      // so at least 7/8 A for cnt < 2^19: below 7/8 of the limit, A is
      // below the limit
      const float lim = __uint_as_float((e_min - 81u + 127u) << 23) * 0.875f;
      if (!(asum < lim) || cnt >= (1 << 19)) oor = 1;
    }
    slow = __any_sync(0xffffffffu, oor) != 0;
    if (!slow) {
      if (!done) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sum[e] = fixed40_to_double(acc[e]);
      }
    } else if (lane == 0) {
      atomicAdd((unsigned long long *)n_inexact, 1ull);
    }
  }
  if (slow) {  // double-precision sums in token order
    for (int32_t m0 = 0; m0 < cnt; m0 += kUpdBatch) {
      const int nb = min(kUpdBatch, cnt - m0);
      const int32_t mine = lane < nb ? __ldg(pm + m0 + lane) : 0;
      if constexpr (DT == 1) {
        uint2 raw[kUpdBatch];
        float unused[4];
#pragma unroll
        for (int b = 0; b < kUpdBatch; ++b) {
          const int32_t i = __shfl_sync(0xffffffffu, mine, b);
          if (b < nb) load4<DT>(keys, row0 + i, lane, unused, raw[b]);
        }
#pragma unroll
        for (int b = 0; b < kUpdBatch; ++b) {
          if (b < nb) {
            sum[0] = __dadd_rn(sum[0], (double)__uint_as_float(raw[b].x << 16));
            sum[1] = __dadd_rn(sum[1], (double)__uint_as_float(raw[b].x & 0xffff0000u));
            sum[2] = __dadd_rn(sum[2], (double)__uint_as_float(raw[b].y << 16));
            sum[3] = __dadd_rn(sum[3], (double)__uint_as_float(raw[b].y & 0xffff0000u));
          }
        }
      } else {
        float4 x[kUpdBatch];
#pragma unroll
        for (int b = 0; b < kUpdBatch; ++b) {
          const int32_t i = __shfl_sync(0xffffffffu, mine, b);
          if (b < nb) x[b] = __ldg((const float4 *)((const float *)keys + (row0 + i) * kHeadDim + lane * 4));
        }
#pragma unroll
        for (int b = 0; b < kUpdBatch; ++b) {
          if (b < nb) {
            sum[0] = __dadd_rn(sum[0], (double)x[b].x);
            sum[1] = __dadd_rn(sum[1], (double)x[b].y);
            sum[2] = __dadd_rn(sum[2], (double)x[b].z);
            sum[3] = __dadd_rn(sum[3], (double)x[b].w);
          }
        }
      }
    }
  }
  float *dst = cent32 + (gs * u_cap + j) * kHeadDim + lane * 4;
  *(float4 *)dst = make_float4(mean_rn(sum[0], cd, y), mean_rn(sum[1], cd, y), mean_rn(sum[2], cd, y),
                               mean_rn(sum[3], cd, y));
  }
}

// Resident blocks of the update on this device (its persistent grid).
template <int DT>
static int update_grid() {
  static int grid[2] = {0, 0};
  if (!grid[DT]) {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_update<DT>, kUpdThreads, 0);
    grid[DT] = (sms > 0 ? sms : 1) * (per > 0 ? per : 1);
  }
  return grid[DT];
}

// ---------------------------------------------------------------- pool

// Warp per pool row: row pos of slice s receives token perm[pos].
template <int DT>
__global__ void k_pool_build(const void *keys, const void *values, int64_t n, int64_t n_cap,
                             int64_t gs0, const int32_t *perm, void *pool_k, void *pool_v,
                             int64_t pool_rows) {
  const int s = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t pos = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (pos >= n) return;
  const int64_t gs = gs0 + s;
  const int64_t i = perm[gs * n_cap + pos];
  constexpr int row_bytes = kHeadDim * elem_bytes<DT>();
  constexpr int chunks = row_bytes / 16;
  if (lane < chunks) {
    const uint4 *ks = (const uint4 *)((const char *)keys + ((int64_t)s * n + i) * row_bytes) + lane;
    const uint4 *vs = (const uint4 *)((const char *)values + ((int64_t)s * n + i) * row_bytes) + lane;
    uint4 *kd = (uint4 *)((char *)pool_k + (gs * pool_rows + pos) * row_bytes) + lane;
    uint4 *vd = (uint4 *)((char *)pool_v + (gs * pool_rows + pos) * row_bytes) + lane;
    *kd = *ks;
    *vd = *vs;
  }
}

__global__ void k_unit_table(int32_t c, int32_t c_cap, int32_t u_cap, int64_t gs0,
                             const int32_t *count, const int32_t *offs, int32_t *unit_row,
                             int32_t *unit_len) {
  const int s = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= c) return;
  unit_row[(gs0 + s) * u_cap + j] = offs[(int64_t)s * c_cap + j];
  unit_len[(gs0 + s) * u_cap + j] = count[(int64_t)s * c_cap + j];
}

// Reset of one layer's decode state after a (re)build.
__global__ void k_reset_layer(CtxView v, int layer, int32_t c) {
  const int b = blockIdx.x;
  const int64_t lb = (int64_t)layer * v.B + b;
  if (threadIdx.x == 0) {
    DecState st = {};
    st.n_clusters = c;
    st.n_units = c;
    v.st[lb] = st;
  }
  for (int h = 0; h < v.Hkv; ++h) {
    const int64_t gs = lb * v.Hkv + h;
    for (int k = threadIdx.x; k < kHeadDim; k += blockDim.x) v.segsum[gs * kHeadDim + k] = 0;
    if (threadIdx.x == 0) {
      for (int p = 0; p < v.plan_ring; ++p) {  // every plan slot starts empty
        *plan_nsel(v, p, gs) = 0;
        *plan_ntok(v, p, gs) = 0;
        if (v.hsel_n)
          for (int g = 0; g < kMaxGroup; ++g) plan_hsel_n(v, p, gs)[g] = plan_hsel_tok(v, p, gs)[g] = 0;
      }
      for (int p = 0; p < kRing; ++p) v.attn_count[p * v.S_all + gs] = 0;
    }
  }
}

// ---------------------------------------------------------------- host driver

static int parts_for(int64_t n) {
  int64_t p = (n + 2047) / 2048;
  return (int)(p < 1 ? 1 : (p > kMaxParts ? kMaxParts : p));
}

template <int DT>
static cudaError_t group_and_pool(const CtxView &v, int layer, const KmeansScratch &ks,
                                  int64_t n, int32_t c, int64_t gs0, int S,
                                  cudaStream_t st, Prof &prof) {
  const int parts = parts_for(n);
  prof.begin(kPKmSort, st, 3);
  const int c_cap = v.u_cap - v.t_cap;
  k_count_parts<<<dim3(parts, S), 256, c * sizeof(int32_t), st>>>(
      v.assign, n, v.n_cap, c, c_cap, parts, gs0, ks.cnt_part);
  k_scan_parts<<<S, 1024, 0, st>>>(c, c_cap, parts, ks.cnt_part, ks.count, ks.offs);
  k_scatter<<<dim3(parts, S), 128, c * sizeof(int32_t), st>>>(
      v.assign, n, v.n_cap, c, c_cap, parts, gs0, ks.cnt_part, v.perm);
  prof.end(st);
  return cudaGetLastError();
}

template <int DT>
static cudaError_t finish_pool(const CtxView &v, int layer, const KmeansScratch &ks,
                               const void *keys, const void *values, int64_t n, int32_t c,
                               int64_t gs0, int S, cudaStream_t st, Prof &prof) {
  const int c_cap = v.u_cap - v.t_cap;
  prof.begin(kPKmPool, st, 3);
  k_pool_build<DT><<<dim3((unsigned)((n + 7) / 8), S), 256, 0, st>>>(
      keys, values, n, v.n_cap, gs0, v.perm, v.pool_k, v.pool_v, v.pool_rows);
  k_unit_table<<<dim3((c + 255) / 256, S), 256, 0, st>>>(c, c_cap, v.u_cap, gs0, ks.count,
                                                         ks.offs, v.unit_row, v.unit_len);
  k_reset_layer<<<v.B, 128, 0, st>>>(v, layer, c);
  prof.end(st);
  return cudaGetLastError();
}

// Dynamic shared-memory limits of the K-means kernels. A kernel attribute
// applies to the current device only, so it is set once per (device, key
// dtype), under a lock, and every return code is checked.
static std::mutex g_km_attr_mu;
static bool g_km_attr_done[64][2] = {};

template <int DT>
static cudaError_t kmeans_kernel_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_km_attr_mu);
  if (g_km_attr_done[dev][DT]) return cudaSuccess;
  e = cudaFuncSetAttribute(k_assign_simt<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAsSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_assign_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_refine_crowded<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
  if (e == cudaSuccess) g_km_attr_done[dev][DT] = true;
  return e;
}

template <int DT>
static cudaError_t kmeans_build_t(const CtxView &v, int layer, const KmeansScratch &ks,
                                  const void *keys, const void *values, int64_t n,
                                  int32_t c, int32_t iters, bool use_tc, cudaStream_t st,
                                  Prof &prof) {
  const int S = v.B * v.Hkv;
  const int64_t gs0 = (int64_t)layer * S;
  const int c_cap = v.u_cap - v.t_cap;
  const int c_pad = (c + kTcN - 1) / kTcN * kTcN;  // |c|^2 table padded with +inf
  const int64_t amb_cap = (int64_t)S * v.n_cap;
  {
    cudaError_t e = kmeans_kernel_attributes<DT>();
    if (e != cudaSuccess) return e;
  }
  // tensor-core filter (bf16 keys): TMA descriptors of the keys and of the
  // whole centroid-operand table, one persistent CTA per SM
  CUtensorMap keys_map, cent_map, c2b_map;
  int tc_grid = 0;
  if (DT == 1 && use_tc) {
    if (!ks.c2b || !make_map(&keys_map, keys, (uint64_t)S * (uint64_t)n, kTcM) ||
        !make_map(&cent_map, v.cent_op, (uint64_t)v.u_cap, kTcN, (uint64_t)(gs0 + S)) ||
        !make_c2b_map(&c2b_map, ks.c2b, (uint64_t)ks.c2_pitch, (uint64_t)S)) {
      use_tc = false;
    } else {
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const int64_t items = (int64_t)S * ((n + kTcM - 1) / kTcM);
      tc_grid = (int)(items < sms ? items : sms);
    }
  } else {
    use_tc = false;
  }
  prof.begin(kPKmInit, st, 2);
  k_init_cent<DT><<<dim3(c, S), kHeadDim, 0, st>>>(keys, n, c, ks.init_idx, v.cent32, gs0, v.u_cap);
  k_key_norms<DT><<<dim3((unsigned)((n + 7) / 8), S), 256, 0, st>>>(keys, n, v.n_cap, ks.knorm);
  prof.end(st);
  const float eps = 0x1p-15f;  // fp32 FMA dot of 128 terms: 2*gamma_128 < 2^-16
  for (int it = 0; it < iters; ++it) {
    prof.begin(kPKmOperand, st);
    cudaMemsetAsync(ks.cstat, 0, sizeof(float) * 2 * S, st);
    launch_prepare<DT>(v, c, c_pad, ks.c2_pitch, gs0, S, ks.c2, ks.cstat, st, use_tc ? ks.c2b : nullptr);
    cudaMemsetAsync(ks.amb_count, 0, 2 * sizeof(int32_t), st);  // both ends of the queue
    prof.end(st);
    prof.begin(use_tc ? kPKmAssignTc : kPKmAssign, st);
    if (use_tc) {
      k_assign_tc<<<tc_grid, kTcThreads, kTcSmem, st>>>(keys_map, cent_map, c2b_map, n, c, v.u_cap,
                                                        ks.knorm, v.n_cap, ks.cstat, kTcEps, v.assign,
                                                        gs0, S, ks.amb, ks.amb_count, ks.amb_count + 1,
                                                        (int32_t)amb_cap, v.err, 1u << 29, 8u);
    } else {
      k_assign_simt<DT><<<dim3((unsigned)((n + kAsTile - 1) / kAsTile), S), kAsThreads, kAsSmem, st>>>(
          keys, n, c, v.cent_op, v.u_cap, ks.c2, ks.c2_pitch, ks.knorm, v.n_cap, ks.cstat, eps,
          v.assign, gs0, ks.amb, ks.amb_count, ks.amb_count + 1, (int32_t)amb_cap, v.err);
    }
    prof.end(st);
    prof.begin(kPKmRefine, st);
    launch_refine<DT>(keys, n, c, v.cent_op, v.u_cap, v.assign, v.n_cap, gs0, ks.amb, ks.amb_count,
                      ks.amb_count + 1, (int32_t)amb_cap, ks.n_refined, st);
    prof.end(st);
    cudaError_t e = group_and_pool<DT>(v, layer, ks, n, c, gs0, S, st, prof);
    if (e != cudaSuccess) return e;
    prof.begin(kPKmUpdate, st);
    k_update<DT><<<update_grid<DT>(), kUpdThreads, 0, st>>>(keys, n, v.n_cap, c, c_cap, v.u_cap, gs0,
                                                           v.perm, ks.count, ks.offs, v.cent32,
                                                           ks.n_inexact, S);
    prof.end(st);
  }
  prof.begin(kPKmOperand, st);
  cudaMemsetAsync(ks.cstat, 0, sizeof(float) * 2 * S, st);
  launch_prepare<DT>(v, c, c_pad, ks.c2_pitch, gs0, S, ks.c2, ks.cstat, st);
  prof.end(st);
  return finish_pool<DT>(v, layer, ks, keys, values, n, c, gs0, S, st, prof);
}

cudaError_t launch_kmeans_build(const CtxView &v, int layer, const KmeansScratch &ks,
                                const void *keys, const void *values, int64_t n, int32_t c,
                                int32_t iters, bool use_tc, cudaStream_t stream, Prof &prof) {
  if (v.dtype == 1) return kmeans_build_t<1>(v, layer, ks, keys, values, n, c, iters, use_tc, stream, prof);
  return kmeans_build_t<0>(v, layer, ks, keys, values, n, c, iters, false, stream, prof);
}

// Teacher-forced index: centroids and assignment given.
template <int DT>
__global__ void k_copy_given(const int32_t *assign_in, const float *cent_in, int64_t n,
                             int32_t c, int64_t n_cap, int32_t u_cap, int64_t gs0,
                             int32_t *assign, float *cent32, int32_t *err) {
  const int s = blockIdx.y;
  const int64_t gs = gs0 + s;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int32_t a = assign_in[(int64_t)s * n + i];
    if (a < 0 || a >= c) { set_err(err, kErrInternal); a = 0; }
    assign[gs * n_cap + i] = a;
  }
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < (int64_t)c * kHeadDim;
       k += (int64_t)gridDim.x * blockDim.x)
    cent32[gs * u_cap * kHeadDim + k] = cent_in[(int64_t)s * c * kHeadDim + k];
}

template <int DT>
static cudaError_t load_index_t(const CtxView &v, int layer, const KmeansScratch &ks,
                                const void *keys, const void *values, int64_t n, int32_t c,
                                const int32_t *assign, const float *cent, cudaStream_t st,
                                Prof &prof) {
  const int S = v.B * v.Hkv;
  const int64_t gs0 = (int64_t)layer * S;
  const int c_pad = (c + kTcN - 1) / kTcN * kTcN;
  k_copy_given<DT><<<dim3(64, S), 256, 0, st>>>(assign, cent, n, c, v.n_cap, v.u_cap, gs0,
                                                v.assign, v.cent32, v.err);
  cudaMemsetAsync(ks.cstat, 0, sizeof(float) * 2 * S, st);
  launch_prepare<DT>(v, c, c_pad, ks.c2_pitch, gs0, S, ks.c2, ks.cstat, st);
  cudaError_t e = group_and_pool<DT>(v, layer, ks, n, c, gs0, S, st, prof);
  if (e != cudaSuccess) return e;
  return finish_pool<DT>(v, layer, ks, keys, values, n, c, gs0, S, st, prof);
}

cudaError_t launch_load_index(const CtxView &v, int layer, const KmeansScratch &ks,
                              const void *keys, const void *values, int64_t n, int32_t c,
                              const int32_t *assign, const float *cent, cudaStream_t stream,
                              Prof &prof) {
  if (v.dtype == 1) return load_index_t<1>(v, layer, ks, keys, values, n, c, assign, cent, stream, prof);
  return load_index_t<0>(v, layer, ks, keys, values, n, c, assign, cent, stream, prof);
}

// Page-mean index [CTkvr, 1.1: block-level indexes mean-pool runs of
// consecutive tokens]: token i of every slice is in unit i / page; the units'
// index vectors come from the same exact-sum update as a Lloyd round (every
// page has at least one token, so none keeps a stale value).
__global__ void k_page_assign(int64_t n, int32_t page, int64_t n_cap, int64_t gs0, int32_t *assign) {
  const int64_t gs = gs0 + blockIdx.y;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    assign[gs * n_cap + i] = (int32_t)(i / page);
}

template <int DT>
static cudaError_t page_index_t(const CtxView &v, int layer, const KmeansScratch &ks, const void *keys,
                                const void *values, int64_t n, int32_t page, cudaStream_t st, Prof &prof) {
  const int S = v.B * v.Hkv;
  const int64_t gs0 = (int64_t)layer * S;
  const int c_cap = v.u_cap - v.t_cap;
  const int32_t c = (int32_t)((n + page - 1) / page);
  const int c_pad = (c + kTcN - 1) / kTcN * kTcN;
  {
    cudaError_t e = kmeans_kernel_attributes<DT>();
    if (e != cudaSuccess) return e;
  }
  prof.begin(kPKmInit, st);
  k_page_assign<<<dim3(64, S), 256, 0, st>>>(n, page, v.n_cap, gs0, v.assign);
  prof.end(st);
  cudaError_t e = group_and_pool<DT>(v, layer, ks, n, c, gs0, S, st, prof);
  if (e != cudaSuccess) return e;
  prof.begin(kPKmUpdate, st);
  k_update<DT><<<update_grid<DT>(), kUpdThreads, 0, st>>>(keys, n, v.n_cap, c, c_cap, v.u_cap, gs0, v.perm,
                                                         ks.count, ks.offs, v.cent32, ks.n_inexact, S);
  prof.end(st);
  prof.begin(kPKmOperand, st);
  cudaMemsetAsync(ks.cstat, 0, sizeof(float) * 2 * S, st);
  launch_prepare<DT>(v, c, c_pad, ks.c2_pitch, gs0, S, ks.c2, ks.cstat, st);
  prof.end(st);
  return finish_pool<DT>(v, layer, ks, keys, values, n, c, gs0, S, st, prof);
}

cudaError_t launch_page_index(const CtxView &v, int layer, const KmeansScratch &ks, const void *keys,
                              const void *values, int64_t n, int32_t page, cudaStream_t stream, Prof &prof) {
  if (v.dtype == 1) return page_index_t<1>(v, layer, ks, keys, values, n, page, stream, prof);
  return page_index_t<0>(v, layer, ks, keys, values, n, page, stream, prof);
}

// ---------------------------------------------------------------- allocation-free K-means

// lkv_kmeans_static runs the same K-means as lkv_build_index for one
// (sequence, KV head) slice, but every intermediate buffer lives in the
// fixed array below instead of memory obtained from cudaMalloc. The array is
// part of the library image: each GPU that loads the library holds it until
// the process exits, and all calls on a GPU share it.
constexpr int64_t kStaticMaxTokens = 32768;
constexpr int32_t kStaticMaxClusters = 2048;
constexpr size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kSoKnorm = 0;
constexpr size_t kSoC2 = kSoKnorm + al256(kStaticMaxTokens * 4);
constexpr size_t kSoCstat = kSoC2 + al256(kStaticMaxClusters * 4);
constexpr size_t kSoCntPart = kSoCstat + 256;
constexpr size_t kSoCount = kSoCntPart + al256((size_t)kMaxParts * kStaticMaxClusters * 4);
constexpr size_t kSoOffs = kSoCount + al256(kStaticMaxClusters * 4);
constexpr size_t kSoAmb = kSoOffs + al256(kStaticMaxClusters * 4);
constexpr size_t kSoMisc = kSoAmb + al256(kStaticMaxTokens * sizeof(int4));
// misc: amb_count (int32 at 0), n_refined and n_inexact (int64 at 8, 16),
// amb_crowd (int32 at 24), all cleared by every call; the device error bits
// (int32 at kSoErr) are sticky until lkv_kmeans_static_status reads them
constexpr size_t kSoErr = 128;
constexpr size_t kSoInit = kSoMisc + 256;
constexpr size_t kSoShuffle = kSoInit + al256(kStaticMaxClusters * 8);
constexpr size_t kSoCentOp = kSoShuffle + al256(kStaticMaxTokens * 8);
constexpr size_t kSoPerm = kSoCentOp + al256((size_t)kStaticMaxClusters * kHeadDim * 4);
constexpr size_t kStaticScratchBytes = kSoPerm + al256(kStaticMaxTokens * 4);

static __device__ __align__(256) unsigned char g_kmeans_scratch[kStaticScratchBytes];

__device__ __forceinline__ uint64_t splitmix64_dev(uint64_t &state) {
  uint64_t z = (state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// The initial centroid indices of lkv_build_index (first c entries of a
// splitmix64-driven partial Fisher-Yates shuffle of [0, n)), drawn on the
// device so that no host buffer is needed. One block.
__global__ void k_static_init_indices(int64_t n, int32_t c, uint64_t seed, int64_t *shuffle,
                                      int64_t *idx) {
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) shuffle[i] = i;
  __syncthreads();
  if (threadIdx.x != 0) return;
  uint64_t st = seed;
  for (int32_t i = 0; i < c; ++i) {
    const uint64_t r = splitmix64_dev(st);
    const int64_t j = (int64_t)i + (int64_t)(r % (uint64_t)(n - i));
    const int64_t t = shuffle[i];
    shuffle[i] = shuffle[j];
    shuffle[j] = t;
    idx[i] = shuffle[i];
  }
}

template <int DT>
static cudaError_t kmeans_static_t(unsigned char *base, const void *keys, int64_t n, int32_t c,
                                   int32_t iters, uint64_t seed, float *cent, int32_t *assign,
                                   cudaStream_t st) {
  CtxView v{};
  v.dtype = DT;
  v.B = 1;
  v.Hkv = 1;
  v.n_cap = n;
  v.t_cap = 0;
  v.u_cap = c;
  v.cent32 = cent;
  v.cent_op = base + kSoCentOp;
  v.assign = assign;
  v.perm = (int32_t *)(base + kSoPerm);
  v.err = (int32_t *)(base + kSoMisc + kSoErr);
  KmeansScratch ks{};
  ks.knorm = (float *)(base + kSoKnorm);
  ks.c2 = (float *)(base + kSoC2);
  ks.c2_pitch = c;
  ks.cstat = (float *)(base + kSoCstat);
  ks.cnt_part = (int32_t *)(base + kSoCntPart);
  ks.count = (int32_t *)(base + kSoCount);
  ks.offs = (int32_t *)(base + kSoOffs);
  ks.amb = (int4 *)(base + kSoAmb);
  ks.amb_count = (int32_t *)(base + kSoMisc);
  int32_t *amb_crowd = (int32_t *)(base + kSoMisc + 24);
  ks.n_refined = (int64_t *)(base + kSoMisc + 8);
  ks.n_inexact = (int64_t *)(base + kSoMisc + 16);
  ks.init_idx = (int64_t *)(base + kSoInit);
  Prof quiet;
  quiet.counting = false;
  const int64_t amb_cap = n;
  const float eps = 0x1p-15f;
  // the array keeps the previous call's contents: clear what must start at
  // zero (the error bits stay until lkv_kmeans_static_status collects them)
  cudaError_t e = cudaMemsetAsync(base + kSoMisc, 0, kSoErr, st);
  if (e != cudaSuccess) return e;
  k_static_init_indices<<<1, 1024, 0, st>>>(n, c, seed, (int64_t *)(base + kSoShuffle), ks.init_idx);
  k_init_cent<DT><<<dim3(c, 1), kHeadDim, 0, st>>>(keys, n, c, ks.init_idx, v.cent32, 0, v.u_cap);
  k_key_norms<DT><<<dim3((unsigned)((n + 7) / 8), 1), 256, 0, st>>>(keys, n, v.n_cap, ks.knorm);
  for (int it = 0; it < iters; ++it) {
    e = cudaMemsetAsync(ks.cstat, 0, sizeof(float) * 2, st);
    if (e != cudaSuccess) return e;
    launch_prepare<DT>(v, c, c, c, 0, 1, ks.c2, ks.cstat, st);
    e = cudaMemsetAsync(ks.amb_count, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(amb_crowd, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    k_assign_simt<DT><<<dim3((unsigned)((n + kAsTile - 1) / kAsTile), 1), kAsThreads, kAsSmem, st>>>(
        keys, n, c, v.cent_op, v.u_cap, ks.c2, c, ks.knorm, v.n_cap, ks.cstat, eps, v.assign, 0,
        ks.amb, ks.amb_count, amb_crowd, (int32_t)amb_cap, v.err);
    launch_refine<DT>(keys, n, c, v.cent_op, v.u_cap, v.assign, v.n_cap, 0, ks.amb, ks.amb_count,
                      amb_crowd, (int32_t)amb_cap, ks.n_refined, st);
    e = group_and_pool<DT>(v, 0, ks, n, c, 0, 1, st, quiet);
    if (e != cudaSuccess) return e;
    k_update<DT><<<update_grid<DT>(), kUpdThreads, 0, st>>>(keys, n, v.n_cap, c, c, v.u_cap, 0, v.perm,
                                                           ks.count, ks.offs, v.cent32, ks.n_inexact, 1);
  }
  return cudaGetLastError();
}

// Per-device address of g_kmeans_scratch. In host code the array's name is
// only a host-side stand-in, so the device address is looked up once per
// device (with that device current) and cached for the life of the process;
// a cudaDeviceReset reloads the module and invalidates the cached address, so
// calls after a reset are not supported.
static std::mutex g_static_mu;
static void *g_static_addr[64] = {};

static cudaError_t static_scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_kmeans_scratch);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_assign_simt<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAsSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_assign_simt<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAsSmem);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

}  // namespace lkv

extern "C" lkv_status lkv_kmeans_static(const void *keys, int32_t dtype, int64_t n_tokens,
                                        int32_t n_clusters, int32_t iters, uint64_t seed,
                                        float *centroids, int32_t *assign, void *stream) {
  using namespace lkv;
  if (!keys || !centroids || !assign) {
    set_unbound_error("lkv_kmeans_static: null keys, centroids or assign");
    return LKV_EINVAL;
  }
  if (dtype != LKV_DTYPE_FP32 && dtype != LKV_DTYPE_BF16) {
    set_unbound_error("lkv_kmeans_static: bad dtype");
    return LKV_EINVAL;
  }
  if (n_tokens < 1 || n_tokens > kStaticMaxTokens) {
    set_unbound_error("lkv_kmeans_static: n_tokens must be 1..32768 (size of the built-in scratch)");
    return LKV_EINVAL;
  }
  if (n_clusters < 1 || n_clusters > kStaticMaxClusters || n_clusters > n_tokens) {
    set_unbound_error("lkv_kmeans_static: n_clusters must be 1..min(2048, n_tokens) "
                      "(size of the built-in scratch)");
    return LKV_EINVAL;
  }
  if (iters < 1) {
    set_unbound_error("lkv_kmeans_static: iters must be >= 1");
    return LKV_EINVAL;
  }
  void *base = nullptr;
  cudaError_t e = static_scratch_address(&base);
  if (e == cudaSuccess) {
    cudaStream_t st = (cudaStream_t)stream;
    e = dtype == LKV_DTYPE_BF16
            ? kmeans_static_t<1>((unsigned char *)base, keys, n_tokens, n_clusters, iters, seed, centroids, assign, st)
            : kmeans_static_t<0>((unsigned char *)base, keys, n_tokens, n_clusters, iters, seed, centroids, assign, st);
  }
  if (e != cudaSuccess) {
    set_unbound_error((std::string("lkv_kmeans_static: ") + cudaGetErrorString(e)).c_str());
    return LKV_ECUDA;
  }
  return LKV_OK;
}

extern "C" lkv_status lkv_kmeans_static_status(void *stream) {
  using namespace lkv;
  void *base = nullptr;
  cudaError_t e = static_scratch_address(&base);
  int32_t bits = 0;
  int32_t *err = (int32_t *)((unsigned char *)base + kSoMisc + kSoErr);
  cudaStream_t st = (cudaStream_t)stream;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&bits, err, sizeof bits, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && bits) e = cudaMemsetAsync(err, 0, sizeof bits, st);
  if (e == cudaSuccess && bits) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    set_unbound_error((std::string("lkv_kmeans_static_status: ") + cudaGetErrorString(e)).c_str());
    return LKV_ECUDA;
  }
  if (bits & kErrTimeout) {
    set_unbound_error("lkv_kmeans_static: a device-side wait gave up");
    return LKV_ETIMEOUT;
  }
  if (bits & kErrCapacity) {
    set_unbound_error("lkv_kmeans_static: the settlement queue of the built-in scratch overflowed");
    return LKV_ECAPACITY;
  }
  if (bits) {
    set_unbound_error("lkv_kmeans_static: a device-side invariant check failed");
    return LKV_ECUDA;
  }
  return LKV_OK;
}
