// paris.cu -- index build of the ParisKV-style token selector: the prior
// tables, the pool in token order and the metadata of every prefill token
// (ParisKV technical summary, 核心算法创新 1-2; the selection itself is in
// decode.cu next to the cluster selection).
#include <cmath>

#include "lkv_internal.cuh"
#include "paris.cuh"

namespace lkv {

// A coordinate x of a uniform unit vector in R^8 has density proportional to
// (1 - x^2)^(5/2). With x = sin(th), the mass of [0, x] is
// G(th) = 5 th / 16 + 15 sin(2 th) / 64 + 3 sin(4 th) / 64 + sin(6 th) / 192
// (the integral of cos^6), and the first moment of [a, b] is
// ((1 - a^2)^(7/2) - (1 - b^2)^(7/2)) / 7.
static double cos6_integral(double th) {
  return 5.0 * th / 16.0 + 15.0 * std::sin(2.0 * th) / 64.0 + 3.0 * std::sin(4.0 * th) / 64.0 +
         std::sin(6.0 * th) / 192.0;
}

void paris_levels_host(float thr[7], float lev[8]) {
  const double pi = 3.14159265358979323846;
  const double total = cos6_integral(pi / 2.0);
  double t[9];
  t[0] = 0.0;
  t[8] = 1.0;
  for (int l = 1; l < 8; ++l) {
    double lo = 0.0, hi = 1.0;  // P(|x| < t) = l / 8
    for (int it = 0; it < 100; ++it) {
      const double mid = 0.5 * (lo + hi);
      if (cos6_integral(std::asin(mid)) / total < l / 8.0) lo = mid;
      else hi = mid;
    }
    t[l] = 0.5 * (lo + hi);
    thr[l - 1] = (float)(t[l] * t[l]);
  }
  for (int l = 0; l < 8; ++l) {
    const double a = t[l], b = t[l + 1];
    const double mass = cos6_integral(std::asin(b)) - cos6_integral(std::asin(a));
    const double moment = (std::pow(1.0 - a * a, 3.5) - std::pow(1.0 - b * b, 3.5)) / 7.0;
    lev[l] = (float)(moment / mass);
  }
}

// Identity pool order: prefill token i at pool row i.
__global__ void k_perm_identity(int64_t n, int64_t n_cap, int64_t gs0, int32_t *perm) {
  const int64_t gs = gs0 + blockIdx.y;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    perm[gs * n_cap + i] = (int32_t)i;
}

// Metadata of every prefill token: one warp per (token, slice).
__global__ void __launch_bounds__(256) k_paris_encode(CtxView v, const uint16_t *keys, int64_t n, int64_t gs0) {
  const int s = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (i >= n) return;
  const int lane = threadIdx.x & 31;
  uint16_t k4[4];
  const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(keys + ((int64_t)s * n + i) * kHeadDim) + lane);
  k4[0] = (uint16_t)(raw.x & 0xffffu);
  k4[1] = (uint16_t)(raw.x >> 16);
  k4[2] = (uint16_t)(raw.y & 0xffffu);
  k4[3] = (uint16_t)(raw.y >> 16);
  const int64_t row = (gs0 + s) * v.pool_rows + i;
  paris_encode_warp(k4, v.paris_sign, v.paris_thr, v.paris_lev, v.pk_bucket + row * kParisSub,
                    v.pk_code + row * 64, v.pk_w + row * kParisSub);
}

// Rows in token order: a warp copies one K row and one V row (16-byte vectors).
__global__ void k_pool_copy(const uint16_t *keys, const uint16_t *values, int64_t n, int64_t gs0, uint16_t *pool_k,
                            uint16_t *pool_v, int64_t pool_rows) {
  const int s = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (i >= n || lane >= 16) return;
  const int64_t src = ((int64_t)s * n + i) * kHeadDim, dst = ((gs0 + s) * pool_rows + i) * kHeadDim;
  reinterpret_cast<uint4 *>(pool_k + dst)[lane] = __ldg(reinterpret_cast<const uint4 *>(keys + src) + lane);
  reinterpret_cast<uint4 *>(pool_v + dst)[lane] = __ldg(reinterpret_cast<const uint4 *>(values + src) + lane);
}

// Reset of one layer's decode state (no clusters: every unit is a segment).
__global__ void k_paris_reset(CtxView v, int layer, int64_t n) {
  const int b = blockIdx.x;
  const int64_t lb = (int64_t)layer * v.B + b;
  if (threadIdx.x == 0) {
    DecState st = {};
    st.n_prefill = (int32_t)n;
    v.st[lb] = st;
  }
  for (int h = 0; h < v.Hkv; ++h) {
    const int64_t gs = lb * v.Hkv + h;
    for (int k = threadIdx.x; k < kHeadDim; k += blockDim.x) v.segsum[gs * kHeadDim + k] = 0;
    if (threadIdx.x == 0) {
      for (int p = 0; p < v.plan_ring; ++p) {
        *plan_nsel(v, p, gs) = 0;
        *plan_ntok(v, p, gs) = 0;
      }
      for (int p = 0; p < kRing; ++p) v.attn_count[p * v.S_all + gs] = 0;
    }
  }
}

cudaError_t launch_paris_index(const CtxView &v, int layer, const KmeansScratch &ks, const void *keys,
                               const void *values, int64_t n, cudaStream_t st, Prof &prof) {
  (void)ks;
  const int S = v.B * v.Hkv;
  const int64_t gs0 = (int64_t)layer * S;
  prof.begin(kPKmPool, st, 4);
  k_perm_identity<<<dim3(64, S), 256, 0, st>>>(n, v.n_cap, gs0, v.perm);
  k_pool_copy<<<dim3((unsigned)((n + 7) / 8), S), 256, 0, st>>>(
      (const uint16_t *)keys, (const uint16_t *)values, n, gs0, (uint16_t *)v.pool_k, (uint16_t *)v.pool_v,
      v.pool_rows);
  k_paris_encode<<<dim3((unsigned)((n + 7) / 8), S), 256, 0, st>>>(v, (const uint16_t *)keys, n, gs0);
  k_paris_reset<<<v.B, 128, 0, st>>>(v, layer, n);
  prof.end(st);
  return cudaGetLastError();
}

}  // namespace lkv
