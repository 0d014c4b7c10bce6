// paris.cuh -- per-key metadata of the ParisKV-style token selector, shared by
// the prefill encoder (paris.cu) and the decode-step append (decode.cu).
//
// ParisKV technical summary, 核心算法创新 1 and 2: keys are normalised and
// rotated by a shared random orthogonal rotation (SRHT), the rotated key is
// split into B subspaces, each subspace direction is assigned to the nearest
// analytic sign centroid (its bucket) and coded with 1 sign bit and 3
// magnitude bits per coordinate against the Beta prior that the rotation
// induces, with a per-subspace scale w that calibrates the dequantised
// direction. Here d = 128, B = 16 subspaces of m = 8 coordinates, and the
// rotation is H diag(D) / sqrt(128) (H the Sylvester-Hadamard matrix, D the
// context's random signs). The rotation is exact: a key's bf16 values are
// taken as integers k * 2^40 (truncated toward zero; exact for the bf16
// values of magnitude 2^-33 .. 2^22), and the Hadamard transform of those
// integers has no rounding, so the buckets and codes do not depend on the
// order of the butterfly.
#pragma once

#include "lkv_internal.cuh"

namespace lkv {

constexpr int kParisSub = 16;      // subspaces B
constexpr int kParisDim = 8;       // coordinates per subspace m
constexpr int kParisMaxRho = 15;   // votes per subspace: a coarse score fits in 8 bits
constexpr int kParisMaxCand = 4096;

// Metadata of one key, computed by one warp: lane L holds coordinates
// 4L .. 4L + 3 of the key (bf16 bits). Writes the 16 bucket bytes (bit j of
// byte b: rotated coordinate 8b + j is negative), the 64 code bytes (byte k:
// magnitude level of coordinate 2k in the low nibble, 2k + 1 in the high one)
// and the 16 scales. thr: the 7 prior thresholds on x^2, lev: the 8 bin means.
__device__ __forceinline__ void paris_encode_warp(const uint16_t *key4, const uint64_t sign[2],
                                                  const float *thr, const float *lev,
                                                  uint8_t *bucket_out, uint8_t *code_out,
                                                  float *w_out) {
  const int lane = threadIdx.x & 31;
  long long y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = 4 * lane + e;
    const double kv = (double)bf16_bits_to_f32(key4[e]);
    long long k40 = __double2ll_rz(kv * 0x1p40);
    if ((sign[j >> 6] >> (j & 63)) & 1ull) k40 = -k40;
    y[e] = k40;
  }
  // fast Walsh-Hadamard transform (Sylvester order), exact in 64-bit integers
  {
    const long long a0 = y[0] + y[1], a1 = y[0] - y[1], a2 = y[2] + y[3], a3 = y[2] - y[3];
    y[0] = a0 + a2;
    y[2] = a0 - a2;
    y[1] = a1 + a3;
    y[3] = a1 - a3;
  }
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {  // stride 4 * hl in coordinates
    const bool upper = (lane & hl) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const long long o = __shfl_xor_sync(0xffffffffu, y[e], hl);
      y[e] = upper ? o - y[e] : y[e] + o;
    }
  }
  // lane b < 16 codes subspace b (coordinates 8b .. 8b + 7: lanes 2b, 2b + 1)
  long long z[8];
  const int src = (2 * lane) & 31;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    z[e] = __shfl_sync(0xffffffffu, y[e], src);
    z[4 + e] = __shfl_sync(0xffffffffu, y[e], src + 1);
  }
  if (lane >= kParisSub) return;
  // (double products and sums in index order, no contraction; the products
  // thr_k * n2 and z_j^2 are formed once and compared, which gives the same
  // values as forming them at every comparison)
  unsigned bits = 0;
  double sq[kParisDim], n2 = 0.0;
#pragma unroll
  for (int j = 0; j < kParisDim; ++j) {
    if (z[j] < 0) bits |= 1u << j;
    sq[j] = __dmul_rn((double)z[j], (double)z[j]);
    n2 = __dadd_rn(n2, sq[j]);
  }
  double tn[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) tn[k] = __dmul_rn((double)thr[k], n2);
  double num = 0.0, den = 0.0;
  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < kParisDim; ++j) {
    int l = 0;
#pragma unroll
    for (int k = 0; k < 7; ++k) l += sq[j] >= tn[k];
    packed |= (uint32_t)l << (4 * j);
    const double vj = z[j] < 0 ? -(double)lev[l] : (double)lev[l];
    num = __dadd_rn(num, __dmul_rn((double)z[j], vj));
    den = __dadd_rn(den, __dmul_rn(vj, vj));
  }
  bucket_out[lane] = (uint8_t)bits;
  reinterpret_cast<uint32_t *>(code_out)[lane] = packed;
  constexpr double kSqrt128 = 0x1.6a09e667f3bcdp+3;  // sqrt(128), correctly rounded
  w_out[lane] = __double2float_rn(__ddiv_rn(__dmul_rn(__ddiv_rn(num, den), 0x1p-40), kSqrt128));
}

}  // namespace lkv
