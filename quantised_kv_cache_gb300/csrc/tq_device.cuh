// Device helpers shared by the libtq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)
constexpr float kSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi / 2)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Orthonormal Sylvester Walsh-Hadamard transform of a 128-vector held by one
// warp, lane L owning coordinates 4L..4L+3 (index bits 0-1 in-lane, bits 2-6
// across lanes). Natural order: y_i = sum_j (-1)^{popcount(i&j)} x_j / sqrt(128).
__device__ __forceinline__ void wht128(float (&v)[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float o = __shfl_xor_sync(kFull, v[j], m);
      v[j] = upper ? (o - v[j]) : (v[j] + o);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] *= kInvSqrtD;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Four consecutive inputs starting at element offset `off` (a multiple of 4).
__device__ __forceinline__ void load4(const void *base, size_t off, bool bf16, float (&v)[4]) {
  if (bf16) {
    uint2 w = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + off));
    v[0] = bf16_bits_to_float(w.x & 0xffffu);
    v[1] = bf16_bits_to_float(w.x >> 16);
    v[2] = bf16_bits_to_float(w.y & 0xffffu);
    v[3] = bf16_bits_to_float(w.y >> 16);
  } else {
    float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off));
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}

__device__ __forceinline__ void set_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// The 4*BITS-bit field holding lane's four codes (coordinates 4L..4L+3) in a
// record of 4*BITS 32-bit words.
template <int BITS>
__device__ __forceinline__ uint32_t lane_code_field(const uint32_t *rec, int lane) {
  constexpr int W = 4 * BITS;
  const int bit = 4 * BITS * lane;
  const int wi = bit >> 5, off = bit & 31;
  uint32_t lo = __ldg(rec + wi);
  if (off + 4 * BITS <= 32) return lo >> off;
  uint32_t hi = __ldg(rec + ((wi + 1 < W) ? wi + 1 : wi));
  return __funnelshift_r(lo, hi, off);
}

// Pack each lane's 4*BITS-bit field into the record's little-endian bit
// string; lanes 0..4*BITS-1 return their 32-bit word.
template <int BITS>
__device__ __forceinline__ uint32_t pack_record_word(uint32_t field, int lane) {
  constexpr int F = 4 * BITS;                    // bits per lane
  constexpr int K = (32 + F - 1) / F + 1;        // lanes touching one word
  const int first = (32 * lane) / F;
  uint32_t word = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int src = first + k;
    uint32_t c = __shfl_sync(kFull, field, src & 31);
    const int shift = F * src - 32 * lane;
    if (src < 32 && shift > -F && shift < 32) word |= (shift >= 0) ? (c << shift) : (c >> (-shift));
  }
  return word;
}

}  // namespace tq
