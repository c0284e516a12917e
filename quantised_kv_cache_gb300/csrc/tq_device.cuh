// Device helpers shared by the libtq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)
constexpr float kSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi / 2)

// Paged caches: the physical slot of virtual slot `vslot` (= sequence-head * cap16 + t).
// Without a block table the two coincide; with one, block vslot >> 4 of the virtual
// grid lives at pool block bt[vslot >> 4]. Returns -1 for an entry outside
// [0, pool_blocks) and records TQ_ERR_ARG in the error word (the caller skips the access).
__device__ __forceinline__ long long phys_slot(const int32_t *bt, int pool_blocks, long long vslot, int *error) {
  if (bt == nullptr || vslot < 0) return vslot;
  const int pb = __ldg(bt + (vslot >> 4));
  if (pb < 0 || pb >= pool_blocks) {
    if (error) atomicCAS(error, 0, (int)TQ_ERR_ARG);
    return -1;
  }
  return ((long long)pb << 4) | (vslot & 15);
}

// v <- A^T v for a d x d row-major matrix A (d = 128) held by one warp, lane L owning
// coordinates 4L..4L+3: lane L sums A[k][4L..4L+3] v_k over k, each v_k reaching it by a
// shuffle and each row of A read as one coalesced 512-byte line. With A = M^T this is
// the dense rotation y = M v; with A = M its inverse x = M^T y.
__device__ __forceinline__ void matvec_t_warp(const float *A, float (&v)[4], int lane) {
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int k4 = 0; k4 < 32; ++k4) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float vk = __shfl_sync(0xffffffffu, v[j], k4);
      const float4 a = __ldg(reinterpret_cast<const float4 *>(A + (4 * k4 + j) * 128) + lane);
      y[0] = fmaf(a.x, vk, y[0]);
      y[1] = fmaf(a.y, vk, y[1]);
      y[2] = fmaf(a.z, vk, y[2]);
      y[3] = fmaf(a.w, vk, y[3]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = y[j];
}

// Side code of one key held by a warp (lane L: unit-domain residual r[4L..4L+3] in the
// coordinates the codes live in): z_k = fp16(nu sum_i U[i][k] r_i) for k < rank, with U the
// key head's basis in those coordinates ([d][rank], natural order); lane k < rank stores z_k
// at token `slot` of the side plane (nothing when slot < 0).
__device__ __forceinline__ void side_code_warp(const float *U, int rank, float nu, const float (&r)[4],
                                               uint16_t *side_plane, long long slot, int bb, int lane) {
  float mine = 0.f;
  for (int k = 0; k < rank; ++k) {
    float p = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) p = fmaf(__ldg(U + (4 * lane + j) * rank + k), r[j], p);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
    if (lane == k) mine = p * nu;
  }
  if (slot >= 0 && lane < rank)
    rec_at(side_plane, slot, bb, 2 * rank)[lane] = __half_as_ushort(__float2half_rn(mine));
}

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

// Record layout of a d = 128 vector's codes (include/tq.h): pair p = (2p, 2p+1),
// p = 4n + t, sits in slot 16t + n; slot s holds 2*BITS bits at bit offset
// 2*BITS*s (low BITS bits: even coordinate). Lane L of a warp that owns
// coordinates 4L..4L+3 owns pairs 2L (slot 32(L&1) + L/2) and 2L+1 (that + 16).
__device__ __forceinline__ int lane_slot_a(int lane) { return 32 * (lane & 1) + (lane >> 1); }

template <int BITS>
__device__ __forceinline__ uint32_t record_field(const uint32_t *rec, int slot) {
  constexpr int F = 2 * BITS;
  constexpr int W = 4 * BITS;  // words in the record
  const int bit = F * slot;
  const int wi = bit >> 5, off = bit & 31;
  uint32_t lo = __ldg(rec + wi);
  uint32_t v;
  if (off + F <= 32) {
    v = lo >> off;
  } else {
    uint32_t hi = __ldg(rec + ((wi + 1 < W) ? wi + 1 : wi));
    v = __funnelshift_r(lo, hi, off);
  }
  return v & ((1u << F) - 1u);
}

// Codes of this lane's coordinates 4L..4L+3 (warp-per-vector layout).
template <int BITS>
__device__ __forceinline__ void lane_codes(const uint32_t *rec, int lane, uint32_t (&c)[4]) {
  constexpr uint32_t M = (1u << BITS) - 1u;
  const int sa = lane_slot_a(lane);
  const uint32_t fa = record_field<BITS>(rec, sa);
  const uint32_t fb = record_field<BITS>(rec, sa + 16);
  c[0] = fa & M;
  c[1] = fa >> BITS;
  c[2] = fb & M;
  c[3] = fb >> BITS;
}

// Sign bits of this lane's coordinates 4L..4L+3 from a 4-word sign record
// (same slot layout with BITS = 1: word t holds slots 16t..16t+15).
__device__ __forceinline__ void lane_signs(const uint32_t *srec, int lane, uint32_t (&sg)[4]) {
  const int w = 2 * (lane & 1), sh = 2 * (lane >> 1);
  const uint32_t a = __ldg(srec + w) >> sh, b = __ldg(srec + w + 1) >> sh;
  sg[0] = a & 1u;
  sg[1] = (a >> 1) & 1u;
  sg[2] = b & 1u;
  sg[3] = (b >> 1) & 1u;
}

// Assemble the record from every lane's two pair fields; lanes 0..4*BITS-1
// return their 32-bit word of the record.
template <int BITS>
__device__ __forceinline__ uint32_t pack_slot_word(uint32_t field_a, uint32_t field_b, int lane) {
  constexpr int F = 2 * BITS;                  // bits per slot
  constexpr int K = (32 + F - 1) / F + 1;      // slots touching one word
  const uint32_t both = field_a | (field_b << F);
  const int first = (32 * lane) / F;
  uint32_t word = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int slot = first + k;
    const int src = 2 * (slot & 15) + ((slot >> 5) & 1);
    const uint32_t v = __shfl_sync(kFull, both, src & 31);
    const uint32_t f = ((slot >> 4) & 1) ? (v >> F) : (v & ((1u << F) - 1u));
    const int shift = F * slot - 32 * lane;
    if (slot < 64 && shift > -F && shift < 32) word |= (shift >= 0) ? (f << shift) : (f >> (-shift));
  }
  return word;
}

// ---------------------------------------------------------------------------
// Value codes of the TQ schemes are stored pair-interleaved inside each
// 16-token block: row j (j = 0..7) holds tokens 2j and 2j+1; coordinate c sits
// in field o(c) = 16 (c mod 8) + c / 8 of the row, 2*VB bits at bit 2*VB*o, token
// 2j's code in the low VB bits and token 2j+1's in the high VB bits. A row is
// 32*VB bytes (8*VB words); the 16 fields of coordinates c = g (mod 8) are
// contiguous (words VB*g .. VB*g + VB - 1), which is what a tensor-core thread of
// group g reads as its A fragments (coordinate rows, token pairs).
__host__ __device__ __forceinline__ int vt_field(int c) { return 16 * (c & 7) + (c >> 3); }

// bit offset of (token slot's half, coordinate c) inside its row
template <int VB>
__device__ __forceinline__ int vt_bit(int c, int half) { return 2 * VB * vt_field(c) + VB * half; }

// word pointer of the row holding token `slot` (block-0 base of the value-code plane)
template <int VB>
__device__ __forceinline__ uint32_t *vt_row(const uint8_t *vplane, long long slot, int bb) {
  return reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(vplane) + (slot >> 4) * (long long)bb +
                                      ((slot & 15) >> 1) * (32 * VB));
}

// Codes of coordinates 4L..4L+3 of token `slot` (warp-per-vector readers).
template <int VB>
__device__ __forceinline__ void lane_codes_vt(const uint8_t *vplane, long long slot, int bb, int lane,
                                              uint32_t (&c)[4]) {
  const uint32_t *row = vt_row<VB>(vplane, slot, bb);
  const int h = (int)(slot & 1);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int bit = vt_bit<VB>(4 * lane + k, h), wi = bit >> 5, off = bit & 31;
    uint32_t v = __ldg(row + wi) >> off;
    if (off + VB > 32) v |= __ldg(row + wi + 1) << (32 - off);
    c[k] = v & ((1u << VB) - 1u);
  }
}

// Write one code (its VB bits only, the pair partner's bits untouched), atomically.
template <int VB>
__device__ __forceinline__ void store_code_vt(uint32_t *row, int c, int half, uint32_t code) {
  const int bit = vt_bit<VB>(c, half), wi = bit >> 5, off = bit & 31;
  constexpr uint32_t M = (1u << VB) - 1u;
  atomicAnd(row + wi, ~(M << off));
  atomicOr(row + wi, code << off);
  if (off + VB > 32) {
    atomicAnd(row + wi + 1, ~(M >> (32 - off)));
    atomicOr(row + wi + 1, code >> (32 - off));
  }
}

// Thread-per-vector writers: the codes of one chunk of 32 code offsets in the
// key-record order (offset n = 32 t' + 2 m + e holds coordinate 8 m + 2 t' + e)
// land in fields o = 32 t' + 16 e + m, i.e. words 2*VB*t' .. 2*VB*t' + 2*VB - 1 of
// the row. vt_spread builds those words with this token's bits only (half h);
// vt_store_chunk writes them: when the partner token (slot ^ 1) is the vector of
// the neighbouring lane (lane ^ 1), the two lanes merge their words and each
// stores half of them; otherwise each lane merges its bits atomically.
template <int VB>
__device__ __forceinline__ void vt_spread(const uint32_t (&code)[32], int half, uint32_t (&w)[2 * VB]) {
#pragma unroll
  for (int i = 0; i < 2 * VB; ++i) w[i] = 0u;
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    const int o = 16 * (n & 1) + (n >> 1);  // field within the chunk
    const int bit = 2 * VB * o;
    w[bit >> 5] |= code[n] << (bit & 31);
    if ((bit & 31) + VB > 32) w[(bit >> 5) + 1] |= code[n] >> (32 - (bit & 31));
  }
  if (half) {  // move every code to the high half of its field (shift the 64*VB-bit span by VB)
#pragma unroll
    for (int i = 2 * VB - 1; i > 0; --i) w[i] = (w[i] << VB) | (w[i - 1] >> (32 - VB));
    w[0] <<= VB;
  }
}

template <int VB>
__device__ __forceinline__ void vt_store_chunk(uint32_t *row, int chunk, const uint32_t (&w)[2 * VB], int half,
                                               bool paired, bool valid) {
  uint32_t *dst = row + 2 * VB * chunk;
  uint32_t merged[2 * VB];
#pragma unroll
  for (int i = 0; i < 2 * VB; ++i) merged[i] = w[i] | __shfl_xor_sync(kFull, w[i], 1);
  if (!valid) return;
  if (paired) {
    // (a select rather than merged[VB * half + i]: an index known only at run time would
    // put the array in local memory)
#pragma unroll
    for (int i = 0; i < VB; ++i) dst[VB * half + i] = half ? merged[VB + i] : merged[i];
  } else {
    // this token's bits of every field of the chunk: VB ones at 2*VB*o + VB*half
    uint32_t own[2 * VB];
    {
      uint32_t ones[32];
#pragma unroll
      for (int n = 0; n < 32; ++n) ones[n] = (1u << VB) - 1u;
      vt_spread<VB>(ones, half, own);
    }
#pragma unroll
    for (int i = 0; i < 2 * VB; ++i) {
      atomicAnd(dst + i, ~own[i]);
      atomicOr(dst + i, w[i]);
    }
  }
}

// ---------------------------------------------------------------------------
// One vector per warp (lane L holding coordinates 4L..4L+3), as a decode step
// appends its new token: "Statistical Inference and Quality Measures of KV
// Cache Quantisations Inspired by TurboQuant", technical summary,
// "Quantisation schemes" (norm, seeded +/-1 diagonal and Walsh-Hadamard
// rotation, scalar Lloyd-Max codes; the (n-1)-bit role keeps a 1-bit QJL
// sketch of its residual) and "KVQuant++", "Fast codebook lookup" (a code is
// the count of boundaries at or below the coordinate).

// What a warp needs to write one role's record planes (block-0 bases of the blocked records).
struct WarpRole {
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  int bits, rotate, qjl, vt;
  float bounds[kMaxLevels];  // 2^bits - 1 used, +inf after
  float centroids[kMaxLevels];
};

template <int BITS>
__device__ __forceinline__ void warp_store_codes(uint8_t *codes, long long slot, int bb, const int (&idx)[4],
                                                 int lane) {
  const uint32_t fa = (uint32_t)idx[0] | ((uint32_t)idx[1] << BITS);
  const uint32_t fb = (uint32_t)idx[2] | ((uint32_t)idx[3] << BITS);
  const uint32_t word = pack_slot_word<BITS>(fa, fb, lane);  // every lane takes part
  if (slot >= 0 && lane < 4 * BITS)
    reinterpret_cast<uint32_t *>(rec_at(codes, slot, bb, BITS * kD / 8))[lane] = word;
}

// value codes (pair-interleaved layout): each lane merges its four codes into the
// token pair's row atomically (the partner token's bits are left alone)
template <int VB>
__device__ __forceinline__ void warp_store_codes_vt(uint8_t *vplane, long long slot, int bb, const int (&idx)[4],
                                                    int lane) {
  if (slot < 0) return;
  uint32_t *row = vt_row<VB>(vplane, slot, bb);
#pragma unroll
  for (int k = 0; k < 4; ++k) store_code_vt<VB>(row, 4 * lane + k, (int)(slot & 1), (uint32_t)idx[k]);
}

// Norm nu, unit rotated coordinates, codes; writes the code plane (and, for roles
// without a sketch, the norm) of token `slot` (nothing when slot < 0). For sketched
// roles returns the unit-domain residual r = y - c[code] (zero for a zero vector) and
// sum r^2 over the warp.
template <typename R>
__device__ __forceinline__ void encode_vector_warp(const R &ro, const float (&x)[4], long long slot, int bb,
                                                   const float *diag, int lane, float &nu, float (&r)[4],
                                                   float &rr) {
  nu = sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]));
  float y[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float dg = ro.rotate ? __ldg(diag + 4 * lane + j) : 1.f;
    y[j] = (nu > 0.f) ? (x[j] / nu) * dg : 0.f;
  }
  if (ro.rotate) wht128(y, lane);
  int idx[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int c = 0;
#pragma unroll
    for (int k = 0; k < kMaxLevels - 1; ++k) c += (y[j] >= ro.bounds[k]) ? 1 : 0;
    idx[j] = c;
  }
  if (ro.vt) {
    switch (ro.bits) {
      case 1: warp_store_codes_vt<1>(ro.codes, slot, bb, idx, lane); break;
      case 2: warp_store_codes_vt<2>(ro.codes, slot, bb, idx, lane); break;
      case 3: warp_store_codes_vt<3>(ro.codes, slot, bb, idx, lane); break;
      default: warp_store_codes_vt<4>(ro.codes, slot, bb, idx, lane); break;
    }
  } else {
    switch (ro.bits) {
      case 1: warp_store_codes<1>(ro.codes, slot, bb, idx, lane); break;
      case 2: warp_store_codes<2>(ro.codes, slot, bb, idx, lane); break;
      case 3: warp_store_codes<3>(ro.codes, slot, bb, idx, lane); break;
      default: warp_store_codes<4>(ro.codes, slot, bb, idx, lane); break;
    }
  }
  if (!ro.qjl && slot >= 0 && lane == 0) *rec_at(ro.norms, slot, bb, 4) = nu;
  rr = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = 0.f;
  if (ro.qjl) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float rj = y[j] - ro.centroids[idx[j]];
      s += rj * rj;
      r[j] = (nu > 0.f) ? rj : 0.f;
    }
    rr = warp_sum(s);
  }
}

// encode_vector_warp with two run-time options, for the warp-per-vector append: rot_t, the
// dense rotation's M^T (row-major) for contexts set to TQ_ROTATION_DENSE, else nullptr (the
// randomised Walsh-Hadamard transform with diagonal `diag`); want_res, return the residual of
// an unsketched role too (for its side code). A function of its own: the fused decode step,
// which encodes its new token with encode_vector_warp, ran 5 % slower when that function
// carried these options.
template <typename R>
__device__ __forceinline__ void encode_vector_warp_general(const R &ro, const float (&x)[4], long long slot, int bb,
                                                           const float *diag, int lane, float &nu, float (&r)[4],
                                                           float &rr, const float *rot_t, bool want_res) {
  nu = sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]));
  float y[4];
  const bool wht = ro.rotate && rot_t == nullptr;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float dg = wht ? __ldg(diag + 4 * lane + j) : 1.f;
    y[j] = (nu > 0.f) ? (x[j] / nu) * dg : 0.f;
  }
  if (wht) wht128(y, lane);
  else if (ro.rotate) matvec_t_warp(rot_t, y, lane);
  int idx[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int c = 0;
#pragma unroll
    for (int k = 0; k < kMaxLevels - 1; ++k) c += (y[j] >= ro.bounds[k]) ? 1 : 0;
    idx[j] = c;
  }
  if (ro.vt) {
    switch (ro.bits) {
      case 1: warp_store_codes_vt<1>(ro.codes, slot, bb, idx, lane); break;
      case 2: warp_store_codes_vt<2>(ro.codes, slot, bb, idx, lane); break;
      case 3: warp_store_codes_vt<3>(ro.codes, slot, bb, idx, lane); break;
      default: warp_store_codes_vt<4>(ro.codes, slot, bb, idx, lane); break;
    }
  } else {
    switch (ro.bits) {
      case 1: warp_store_codes<1>(ro.codes, slot, bb, idx, lane); break;
      case 2: warp_store_codes<2>(ro.codes, slot, bb, idx, lane); break;
      case 3: warp_store_codes<3>(ro.codes, slot, bb, idx, lane); break;
      default: warp_store_codes<4>(ro.codes, slot, bb, idx, lane); break;
    }
  }
  if (!ro.qjl && slot >= 0 && lane == 0) *rec_at(ro.norms, slot, bb, 4) = nu;
  rr = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = 0.f;
  if (ro.qjl || want_res) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float rj = y[j] - ro.centroids[idx[j]];
      s += rj * rj;
      r[j] = (nu > 0.f) ? rj : 0.f;
    }
    rr = warp_sum(s);
  }
}

// The four QJL sign words of one vector (all lanes): word m, bit L = [ (S r)_row >= 0 ] for
// the sketch row whose sign sits there, read from the permuted transpose of S
// (entry (i, 4L + m) = that row's column i; a copy in shared memory); lane L forms its
// four rows, summing over i in ascending order.
__device__ __forceinline__ void sketch_signs_warp(const float *sketch_tp, const float (&r)[4], int lane,
                                                  uint32_t (&w)[4]) {
  float z[4] = {0.f, 0.f, 0.f, 0.f};
  const float4 *col = reinterpret_cast<const float4 *>(sketch_tp) + lane;
#pragma unroll 4
  for (int i4 = 0; i4 < kD / 4; ++i4) {
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const float ri = __shfl_sync(kFull, r[ii], i4);
      const float4 sv = col[(4 * i4 + ii) * (kD / 4)];
      z[0] = fmaf(sv.x, ri, z[0]);
      z[1] = fmaf(sv.y, ri, z[1]);
      z[2] = fmaf(sv.z, ri, z[2]);
      z[3] = fmaf(sv.w, ri, z[3]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) w[m] = __ballot_sync(kFull, z[m] >= 0.f);
}

// KIVI records keep the plain order: channel i's 2-bit code at bits [2i, 2i+2).
__device__ __forceinline__ uint32_t kivi_lane_field(const uint32_t *rec, int lane) {
  return __ldg(rec + (lane >> 2)) >> (8 * (lane & 3));  // 8 bits: channels 4L..4L+3
}

// lanes 0..7 return word w = the 8-bit fields of lanes 4w..4w+3
__device__ __forceinline__ uint32_t kivi_pack_word(uint32_t field8, int lane) {
  uint32_t w = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) w |= (__shfl_sync(kFull, field8 & 0xffu, (4 * lane + k) & 31)) << (8 * k);
  return w;
}

}  // namespace tq
