// KIVI-style asymmetric 2-bit grouped quantisation with a bfloat16 window of
// recent tokens ("Your KV cache is not a bit problem but a geometry problem":
// "What quantisation error is made of" -- zero point = group minimum, step =
// range / (2^B - 1), round to nearest; "Keys" / "Values" -- group keys per
// channel along tokens and values per token along channels, or the flips;
// "The systems tax" -- keep the most recent tokens in full precision and
// quantise them in groups once enough have accumulated).
//
// Append of n_new tokens to a sequence holding N0 tokens, N = N0 + n_new:
// the window rule leaves tokens [0, nq(N)) quantised and [nq(N), N) in the
// window, nq(N) = G floor((N - W) / G) once N >= W + G. Stream-ordered launches
// keep each ring consistent:
//   flush  -- (one per tensor) quantise every group in [nq(N0), nq(N)), reading
//             tokens < N0 from the ring and later ones from the input;
//   window -- (one for both tensors, after both flushes) copy tokens
//             [max(nq(N), N0), N) from the input into the ring.

#include <cuda_fp16.h>

#include <algorithm>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kG = 32;  // group size this build implements

__device__ __forceinline__ int kivi_nq(int n, int window) {
  return (n < window + kG) ? 0 : kG * ((n - window) / kG);
}

struct KiviTensorArgs {
  const void *x;  // [batch][heads][n_new][d] input
  int bf16;
  int batch, heads, n_new, capacity, window;
  const int32_t *seq_lens;
  uint8_t *codes;      // [batch][heads][capacity][d/4]
  uint16_t *stats;     // fp16 (zero, step) pairs
  uint16_t *ring;      // bf16 [batch][heads][window + G][d]
  int *error;
  FastDiv div_units, div_heads;  // by the flush kernel's warps per (batch, head), and by heads
};

// token j's four channels 4L..4L+3 from the ring (j < n0) or the input
__device__ __forceinline__ void kivi_load(const KiviTensorArgs &a, long long bh, int n0, int j, int lane,
                                          float (&x)[4]) {
  if (j < n0) {
    const int R = a.window + kG;
    const uint16_t *src = a.ring + ((size_t)bh * R + (j % R)) * kD + 4 * lane;
    load4(src, 0, true, x);
  } else {
    load4(a.x, ((size_t)bh * a.n_new + (j - n0)) * kD + 4 * lane, a.bf16 != 0, x);
  }
}

// The step fp16((max - min) / 3) with the quotient taken in fp64 and then rounded to fp16
// (mx >= mn), without fp64 division, which this GPU runs at a small fraction of its fp32
// rate. D = mx - mn is held exactly as d + e (two-sum). The product q = d * fp32(1/3) lies
// within 2^-22 (relative) of D / 3, far inside one fp16 step, so its nearest fp16 value c is
// the answer or one of its neighbours; the
// exact sign of D - 3m at the midpoints m between c and its neighbours decides (3m has at
// most 14 significant bits, and d - 3m is exact because d and 3m are within a factor of 2),
// ties going to the even value as they do from an fp64 quotient that lands on a midpoint.
// Where D - 3m is nonzero but within the fp64 quotient's own rounding error of zero, that
// rounding could itself land on the midpoint: those groups, and quotients outside the
// normal fp16 range, take the fp64 path.
__device__ __forceinline__ __half kivi_step(float mn, float mx) {
  const float d = __fsub_rn(mx, mn);
  const float bv = __fsub_rn(d, mx);
  const float av = __fsub_rn(d, bv);
  const float e = __fadd_rn(__fsub_rn(mx, av), __fsub_rn(-mn, bv));
  const float q = __fmul_rn(d, 1.f / 3.f);
  if (!(q >= 0x1p-13f && q <= 60000.f)) return __double2half(((double)mx - (double)mn) / 3.0);
  const __half c = __float2half_rn(q);
  const unsigned short cb = __half_as_ushort(c);
  const float cf = __half2float(c);
  const float up = __half2float(__ushort_as_half((unsigned short)(cb + 1)));
  const float dn = __half2float(__ushort_as_half((unsigned short)(cb - 1)));
  const float mu = __fmul_rn(__fadd_rn(cf, up), 0.5f), ml = __fmul_rn(__fadd_rn(cf, dn), 0.5f);
  const float tu = __fadd_rn(__fsub_rn(d, __fmul_rn(3.f, mu)), e);  // sign of D - 3 mu, exactly
  const float td = __fadd_rn(__fsub_rn(d, __fmul_rn(3.f, ml)), e);  // sign of D - 3 ml, exactly
  if ((tu != 0.f && fabsf(tu) <= mu * 0x1p-50f) || (td != 0.f && fabsf(td) <= ml * 0x1p-50f))
    return __double2half(((double)mx - (double)mn) / 3.0);
  unsigned short r = cb;
  if (tu > 0.f || (tu == 0.f && (cb & 1u))) r = (unsigned short)(cb + 1);
  else if (td < 0.f || (td == 0.f && (cb & 1u))) r = (unsigned short)(cb - 1);
  return __ushort_as_half(r);
}

__device__ __forceinline__ void group_stats(float mn, float mx, __half &z, __half &s) {
  z = __float2half_rn(mn);
  s = kivi_step(mn, mx);
}

// code = clamp(rint((x - z) / s), 0, 3), ties to even, the quotient taken exactly. With
// dx = x - z (fp32) the code is the number of the thresholds c_k = (k + 1/2) s, k = 0, 1, 2, that
// dx passes: c_0 and c_2 strictly, c_1 from the threshold on, since a quotient of exactly 1/2
// or 5/2 rounds down to the even code and 3/2 rounds up. Each threshold is exact in fp32 (s has
// 11 significant bits, k + 1/2 at most 3), so no division is needed and ties, frequent when x
// and z carry few significant bits, come out exactly. The three tests are the signs of
// A = c_0 - dx, B = dx - c_1 and C = c_2 - dx (a difference of equal values is +0): they pass
// as p_0 = sign A, p_1 = not sign B, p_2 = sign C, and since they pass in order the code's
// high bit is p_1 and its low bit p_0 ^ p_1 ^ p_2, i.e. the complements of sign B and of the
// sign of A ^ B ^ C. kivi_push2 shifts these two sign bits into a word from below, so that
// the complement of the word holds the codes, the value pushed last in the lowest bits. A zero
// or infinite step makes every code 0, as a zero quotient would: the thresholds are then +inf
// and x is compared as is (so that an infinite zero point gives no inf - inf).
struct KiviCoder {
  float nz, c0, c1, c2;  // -z (0 for a degenerate step) and the thresholds
};
__device__ __forceinline__ KiviCoder kivi_coder(__half z, __half s) {
  const float sf = __half2float(s);
  if (!(sf > 0.f && sf < INFINITY)) return KiviCoder{0.f, INFINITY, INFINITY, INFINITY};
  return KiviCoder{-__half2float(z), 0.5f * sf, 1.5f * sf, 2.5f * sf};
}
// push the codes of x.y, then x.x (coders kx for x.x, ky for x.y)
__device__ __forceinline__ void kivi_push2(float2 x, const KiviCoder &kx, const KiviCoder &ky, uint32_t &acc) {
  const float2 dx = __fadd2_rn(x, make_float2(kx.nz, ky.nz));
  const float2 A = __ffma2_rn(dx, make_float2(-1.f, -1.f), make_float2(kx.c0, ky.c0));
  const float2 B = __fadd2_rn(dx, make_float2(-kx.c1, -ky.c1));
  const float2 C = __ffma2_rn(dx, make_float2(-1.f, -1.f), make_float2(kx.c2, ky.c2));
  const uint32_t bx = __float_as_uint(B.x), by = __float_as_uint(B.y);
  const uint32_t tx = __float_as_uint(A.x) ^ bx ^ __float_as_uint(C.x);
  const uint32_t ty = __float_as_uint(A.y) ^ by ^ __float_as_uint(C.y);
  acc = __funnelshift_l(by, acc, 1);
  acc = __funnelshift_l(ty, acc, 1);
  acc = __funnelshift_l(bx, acc, 1);
  acc = __funnelshift_l(tx, acc, 1);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) {
  __nv_bfloat162 h;
  memcpy(&h, &w, 4);
  return h;
}
__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 h) {
  uint32_t w;
  memcpy(&w, &h, 4);
  return w;
}

// Group-per-channel coding of one group, rows j0 .. j0 + 31, lane L: channels 4L..4L+3. The rows
// are read twice, for the statistics and for the codes (the second time mostly from L2), which
// keeps registers and so leaves room for more warps to hide the loads. IN: every row comes from
// the input, at constant strides; otherwise rows before n0 come from the window ring.
template <bool BF16, bool IN>
__device__ __forceinline__ void code_channel_group(const KiviTensorArgs &a, long long bh, int n0, int j0, int lane) {
  const int R = a.window + kG;
  // input row j0 + k at in0 + k * kD elements (j0 - n0 is negative only when !IN)
  const long long in0 = ((long long)bh * a.n_new + (j0 - n0)) * kD + 4 * lane;
  // row k's four channels: raw bfloat16 pairs (BF16), or floats
  auto row_bf16 = [&](int k) -> uint2 {
    const int j = j0 + k;
    if (IN || j >= n0) return __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.x) + in0 + k * kD));
    return __ldg(reinterpret_cast<const uint2 *>(a.ring + ((size_t)bh * R + (j % R)) * kD + 4 * lane));
  };
  auto row_f32 = [&](int k, float (&x)[4]) {
    const int j = j0 + k;
    if (IN || j >= n0) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + in0 + k * kD));
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else {
      load4(a.ring + ((size_t)bh * R + (j % R)) * kD + 4 * lane, 0, true, x);
    }
  };
  float mn[4], mx[4];
  if constexpr (BF16) {
    // bfloat16 minima and maxima are exact, two channels per instruction
    const uint2 r0 = row_bf16(0);
    __nv_bfloat162 lo01 = as_bf162(r0.x), hi01 = lo01, lo23 = as_bf162(r0.y), hi23 = lo23;
#pragma unroll 8
    for (int k = 1; k < kG; ++k) {
      const uint2 r = row_bf16(k);
      lo01 = __hmin2(lo01, as_bf162(r.x));
      hi01 = __hmax2(hi01, as_bf162(r.x));
      lo23 = __hmin2(lo23, as_bf162(r.y));
      hi23 = __hmax2(hi23, as_bf162(r.y));
    }
    mn[0] = bf16_lo(bf162_bits(lo01));
    mn[1] = bf16_hi(bf162_bits(lo01));
    mn[2] = bf16_lo(bf162_bits(lo23));
    mn[3] = bf16_hi(bf162_bits(lo23));
    mx[0] = bf16_lo(bf162_bits(hi01));
    mx[1] = bf16_hi(bf162_bits(hi01));
    mx[2] = bf16_lo(bf162_bits(hi23));
    mx[3] = bf16_hi(bf162_bits(hi23));
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mn[c] = INFINITY;
      mx[c] = -INFINITY;
    }
#pragma unroll 8
    for (int k = 0; k < kG; ++k) {
      float x[4];
      row_f32(k, x);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mn[c] = fminf(mn[c], x[c]);
        mx[c] = fmaxf(mx[c], x[c]);
      }
    }
  }
  KiviCoder kc[4];
  uint32_t st[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    __half z, s;
    group_stats(mn[c], mx[c], z, s);
    kc[c] = kivi_coder(z, s);
    st[c] = (uint32_t)__half_as_ushort(z) | ((uint32_t)__half_as_ushort(s) << 16);
  }
  uint4 *srec = reinterpret_cast<uint4 *>(a.stats + (((size_t)bh * (a.capacity / kG) + j0 / kG) * kD) * 2);
  srec[lane] = make_uint4(st[0], st[1], st[2], st[3]);
  uint8_t *crow = a.codes + ((size_t)bh * a.capacity + j0) * (kD / 4) + lane;
#pragma unroll 8
  for (int k = 0; k < kG; ++k) {
    float x[4];
    if constexpr (BF16) {
      const uint2 r = row_bf16(k);
      x[0] = bf16_lo(r.x);
      x[1] = bf16_hi(r.x);
      x[2] = bf16_lo(r.y);
      x[3] = bf16_hi(r.y);
    } else {
      row_f32(k, x);
    }
    uint32_t acc = 0;
    kivi_push2(make_float2(x[2], x[3]), kc[2], kc[3], acc);
    kivi_push2(make_float2(x[0], x[1]), kc[0], kc[1], acc);
    crow[k * (kD / 4)] = (uint8_t)~acc;
  }
}

// one warp per (batch, head, group of 32 tokens); lane L owns channels 4L..4L+3 and writes
// byte L of each token's 32-byte code record
template <bool BF16>
__global__ void __launch_bounds__(256) kivi_flush_per_channel(KiviTensorArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t unit = blockIdx.x * 8u + (threadIdx.x >> 5);
  const uint32_t bh = fast_div(unit, a.div_units);
  if (bh >= (uint32_t)(a.batch * a.heads)) return;
  const int n0 = __ldg(a.seq_lens + fast_div(bh, a.div_heads));
  const int n1 = n0 + a.n_new;
  const int u = (int)(unit - bh * a.div_units.d);
  if (n1 > a.capacity) {
    if (lane == 0 && u == 0) set_error(a.error, TQ_ERR_CAPACITY);
    return;
  }
  const int j0 = kivi_nq(n0, a.window) + kG * u;
  if (j0 >= kivi_nq(n1, a.window)) return;
  if (j0 >= n0) code_channel_group<BF16, true>(a, bh, n0, j0, lane);
  else code_channel_group<BF16, false>(a, bh, n0, j0, lane);
}

// one warp per (batch, head, run of kTokRun = 8 consecutive tokens); lane L codes group L mod 4
// (channels 32 (L mod 4) .. + 31) of token L / 4 by itself: statistics, step and codes, no
// exchange between lanes. Its 64 code bits are bytes 8 (L mod 4) .. + 7 of the token's record.
// (bfloat16: six blocks of 256 per SM, 40 registers; the loads' latency, not the arithmetic,
// leads.)
constexpr int kTokRun = 8;
template <bool BF16>
__global__ void __launch_bounds__(256, BF16 ? 6 : 4) kivi_flush_per_token(KiviTensorArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t unit = blockIdx.x * 8u + (threadIdx.x >> 5);
  const uint32_t bh = fast_div(unit, a.div_units);
  if (bh >= (uint32_t)(a.batch * a.heads)) return;
  const int n0 = __ldg(a.seq_lens + fast_div(bh, a.div_heads));
  const int n1 = n0 + a.n_new;
  const int u = (int)(unit - bh * a.div_units.d);
  if (n1 > a.capacity) {
    if (lane == 0 && u == 0) set_error(a.error, TQ_ERR_CAPACITY);
    return;
  }
  const int j = kivi_nq(n0, a.window) + kTokRun * u + (lane >> 2);
  if (j >= kivi_nq(n1, a.window)) return;  // lanes work independently from here on
  const int grp = lane & 3;
  float x[kG];
  float mn, mx;
  const bool from_ring = j < n0;
  if (BF16 || from_ring) {
    const uint16_t *row = from_ring ? a.ring + ((size_t)bh * (a.window + kG) + (j % (a.window + kG))) * kD
                                    : static_cast<const uint16_t *>(a.x) + ((size_t)bh * a.n_new + (j - n0)) * kD;
    const uint4 *src = reinterpret_cast<const uint4 *>(row + kG * grp);
    uint32_t w[kG / 2];
#pragma unroll
    for (int i = 0; i < kG / 8; ++i) {
      const uint4 q4 = __ldg(src + i);
      w[4 * i] = q4.x;
      w[4 * i + 1] = q4.y;
      w[4 * i + 2] = q4.z;
      w[4 * i + 3] = q4.w;
    }
    __nv_bfloat162 lo = as_bf162(w[0]), hi = lo;
#pragma unroll
    for (int i = 1; i < kG / 2; ++i) {
      lo = __hmin2(lo, as_bf162(w[i]));
      hi = __hmax2(hi, as_bf162(w[i]));
    }
    mn = fminf(bf16_lo(bf162_bits(lo)), bf16_hi(bf162_bits(lo)));
    mx = fmaxf(bf16_lo(bf162_bits(hi)), bf16_hi(bf162_bits(hi)));
#pragma unroll
    for (int i = 0; i < kG / 2; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) +
                                                         ((size_t)bh * a.n_new + (j - n0)) * kD + kG * grp);
#pragma unroll
    for (int i = 0; i < kG / 4; ++i) {
      const float4 f = __ldg(src + i);
      x[4 * i] = f.x;
      x[4 * i + 1] = f.y;
      x[4 * i + 2] = f.z;
      x[4 * i + 3] = f.w;
    }
    mn = x[0];
    mx = x[0];
#pragma unroll
    for (int c = 1; c < kG; ++c) {
      mn = fminf(mn, x[c]);
      mx = fmaxf(mx, x[c]);
    }
  }
  __half z, s;
  group_stats(mn, mx, z, s);
  const KiviCoder kc = kivi_coder(z, s);
  const size_t slot = (size_t)bh * a.capacity + j;
  reinterpret_cast<uint32_t *>(a.stats + slot * (kD / kG) * 2)[grp] =
      (uint32_t)__half_as_ushort(z) | ((uint32_t)__half_as_ushort(s) << 16);
  uint32_t word[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0;
#pragma unroll
    for (int i = 7; i >= 0; --i) kivi_push2(make_float2(x[16 * h + 2 * i], x[16 * h + 2 * i + 1]), kc, kc, acc);
    word[h] = ~acc;
  }
  reinterpret_cast<uint2 *>(a.codes + slot * (kD / 4))[grp] = make_uint2(word[0], word[1]);
}

// Window tokens go to the bf16 ring. Tokens j < nq(n1) are quantised, and nq(n1) > n1 - W - G,
// so only the last W + G - 1 new tokens can stay in the window: t_first = max(0, n_new - (W + G -
// 1)). One warp per (batch, head, run of kWinRun new tokens from t_first on); a half-warp moves
// one token row, 16 bytes (8 channels) per lane.
constexpr int kWinRun = 8;
// (one launch for both tensors: blockIdx.y = 0 keys, 1 values)
struct KiviWindowArgs {
  KiviTensorArgs t[2];
};
__global__ void __launch_bounds__(256) kivi_window_write(const __grid_constant__ KiviWindowArgs w, int t_first,
                                                         FastDiv div_runs) {
  const KiviTensorArgs &a = w.t[blockIdx.y];
  const int lane = threadIdx.x & 31;
  const uint32_t unit = blockIdx.x * 8u + (threadIdx.x >> 5);
  const uint32_t bh = fast_div(unit, div_runs);
  if (bh >= (uint32_t)(a.batch * a.heads)) return;
  const int n0 = __ldg(a.seq_lens + fast_div(bh, a.div_heads));
  const int n1 = n0 + a.n_new;
  if (n1 > a.capacity) return;
  const int nq1 = kivi_nq(n1, a.window);
  const int R = a.window + kG;
  const int t0 = t_first + kWinRun * (int)(unit - bh * div_runs.d);
  const int piece = lane & 15;
#pragma unroll
  for (int i = 0; i < kWinRun / 2; ++i) {
    const int t = t0 + 2 * i + (lane >> 4);
    const int j = n0 + t;
    if (t >= a.n_new || j < nq1) continue;
    const size_t row = ((size_t)bh * a.n_new + t) * kD;
    uint4 w;
    if (a.bf16) {
      w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + row) + piece);
    } else {
      const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + row) + 2 * piece;
      const float4 f0 = __ldg(src), f1 = __ldg(src + 1);
      w = make_uint4(bf162_bits(__floats2bfloat162_rn(f0.x, f0.y)), bf162_bits(__floats2bfloat162_rn(f0.z, f0.w)),
                     bf162_bits(__floats2bfloat162_rn(f1.x, f1.y)), bf162_bits(__floats2bfloat162_rn(f1.z, f1.w)));
    }
    reinterpret_cast<uint4 *>(a.ring + ((size_t)bh * R + (j % R)) * kD)[piece] = w;
  }
}

struct KiviDequantKernelArgs {
  const uint8_t *codes;
  const uint16_t *stats;
  const uint16_t *ring;
  int per_channel, batch, heads, capacity, window, t0, t1;
  const int32_t *seq_lens;
  float *out;
};

__global__ void __launch_bounds__(256) kivi_dequant_kernel(KiviDequantKernelArgs a) {
  const int lane = threadIdx.x & 31;
  const int n = a.t1 - a.t0;
  const long long vec = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (vec >= (long long)a.batch * a.heads * n) return;
  const long long bh = vec / n;
  const int j = a.t0 + (int)(vec % n);
  const int len = min(max(__ldg(a.seq_lens + bh / a.heads), 0), a.capacity);
  const int nq = kivi_nq(len, a.window);
  float y[4] = {0.f, 0.f, 0.f, 0.f};
  const size_t slot = (size_t)bh * a.capacity + j;
  if (j < nq) {
    const uint32_t f = kivi_lane_field(reinterpret_cast<const uint32_t *>(a.codes) + slot * (kD / 16), lane);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t st;
      if (a.per_channel)
        st = __ldg(reinterpret_cast<const uint32_t *>(a.stats) + ((size_t)bh * (a.capacity / kG) + j / kG) * kD +
                   4 * lane + c);
      else
        st = __ldg(reinterpret_cast<const uint32_t *>(a.stats) + slot * (kD / kG) + (lane >> 3));
      const float z = __half2float(__ushort_as_half((unsigned short)(st & 0xffffu)));
      const float s = __half2float(__ushort_as_half((unsigned short)(st >> 16)));
      y[c] = fmaf(s, (float)((f >> (2 * c)) & 3u), z);
    }
  } else if (j < len) {
    const int R = a.window + kG;
    load4(a.ring + ((size_t)bh * R + (j % R)) * kD, 4 * lane, true, y);
  }
  reinterpret_cast<float4 *>(a.out + (size_t)vec * kD)[lane] = make_float4(y[0], y[1], y[2], y[3]);
}

int flush(KiviTensorArgs t, bool per_channel, cudaStream_t st) {
  const long long bh = (long long)t.batch * t.heads;
  // groups (or tokens) newly quantised by one append: at most (n_new + G - 1) tokens
  const int max_tokens = t.n_new + kG - 1;
  const int units = per_channel ? (max_tokens + kG - 1) / kG + 1 : (max_tokens + kTokRun - 1) / kTokRun;
  const long long warps = bh * units;
  if (warps >= 0xffffffffLL - 8) return TQ_ERR_ARG;  // warp indices are 32-bit
  t.div_units = make_fastdiv((uint32_t)units);
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (per_channel) {
    if (t.bf16) kivi_flush_per_channel<true><<<blocks, 256, 0, st>>>(t);
    else kivi_flush_per_channel<false><<<blocks, 256, 0, st>>>(t);
  } else {
    if (t.bf16) kivi_flush_per_token<true><<<blocks, 256, 0, st>>>(t);
    else kivi_flush_per_token<false><<<blocks, 256, 0, st>>>(t);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// window tokens of both tensors; after both flushes (each tensor's flush reads its ring first)
int window(const KiviWindowArgs &w, cudaStream_t st) {
  const KiviTensorArgs &t = w.t[0];
  const long long bh = (long long)t.batch * t.heads;
  const int t_first = std::max(0, t.n_new - (t.window + kG - 1));
  const int runs = (t.n_new - t_first + kWinRun - 1) / kWinRun;
  const long long wwarps = bh * runs;
  kivi_window_write<<<dim3((unsigned)((wwarps + 7) / 8), 2), 256, 0, st>>>(w, t_first, make_fastdiv((uint32_t)runs));
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

int launch_append_kivi(const KiviAppendArgs &a, void *stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const tq_ctx *ctx = a.ctx;
  const tq_cache *c = a.cache;
  if (ctx->kivi_group != kG) return TQ_ERR_UNSUPPORTED;
  KiviTensorArgs t{};
  t.bf16 = a.dtype == TQ_BF16;
  t.batch = a.batch;
  t.heads = a.heads;
  t.n_new = a.n_new;
  t.capacity = c->capacity;
  t.window = ctx->kivi_window;
  t.seq_lens = a.seq_lens;
  t.error = a.error;
  t.div_heads = make_fastdiv((uint32_t)a.heads);
  KiviWindowArgs w{};
  w.t[0] = w.t[1] = t;
  w.t[0].x = a.k;
  w.t[0].codes = c->k_codes;
  w.t[0].stats = c->k_stats;
  w.t[0].ring = c->k_window;
  w.t[1].x = a.v;
  w.t[1].codes = c->v_codes;
  w.t[1].stats = c->v_stats;
  w.t[1].ring = c->v_window;
  int r = flush(w.t[0], ctx->kivi_k_per_channel != 0, st);
  if (r == TQ_OK) r = flush(w.t[1], ctx->kivi_v_per_token == 0, st);
  if (r == TQ_OK) r = window(w, st);
  return r;
}

int launch_dequant_kivi(const KiviDequantArgs &a, void *stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const tq_ctx *ctx = a.ctx;
  const tq_cache *c = a.cache;
  const long long total = (long long)a.batch * a.heads * (a.t1 - a.t0);
  const unsigned blocks = (unsigned)((total + 7) / 8);
  for (int which = 0; which < 2; ++which) {
    float *out = which ? a.v_out : a.k_out;
    if (!out) continue;
    KiviDequantKernelArgs k{};
    k.codes = which ? c->v_codes : c->k_codes;
    k.stats = which ? c->v_stats : c->k_stats;
    k.ring = which ? c->v_window : c->k_window;
    k.per_channel = which ? (ctx->kivi_v_per_token == 0) : (ctx->kivi_k_per_channel != 0);
    k.batch = a.batch;
    k.heads = a.heads;
    k.capacity = c->capacity;
    k.window = ctx->kivi_window;
    k.t0 = a.t0;
    k.t1 = a.t1;
    k.seq_lens = a.seq_lens;
    k.out = out;
    kivi_dequant_kernel<<<blocks, 256, 0, st>>>(k);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace tq
