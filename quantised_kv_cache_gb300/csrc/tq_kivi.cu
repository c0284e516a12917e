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
// window, nq(N) = G floor((N - W) / G) once N >= W + G. Two stream-ordered
// launches per tensor keep the ring consistent:
//   flush  -- quantise every group in [nq(N0), nq(N)), reading tokens < N0
//             from the ring and later ones from the input;
//   window -- copy tokens [max(nq(N), N0), N) from the input into the ring.

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
// rate. D = mx - mn is held exactly as d + e (two-sum). The fp32 quotient d / 3 lies within
// 2^-23 of D / 3, so its nearest fp16 value c is the answer or one of its neighbours; the
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
  const float q = __fdiv_rn(d, 3.f);
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

// code = clamp(rint((x - z) / s), 0, 3), ties to even, with the division as a product by
// inv = 1 / s (0 when s = 0, which makes every code 0). The product is within a few fp32 ulps
// of the quotient, so it decides the code except near a rounding boundary; there, and at
// exact ties (frequent when x and z carry few significant bits), the correctly rounded
// quotient decides.
__device__ __forceinline__ uint32_t kivi_code(float x, float z, float s, float inv) {
  const float dx = x - z;
  const float t = dx * inv;
  float r = rintf(t);
  if (fabsf(t - r) > 0.5f - 0x1p-16f) r = rintf(__fdiv_rn(dx, s));  // within 2^-16 of a half-integer
  r = fminf(fmaxf(r, 0.f), 3.f);
  return (uint32_t)r;
}
__device__ __forceinline__ float kivi_inv(float s) { return (s > 0.f) ? 1.f / s : 0.f; }

// Codes of many values at once. For a value x of a group with statistics (z, s) the code is
// clamp(rint(t), 0, 3), t = (x - z) * inv, exactly as kivi_code computes it; two values go
// through each packed fp32 operation. Rounding uses the magic constant 1.5 * 2^23: for
// |u| < 2^22, u + 1.5 * 2^23 rounds u to the nearest integer, ties to even (the constant is
// even), and leaves it in the low mantissa bits, so the sum's bit pattern minus kMagicBits is
// the code of the clamped u (clamping to the integers 0 and 3 commutes with rounding). The
// distance of the clamped t from its rounding is kept: when it is within 2^-16 of 1/2 the
// product may have decided a rounding that only the exact quotient can (kivi_code's slow
// path), and the caller recomputes those values with kivi_code itself. Outside [0, 3] the clamp
// decides and both paths agree.
constexpr float kMagic = 12582912.f;
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kTieBand = 0.5f - 0x1p-16f;

struct CodePair {
  uint32_t b0, b1;  // kMagicBits + code
  float dev;        // max |clamped t - its rounding| of the two
};

__device__ __forceinline__ CodePair kivi_code_pair(float2 x, float2 nz, float2 inv) {
  const float2 t = __fmul2_rn(__fadd2_rn(x, nz), inv);
  const float2 tc = make_float2(fminf(fmaxf(t.x, 0.f), 3.f), fminf(fmaxf(t.y, 0.f), 3.f));
  const float2 m = __fadd2_rn(tc, make_float2(kMagic, kMagic));
  const float2 r = __fadd2_rn(m, make_float2(-kMagic, -kMagic));
  const float2 d = __ffma2_rn(r, make_float2(-1.f, -1.f), tc);
  return CodePair{__float_as_uint(m.x), __float_as_uint(m.y), fmaxf(fabsf(d.x), fabsf(d.y))};
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

// one warp per (batch, head, group of 32 tokens); lane L owns channels 4L..4L+3 and writes
// byte L of each token's 32-byte code record. bfloat16 rows stay in registers between the
// statistics and the codes; fp32 rows are read twice (the second time mostly from L2).
template <bool BF16>
__global__ void __launch_bounds__(256) kivi_flush_per_channel(KiviTensorArgs a, int units_per_bh) {
  const int lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long bh = unit / units_per_bh;
  if (bh >= (long long)a.batch * a.heads) return;
  const int b = (int)(bh / a.heads);
  const int n0 = __ldg(a.seq_lens + b);
  const int n1 = n0 + a.n_new;
  if (n1 > a.capacity) {
    if (lane == 0 && unit % units_per_bh == 0) set_error(a.error, TQ_ERR_CAPACITY);
    return;
  }
  const int g = kivi_nq(n0, a.window) / kG + (int)(unit % units_per_bh);
  if (g * kG >= kivi_nq(n1, a.window)) return;
  const int j0 = g * kG;
  // a group that starts at or after n0 is read from the input only, at constant row strides
  const bool from_input = j0 >= n0;
  const size_t in0 = ((size_t)bh * a.n_new + (size_t)(from_input ? j0 - n0 : 0)) * kD + 4 * lane;
  float mn[4], mx[4];
  uint2 raw[BF16 ? kG : 1];
  if constexpr (BF16) {
    const uint2 *src = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.x) + in0);
    if (from_input) {
#pragma unroll
      for (int k = 0; k < kG; ++k) raw[k] = __ldg(src + k * (kD / 4));
    } else {
      const int R = a.window + kG;
#pragma unroll
      for (int k = 0; k < kG; ++k) {
        const int j = j0 + k;
        const uint2 *p = (j < n0) ? reinterpret_cast<const uint2 *>(a.ring + ((size_t)bh * R + (j % R)) * kD + 4 * lane)
                                  : reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.x) +
                                                                    ((size_t)bh * a.n_new + (j - n0)) * kD + 4 * lane);
        raw[k] = __ldg(p);
      }
    }
    // bfloat16 minima and maxima are exact, two channels per instruction
    __nv_bfloat162 lo01 = as_bf162(raw[0].x), hi01 = lo01, lo23 = as_bf162(raw[0].y), hi23 = lo23;
#pragma unroll
    for (int k = 1; k < kG; ++k) {
      lo01 = __hmin2(lo01, as_bf162(raw[k].x));
      hi01 = __hmax2(hi01, as_bf162(raw[k].x));
      lo23 = __hmin2(lo23, as_bf162(raw[k].y));
      hi23 = __hmax2(hi23, as_bf162(raw[k].y));
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
      kivi_load(a, bh, n0, j0 + k, lane, x);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mn[c] = fminf(mn[c], x[c]);
        mx[c] = fmaxf(mx[c], x[c]);
      }
    }
  }
  float zf[4], sf[4], inv[4];
  uint32_t st[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    __half z, s;
    group_stats(mn[c], mx[c], z, s);
    zf[c] = __half2float(z);
    sf[c] = __half2float(s);
    inv[c] = kivi_inv(sf[c]);
    st[c] = (uint32_t)__half_as_ushort(z) | ((uint32_t)__half_as_ushort(s) << 16);
  }
  uint4 *srec = reinterpret_cast<uint4 *>(a.stats + (((size_t)bh * (a.capacity / kG) + g) * kD) * 2);
  srec[lane] = make_uint4(st[0], st[1], st[2], st[3]);
  const float2 nz01 = make_float2(-zf[0], -zf[1]), nz23 = make_float2(-zf[2], -zf[3]);
  const float2 iv01 = make_float2(inv[0], inv[1]), iv23 = make_float2(inv[2], inv[3]);
  uint8_t *crow = a.codes + ((size_t)bh * a.capacity + j0) * (kD / 4) + lane;
#pragma unroll  // (whole: raw[] stays in registers)
  for (int k = 0; k < kG; ++k) {
    float x[4];
    if constexpr (BF16) {
      x[0] = bf16_lo(raw[k].x);
      x[1] = bf16_hi(raw[k].x);
      x[2] = bf16_lo(raw[k].y);
      x[3] = bf16_hi(raw[k].y);
    } else {
      kivi_load(a, bh, n0, j0 + k, lane, x);
    }
    const CodePair p = kivi_code_pair(make_float2(x[0], x[1]), nz01, iv01);
    const CodePair q = kivi_code_pair(make_float2(x[2], x[3]), nz23, iv23);
    uint32_t field = p.b0 + 4u * p.b1 + 16u * q.b0 + 64u * q.b1 - 85u * kMagicBits;
    if (fmaxf(p.dev, q.dev) > kTieBand) {
      field = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) field |= kivi_code(x[c], zf[c], sf[c], inv[c]) << (2 * c);
    }
    crow[k * (kD / 4)] = (uint8_t)field;
  }
}

// one warp per (batch, head, run of kTokRun = 8 consecutive tokens); lane L codes group L mod 4
// (channels 32 (L mod 4) .. + 31) of token L / 4 by itself: statistics, step and codes, no
// exchange between lanes. Its 64 code bits are bytes 8 (L mod 4) .. + 7 of the token's record.
constexpr int kTokRun = 8;
template <bool BF16>
__global__ void __launch_bounds__(256) kivi_flush_per_token(KiviTensorArgs a, int units_per_bh) {
  const int lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long bh = unit / units_per_bh;
  if (bh >= (long long)a.batch * a.heads) return;
  const int b = (int)(bh / a.heads);
  const int n0 = __ldg(a.seq_lens + b);
  const int n1 = n0 + a.n_new;
  if (n1 > a.capacity) {
    if (lane == 0 && unit % units_per_bh == 0) set_error(a.error, TQ_ERR_CAPACITY);
    return;
  }
  const int j = kivi_nq(n0, a.window) + kTokRun * (int)(unit % units_per_bh) + (lane >> 2);
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
      const uint4 u = __ldg(src + i);
      w[4 * i] = u.x;
      w[4 * i + 1] = u.y;
      w[4 * i + 2] = u.z;
      w[4 * i + 3] = u.w;
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
  const float zf = __half2float(z), sf = __half2float(s), inv = kivi_inv(sf);
  const size_t slot = (size_t)bh * a.capacity + j;
  reinterpret_cast<uint32_t *>(a.stats + slot * (kD / kG) * 2)[grp] =
      (uint32_t)__half_as_ushort(z) | ((uint32_t)__half_as_ushort(s) << 16);
  const float2 nz = make_float2(-zf, -zf), iv = make_float2(inv, inv);
  uint32_t word[2];
  float dev = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0u - 0x55555555u * kMagicBits;  // the sum of kMagicBits * 4^i, i < 16, taken off
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const CodePair p = kivi_code_pair(make_float2(x[16 * h + 2 * i], x[16 * h + 2 * i + 1]), nz, iv);
      acc += p.b0 * (1u << (4 * i)) + p.b1 * (1u << (4 * i + 2));
      dev = fmaxf(dev, p.dev);
    }
    word[h] = acc;
  }
  if (dev > kTieBand) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc |= kivi_code(x[16 * h + i], zf, sf, inv) << (2 * i);
      word[h] = acc;
    }
  }
  reinterpret_cast<uint2 *>(a.codes + slot * (kD / 4))[grp] = make_uint2(word[0], word[1]);
}

// one warp per (batch, head, new token t >= t_first): window tokens go to the bf16 ring.
// Tokens j < nq(n1) are quantised, and nq(n1) > n1 - W - G, so only the last W + G - 1 new
// tokens can stay in the window: t_first = max(0, n_new - (W + G - 1)).
__global__ void __launch_bounds__(256) kivi_window_write(KiviTensorArgs a, int t_first) {
  const int lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int span = a.n_new - t_first;
  const long long bh = unit / span;
  if (bh >= (long long)a.batch * a.heads) return;
  const int t = t_first + (int)(unit % span);
  const int b = (int)(bh / a.heads);
  const int n0 = __ldg(a.seq_lens + b);
  const int n1 = n0 + a.n_new;
  if (n1 > a.capacity) return;
  const int j = n0 + t;
  if (j < kivi_nq(n1, a.window)) return;
  float x[4];
  load4(a.x, ((size_t)bh * a.n_new + t) * kD + 4 * lane, a.bf16 != 0, x);
  const int R = a.window + kG;
  uint16_t h[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) h[c] = __bfloat16_as_ushort(__float2bfloat16_rn(x[c]));
  uint2 w;
  w.x = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
  w.y = (uint32_t)h[2] | ((uint32_t)h[3] << 16);
  reinterpret_cast<uint2 *>(a.ring + ((size_t)bh * R + (j % R)) * kD)[lane] = w;
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

int flush_and_window(KiviTensorArgs t, bool per_channel, cudaStream_t st) {
  const long long bh = (long long)t.batch * t.heads;
  // groups (or tokens) newly quantised by one append: at most (n_new + G - 1) tokens
  const int max_tokens = t.n_new + kG - 1;
  const int units = per_channel ? (max_tokens + kG - 1) / kG + 1 : (max_tokens + kTokRun - 1) / kTokRun;
  const long long warps = bh * units;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (per_channel) {
    if (t.bf16) kivi_flush_per_channel<true><<<blocks, 256, 0, st>>>(t, units);
    else kivi_flush_per_channel<false><<<blocks, 256, 0, st>>>(t, units);
  } else {
    if (t.bf16) kivi_flush_per_token<true><<<blocks, 256, 0, st>>>(t, units);
    else kivi_flush_per_token<false><<<blocks, 256, 0, st>>>(t, units);
  }
  const int t_first = std::max(0, t.n_new - (t.window + kG - 1));
  const long long wwarps = bh * (t.n_new - t_first);
  kivi_window_write<<<(unsigned)((wwarps + 7) / 8), 256, 0, st>>>(t, t_first);
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
  t.x = a.k;
  t.codes = c->k_codes;
  t.stats = c->k_stats;
  t.ring = c->k_window;
  int r = flush_and_window(t, ctx->kivi_k_per_channel != 0, st);
  if (r != TQ_OK) return r;
  t.x = a.v;
  t.codes = c->v_codes;
  t.stats = c->v_stats;
  t.ring = c->v_window;
  return flush_and_window(t, ctx->kivi_v_per_token == 0, st);
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
