// Split-K decode attention over the packed cache, one query head per KV head.
//
// Same computation as decode_tq_kernel (softmax(q K_hat^T / sqrt(d)) V_hat
// with keys read through logits and values through the p-weighted sum in the
// rotated domain; "HeadQ", 2.1-2.2; "Statistical Inference ... Inspired by
// TurboQuant", technical summary, "K-V asymmetry", "Main contribution 1"),
// organised for sm_103a:
//
// * record tiles of 64 tokens stream into shared memory through 1-D TMA bulk
//   copies, three stages deep, each completing on an mbarrier (bounded waits);
// * keys: per CTA a float32 table T[v][pos] = sum over the coordinates a code
//   position covers of q_rot[i] c[code_i(v)] turns each token's score into one
//   lookup per byte (or 6-bit slot) of its record -- fp32 throughout, so scores
//   keep full precision whatever the key scale;
// * values and QJL signs: the p-weighted sums over a warp's 16 tokens run on
//   the tensor cores (mma.sync m16n8k16, fp32 accumulate): value codes are
//   decoded to fp16 pairs through a per-lane replicated table and transposed
//   with movmatrix; sign bits become {0, 2^-14} operands built from two
//   tokens' sign words with a byte permute and one funnel shift. The token weights p nu are split into fp16
//   hi + lo parts so the weights add no rounding of their own.
//
// CTA: 4 warps, one (batch, kv head, chunk). A warp owns 16 tokens of each
// 64-token tile: it scores them (16 lanes per token, 2 tokens per step), takes
// the online-softmax step, and issues the value / sign MMAs.

#include <cuda_fp16.h>

#include "tq_ptx.cuh"

namespace tq {
namespace {

constexpr int kWarps2 = 4;
constexpr int kTT = 64;     // tokens per tile
constexpr int kStages = 3;  // TMA pipeline depth (two CTAs per SM fit in shared memory)

template <int KB, int VB, bool KQJL, bool VQJL>
struct Geo {
  // per-token record bytes of each plane
  static constexpr int kc = 16 * KB, vc = 16 * VB;
  // stage layout (bytes), every plane 16-byte aligned
  static constexpr int off_kc = 0;
  static constexpr int off_kn = off_kc + kTT * kc;
  static constexpr int off_ks = off_kn + kTT * 4;
  static constexpr int off_kr = off_ks + (KQJL ? kTT * 16 : 0);
  static constexpr int off_vc = off_kr + (KQJL ? kTT * 4 : 0);
  static constexpr int off_vn = off_vc + kTT * vc;
  static constexpr int off_vs = off_vn + kTT * 4;
  static constexpr int off_vr = off_vs + (VQJL ? kTT * 16 : 0);
  static constexpr int stage = off_vr + (VQJL ? kTT * 4 : 0);
  // key table: positions per record and values per position
  static constexpr int kpos = (KB == 3) ? 64 : 16 * KB;   // 6-bit slots, or bytes
  static constexpr int kval = (KB == 3) ? 64 : 256;
  static constexpr int ktab = kpos * kval;                 // floats
  static constexpr int stab = KQJL ? 16 * 256 : 0;         // sign-byte table (floats)
  static constexpr int vval = 1 << (2 * VB);               // values of one pair field
  static constexpr int vlut = vval * 32;                   // half2 words, replicated per lane
};

struct Decode2Args {
  const uint8_t *k_codes;
  const float *k_norm;
  const uint8_t *k_signs;
  const float *k_rnorm;
  const uint8_t *v_codes;
  const float *v_norm;
  const uint8_t *v_signs;
  const float *v_rnorm;
  int capacity, heads_kv, heads_q, chunk, splits;
  const int32_t *seq_lens;
  const float *qprep;
  float *partials;
  const float *k_centroids;
  const float *v_centroids;
  int *error;
};

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float half_lo_f(uint32_t h2) {
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}
__device__ __forceinline__ float half_hi_f(uint32_t h2) {
  return __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// 2*VB-bit field n (n = 0..15) of a thread's contiguous 32*VB-bit span
template <int VB>
__device__ __forceinline__ uint32_t span_field(const uint32_t (&w)[VB], int n) {
  constexpr int F = 2 * VB;
  const int bit = F * n, wi = bit >> 5, off = bit & 31;
  uint32_t v;
  if (off + F <= 32 || wi + 1 >= VB) v = w[wi] >> off;
  else v = __funnelshift_r(w[wi], w[wi + 1], off);
  return v & ((1u << F) - 1u);
}

template <int KB, int VB, bool KQJL, bool VQJL>
__global__ void __launch_bounds__(kWarps2 * 32, 2) decode2_g1_kernel(Decode2Args a) {
  using Gm = Geo<KB, VB, KQJL, VQJL>;
  extern __shared__ __align__(1024) unsigned char smem[];
  // the value table sits first so that (field << 7) | (lane << 2) needs no base add
  uint32_t *s_vlut = reinterpret_cast<uint32_t *>(smem);                // [vval][32]
  float *s_ktab = reinterpret_cast<float *>(s_vlut + Gm::vlut);         // [kval][kpos]
  float *s_stab = s_ktab + Gm::ktab;                                    // [256][16]
  unsigned char *s_stage = reinterpret_cast<unsigned char *>(s_stab + Gm::stab);
  uint64_t *s_full = reinterpret_cast<uint64_t *>(s_stage + kStages * Gm::stage);
  float *s_q = reinterpret_cast<float *>(s_full + kStages);       // [128] q_rot / sqrt(d), [128] S q
  float *s_m = s_q + 2 * kD;                                       // [warps]
  float *s_l = s_m + kWarps2;
  float *s_wsum = s_l + kWarps2;
  float *s_acc = s_wsum + kWarps2;                                 // [warps][128]
  float *s_sacc = s_acc + kWarps2 * kD;                            // [warps][128]

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = min(max(__ldg(a.seq_lens + b), 0), a.capacity);
  const int t_begin = split * a.chunk;
  const int t_end = min(t_begin + a.chunk, len);
  const int ntiles = (t_end > t_begin) ? (t_end - t_begin + kTT - 1) / kTT : 0;
  const size_t slot0 = ((size_t)b * a.heads_kv + hk) * a.capacity;
  const int hq = hk;  // one query head per KV head

  // ---------------- prologue: barriers, first TMA stages, tables
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&s_full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto issue_tile = [&](int tile) {
    const int stage = tile % kStages;
    unsigned char *st = s_stage + stage * Gm::stage;
    const int t0 = t_begin + tile * kTT;
    const int n = min(kTT, t_end - t0);
    const int n4 = (n + 3) & ~3;  // norms in 16-byte units
    uint32_t bytes = n * Gm::kc + n4 * 4 + n * Gm::vc + n4 * 4;
    if (KQJL) bytes += n * 16 + n4 * 4;
    if (VQJL) bytes += n * 16 + n4 * 4;
    mbar_arrive_expect_tx(&s_full[stage], bytes);
    const size_t s0 = slot0 + t0;
    tma_load_1d(st + Gm::off_kc, a.k_codes + s0 * Gm::kc, n * Gm::kc, &s_full[stage]);
    tma_load_1d(st + Gm::off_kn, a.k_norm + s0, n4 * 4, &s_full[stage]);
    if (KQJL) {
      tma_load_1d(st + Gm::off_ks, a.k_signs + s0 * 16, n * 16, &s_full[stage]);
      tma_load_1d(st + Gm::off_kr, a.k_rnorm + s0, n4 * 4, &s_full[stage]);
    }
    tma_load_1d(st + Gm::off_vc, a.v_codes + s0 * Gm::vc, n * Gm::vc, &s_full[stage]);
    tma_load_1d(st + Gm::off_vn, a.v_norm + s0, n4 * 4, &s_full[stage]);
    if (VQJL) {
      tma_load_1d(st + Gm::off_vs, a.v_signs + s0 * 16, n * 16, &s_full[stage]);
      tma_load_1d(st + Gm::off_vr, a.v_rnorm + s0, n4 * 4, &s_full[stage]);
    }
  };
  if (tid == 0)
    for (int i = 0; i < kStages && i < ntiles; ++i) issue_tile(i);

  // prepared query (already rotated and scaled by 1/sqrt(d); S q scaled by sqrt(pi/2)/m/sqrt(d))
  const float *qp = a.qprep + ((size_t)b * a.heads_q + hq) * 2 * kD;
  s_q[tid] = __ldg(qp + tid);
  if (KQJL) s_q[kD + tid] = __ldg(qp + kD + tid);
  __syncthreads();

  // key table: position pos of a record covers codes of coordinates by the slot order
  {
    const float *kc = a.k_centroids;
    for (int e = tid; e < Gm::ktab; e += blockDim.x) {
      const int v = e / Gm::kpos, pos = e % Gm::kpos;
      float acc = 0.f;
      if (KB == 3) {
        const int s = pos, t = s >> 4, n = s & 15, p = 4 * n + t;
        acc = s_q[2 * p] * __ldg(kc + (v & 7)) + s_q[2 * p + 1] * __ldg(kc + (v >> 3));
      } else {
        constexpr int per = 8 / (2 * KB);  // slots per byte
#pragma unroll
        for (int u = 0; u < per; ++u) {
          const int s = pos * per + u, t = s >> 4, n = s & 15, p = 4 * n + t;
          const int f = (v >> (2 * KB * u)) & ((1 << (2 * KB)) - 1);
          acc += s_q[2 * p] * __ldg(kc + (f & ((1 << KB) - 1))) + s_q[2 * p + 1] * __ldg(kc + (f >> KB));
        }
      }
      s_ktab[e] = acc;
    }
    if (KQJL) {
      // sign byte at position pos (0..15) covers slots 4pos..4pos+3 of the 1-bit layout
      for (int e = tid; e < 16 * 256; e += blockDim.x) {
        const int v = e >> 4, pos = e & 15;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s = 4 * pos + u, t = s >> 4, n = s & 15, p = 4 * n + t;
          acc += ((v >> (2 * u)) & 1 ? 1.f : -1.f) * s_q[kD + 2 * p] +
                 ((v >> (2 * u + 1)) & 1 ? 1.f : -1.f) * s_q[kD + 2 * p + 1];
        }
        s_stab[e] = acc;
      }
    }
    // value pair table: field f -> half2(c[f & mask], c[f >> VB]), replicated for every lane
    const float *vcb = a.v_centroids;
    for (int e = tid; e < Gm::vlut; e += blockDim.x) {
      const int f = e >> 5;
      s_vlut[e] = pack_half2(__ldg(vcb + (f & ((1 << VB) - 1))), __ldg(vcb + (f >> VB)));
    }
  }
  __syncthreads();

  // ---------------- per-lane constants
  const uint32_t ktab_sa = smem_u32(s_ktab);
  const int half = lane >> 4, l = lane & 15;
  const int g = lane >> 2, t4 = lane & 3;
  // reduce-scatter result: lane l (within its half) holds step sigma(l)
  const int my_step = 4 * ((l >> 3) & 1) + 2 * ((l >> 2) & 1) + ((l >> 1) & 1);
  float m_run = -INFINITY, l_run = 0.f, wsum = 0.f;
  float dv[8][4], ds[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int j = 0; j < 4; ++j) dv[mb][j] = ds[mb][j] = 0.f;

  // A wait that runs out of time (it never should) records TQ_ERR_TIMEOUT; the
  // CTA then stops waiting and computing but still reaches every barrier, so
  // no thread is left behind. Its partial record is then meaningless, which the
  // error word reports.
  bool bad = false;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile % kStages;
    const uint32_t parity = (tile / kStages) & 1;
    if (!bad && !mbar_wait_bounded(&s_full[stage], parity, a.error)) bad = true;
    bad = __any_sync(kFull, bad);  // whole warps skip together (the body shuffles)
    if (bad) {
      __syncthreads();
      continue;
    }
    const unsigned char *st = s_stage + stage * Gm::stage;
    const int t0 = t_begin + tile * kTT;
    const int wbase = warp * 16;  // this warp's first token within the tile
    const float *kn = reinterpret_cast<const float *>(st + Gm::off_kn);
    const float *vn = reinterpret_cast<const float *>(st + Gm::off_vn);

    // ---- scores: 8 steps of 2 tokens, 16 lanes per token
    float part[8];
#pragma unroll
    for (int step = 0; step < 8; ++step) {
      const int lt = wbase + 2 * step + half;
      const float nu = kn[lt];
      const unsigned char *rec = st + Gm::off_kc + lt * Gm::kc;
      float acc = 0.f;
      if (KB == 4) {
        // lane l owns bytes 4l..4l+3; byte kk of word w indexes T[v][4l + kk]; the
        // byte address (v << 8) | (4 pos) comes from one byte permute
        const uint32_t w = reinterpret_cast<const uint32_t *>(rec)[l];
        float t[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int kk = (k + (lane >> 3)) & 3;
          const uint32_t off = __byte_perm(w, (uint32_t)(4 * (4 * l + kk)), 0x4440u | (uint32_t)kk << 4);
          t[k] = ld_shared_f32(ktab_sa + off);
        }
        acc = (t[0] + t[1]) + (t[2] + t[3]);
      } else if (KB == 2) {
        const uint32_t w = reinterpret_cast<const uint32_t *>(rec)[l >> 1] >> (16 * (l & 1));
        float t[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int kk = (k + half) & 1;
          const int pos = 2 * l + kk;
          const uint32_t v = (w >> (8 * kk)) & 0xffu;
          t[k] = s_ktab[v * Gm::kpos + pos];
        }
        acc = t[0] + t[1];
      } else if (KB == 1) {
        const uint32_t v = rec[l];
        acc = s_ktab[v * Gm::kpos + l];
      } else {  // KB == 3: lane l owns slots 4l..4l+3 (24 bits at bit 24 l)
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(rec);
        const int bit = 24 * l, wi = bit >> 5, off = bit & 31;
        const uint32_t lo = rw[wi], hi = rw[(wi + 1 < 12) ? wi + 1 : wi];
        const uint32_t f24 = __funnelshift_r(lo, hi, off);
        float t[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int kk = (k + (lane >> 3)) & 3;
          const uint32_t v = (f24 >> (6 * kk)) & 63u;
          t[k] = s_ktab[v * Gm::kpos + 4 * l + kk];
        }
        acc = (t[0] + t[1]) + (t[2] + t[3]);
      }
      acc *= nu;
      if (KQJL) {
        const float rho = reinterpret_cast<const float *>(st + Gm::off_kr)[lt];
        const uint32_t v = (st + Gm::off_ks + lt * 16)[l];
        acc = fmaf(rho, s_stab[v * 16 + l], acc);
      }
      part[step] = acc;
    }
    // reduce-scatter 8 values over the 16 lanes of each half
    float r4[4], r2[2];
    {
      const bool hb = (l & 8) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float send = hb ? part[k] : part[k + 4];
        const float keep = hb ? part[k + 4] : part[k];
        r4[k] = keep + __shfl_xor_sync(kFull, send, 8);
      }
      const bool hb2 = (l & 4) != 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float send = hb2 ? r4[k] : r4[k + 2];
        const float keep = hb2 ? r4[k + 2] : r4[k];
        r2[k] = keep + __shfl_xor_sync(kFull, send, 4);
      }
    }
    const bool hb1 = (l & 2) != 0;
    float sc = (hb1 ? r2[1] : r2[0]) + __shfl_xor_sync(kFull, hb1 ? r2[0] : r2[1], 2);
    sc += __shfl_xor_sync(kFull, sc, 1);
    const int my_tok = wbase + 2 * my_step + half;
    const bool valid = t0 + my_tok < t_end;
    sc = valid ? sc : -INFINITY;

    // ---- online softmax over the warp's 16 tokens
    float tmax = sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
    const float m_new = fmaxf(m_run, tmax);
    const bool any = m_new != -INFINITY;  // at least one valid token seen by this warp
    const float scale = any ? __expf(m_run - m_new) : 1.f;
    const float p = valid ? __expf(sc - m_new) : 0.f;
    float psum = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(kFull, psum, o);
    l_run = l_run * scale + 0.5f * psum;  // every token sits on two lanes
    m_run = m_new;
    if (scale != 1.f) {  // warp-uniform: the running max moved
      wsum *= scale;
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dv[mb][j] *= scale;
          if (VQJL) ds[mb][j] *= scale;
        }
    }

    // ---- B operands: column 0 = this warp's 16 token weights, other columns 0
    // token j (0..15) of the warp sits on lane 16(j&1) + 8((j>>3)&1) + 4((j>>2)&1) + 2((j>>1)&1)
    uint32_t bh0, bh1, bl0, bl1, bs0 = 0, bs1 = 0;
    {
      float w[4], wr[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = 2 * t4 + (c & 1) + 8 * (c >> 1);
        const int src = 16 * (j & 1) + 8 * ((j >> 3) & 1) + 4 * ((j >> 2) & 1) + 2 * ((j >> 1) & 1);
        const float pj = __shfl_sync(kFull, p, src);
        const bool live = (g == 0) && (t0 + wbase + j < t_end);
        w[c] = live ? pj * vn[wbase + j] : 0.f;
        wr[c] = (live && VQJL) ? pj * reinterpret_cast<const float *>(st + Gm::off_vr)[wbase + j] : 0.f;
      }
      bh0 = pack_half2(w[0], w[1]);
      bh1 = pack_half2(w[2], w[3]);
      bl0 = pack_half2(w[0] - half_lo_f(bh0), w[1] - half_hi_f(bh0));
      bl1 = pack_half2(w[2] - half_lo_f(bh1), w[3] - half_hi_f(bh1));
      if (VQJL) {
        bs0 = pack_half2(wr[0], wr[1]);
        bs1 = pack_half2(wr[2], wr[3]);
        // the sign MMA runs on bits b (as 2^-14 b); sum_j w'_j sigma_j = 2 sum_j w'_j b_j - sum_j w'_j
        float ws = half_lo_f(bs0) + half_hi_f(bs0) + half_lo_f(bs1) + half_hi_f(bs1);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) ws += __shfl_xor_sync(kFull, ws, o);  // over t4 (g = 0 lanes)
        wsum += ws;
      }
    }

    // ---- values: decode (token, coordinate-pair) fp16 pairs, transpose, MMA
    {
      uint32_t w0[VB], w1[VB];
      const uint32_t *r0 = reinterpret_cast<const uint32_t *>(st + Gm::off_vc + (wbase + g) * Gm::vc);
      const uint32_t *r1 = reinterpret_cast<const uint32_t *>(st + Gm::off_vc + (wbase + 8 + g) * Gm::vc);
#pragma unroll
      for (int k = 0; k < VB; ++k) {
        w0[k] = r0[VB * t4 + k];
        w1[k] = r1[VB * t4 + k];
      }
      const uint32_t lane_sa = smem_u32(s_vlut) | (uint32_t)(lane << 2);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        const uint32_t x00 = movmatrix_t(ld_shared_u32(lane_sa | (span_field<VB>(w0, 2 * mb) << 7)));
        const uint32_t x01 = movmatrix_t(ld_shared_u32(lane_sa | (span_field<VB>(w0, 2 * mb + 1) << 7)));
        const uint32_t x10 = movmatrix_t(ld_shared_u32(lane_sa | (span_field<VB>(w1, 2 * mb) << 7)));
        const uint32_t x11 = movmatrix_t(ld_shared_u32(lane_sa | (span_field<VB>(w1, 2 * mb + 1) << 7)));
        mma_16816(dv[mb], x00, x01, x10, x11, bh0, bh1);
        mma_16816(dv[mb], x00, x01, x10, x11, bl0, bl1);
      }
    }

    // ---- QJL signs: A(coords x tokens) as 0/1 fp16 pairs built from two tokens' sign words
    if (VQJL) {
      // coordinate 16mb + g (+8) of token j: sign word (g>>1)&3, bit 4mb + (g&1) (+2)
      const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + Gm::off_vs);
      const int wsel = (g >> 1) & 3, e = g & 1;
      const uint32_t wa0 = sw[(wbase + 2 * t4) * 4 + wsel], wb0 = sw[(wbase + 2 * t4 + 1) * 4 + wsel];
      const uint32_t wa1 = sw[(wbase + 2 * t4 + 8) * 4 + wsel], wb1 = sw[(wbase + 2 * t4 + 9) * 4 + wsel];
      // low halves of the two tokens' words side by side (token 2t in bits 0..15, 2t+1 in 16..31)
      const uint32_t lo0 = __byte_perm(wa0, wb0, 0x5410), hi0 = __byte_perm(wa0, wb0, 0x7632);
      const uint32_t lo1 = __byte_perm(wa1, wb1, 0x5410), hi1 = __byte_perm(wa1, wb1, 0x7632);
      // a set bit becomes the fp16 value 2^-14 (bit 10, the smallest normal): one
      // shift lands bits k and 16 + k on bits 10 and 26; the merge rescales by 2^14
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        const int sh0 = (4 * mb + e) & 15, sh1 = (4 * mb + 2 + e) & 15;
        const uint32_t s0 = (mb < 4) ? lo0 : hi0, s1 = (mb < 4) ? lo1 : hi1;
        const uint32_t a0 = __funnelshift_l(s0, s0, 10 - sh0 + 32) & 0x04000400u;
        const uint32_t a2 = __funnelshift_l(s0, s0, 10 - sh1 + 32) & 0x04000400u;
        const uint32_t a4 = __funnelshift_l(s1, s1, 10 - sh0 + 32) & 0x04000400u;
        const uint32_t a6 = __funnelshift_l(s1, s1, 10 - sh1 + 32) & 0x04000400u;
        mma_16816(ds[mb], a0, a2, a4, a6, bs0, bs1);
      }
    }

    __syncthreads();  // every warp is done with this stage
    if (tid == 0 && !bad && tile + kStages < ntiles) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_tile(tile + kStages);
    }
  }

  // ---------------- merge the warps and write this chunk's partial record
  if (lane == 0) {
    s_m[warp] = m_run;
    s_l[warp] = l_run;
    s_wsum[warp] = wsum;
  }
  if (t4 == 0) {  // column 0 of the accumulators: coordinates 16mb + g and 16mb + 8 + g
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      s_acc[warp * kD + 16 * mb + g] = dv[mb][0];
      s_acc[warp * kD + 16 * mb + 8 + g] = dv[mb][2];
      if (VQJL) {
        s_sacc[warp * kD + 16 * mb + g] = ds[mb][0];
        s_sacc[warp * kD + 16 * mb + 8 + g] = ds[mb][2];
      }
    }
  }
  __syncthreads();
  const int i = tid;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps2; ++w) M = fmaxf(M, s_m[w]);
  float L = 0.f, A = 0.f, Sg = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps2; ++w) {
    const float e = (s_m[w] == -INFINITY) ? 0.f : __expf(s_m[w] - M);
    L += s_l[w] * e;
    A += s_acc[w * kD + i] * e;
    if (VQJL) Sg += (2.f * 16384.f * s_sacc[w * kD + i] - s_wsum[w]) * e;
  }
  float *rec = a.partials + (((size_t)b * a.heads_q + hq) * a.splits + split) * kPartialFloats;
  if (i == 0) {
    rec[0] = M;
    rec[1] = L;
  }
  rec[2 + i] = A;
  rec[2 + kD + i] = Sg;
}

template <int KB, int VB, bool KQJL, bool VQJL>
size_t smem_bytes() {
  using Gm = Geo<KB, VB, KQJL, VQJL>;
  return sizeof(float) * (Gm::ktab + Gm::stab) + sizeof(uint32_t) * Gm::vlut + kStages * Gm::stage +
         kStages * sizeof(uint64_t) + sizeof(float) * (2 * kD + 3 * kWarps2 + 2 * kWarps2 * kD);
}

template <int KB, int VB, bool KQJL, bool VQJL>
int launch2(const Decode2Args &k, dim3 grid, cudaStream_t st) {
  const size_t smem = smem_bytes<KB, VB, KQJL, VQJL>();
  auto fn = decode2_g1_kernel<KB, VB, KQJL, VQJL>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  fn<<<grid, kWarps2 * 32, smem, st>>>(k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

// Returns TQ_ERR_UNSUPPORTED when this path does not cover the request (the
// caller then uses the general kernel).
int launch_decode2_g1(const DecodeArgs &a, const float *qprep, float *partials, void *stream) {
  const tq_ctx *ctx = a.ctx;
  if (a.heads_q != a.heads_kv) return TQ_ERR_UNSUPPORTED;
  if (a.cache->capacity % 16) return TQ_ERR_UNSUPPORTED;  // TMA sources need 16-byte aligned rows
  if (a.chunk % 4) return TQ_ERR_UNSUPPORTED;              // tile starts stay 16-byte aligned
  const tq_cache *c = a.cache;
  Decode2Args k{};
  k.k_codes = c->k_codes; k.k_norm = c->k_norm; k.k_signs = c->k_signs; k.k_rnorm = c->k_rnorm;
  k.v_codes = c->v_codes; k.v_norm = c->v_norm; k.v_signs = c->v_signs; k.v_rnorm = c->v_rnorm;
  k.capacity = c->capacity;
  k.heads_kv = a.heads_kv;
  k.heads_q = a.heads_q;
  k.chunk = a.chunk;
  k.splits = a.splits;
  k.seq_lens = a.seq_lens;
  k.qprep = qprep;
  k.partials = partials;
  k.k_centroids = ctx->dparams->k_centroids;
  k.v_centroids = ctx->dparams->v_centroids;
  k.error = &ctx->dparams->error;
  dim3 grid(a.splits, a.heads_kv, a.batch);
  cudaStream_t st = (cudaStream_t)stream;
  const int kb = ctx->k.bits;
  switch (ctx->scheme) {
    case TQ_SCHEME_KV:
      if (kb == 2) return launch2<2, 2, false, false>(k, grid, st);
      if (kb == 3) return launch2<3, 3, false, false>(k, grid, st);
      if (kb == 4) return launch2<4, 4, false, false>(k, grid, st);
      break;
    case TQ_SCHEME_KQV:
      if (kb == 2) return launch2<2, 1, false, true>(k, grid, st);
      if (kb == 3) return launch2<3, 2, false, true>(k, grid, st);
      if (kb == 4) return launch2<4, 3, false, true>(k, grid, st);
      break;
    case TQ_SCHEME_QKQV:
      if (kb == 1) return launch2<1, 1, true, true>(k, grid, st);
      if (kb == 2) return launch2<2, 2, true, true>(k, grid, st);
      if (kb == 3) return launch2<3, 3, true, true>(k, grid, st);
      break;
    default: break;
  }
  return TQ_ERR_UNSUPPORTED;
}

}  // namespace tq
