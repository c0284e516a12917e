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
//   the last warp done with a stage refills it, so warps never wait on one
//   another inside the token loop;
// * keys: per CTA a float32 table T[v][pos] = sum over the coordinates a code
//   position covers of q_rot[i] c[code_i(v)] turns each token's score into one
//   lookup per byte (or 6-bit slot) of its record -- fp32 throughout, so scores
//   keep full precision whatever the key scale. The table is built as an outer
//   sum of two per-position half tables, one add per entry;
// * values and QJL signs: the p-weighted sums over a warp's 16 tokens run on
//   the tensor cores (mma.sync m16n8k16, fp32 accumulate) into ONE accumulator:
//   B column 0/1 carry the fp16 hi/lo parts of p nu (values), columns 2/3 the
//   hi/lo parts of p rho (signs). Value codes are decoded to fp16 pairs through
//   a per-lane replicated table and transposed with movmatrix; a sign bit
//   becomes a power of two (its bit moved into the fp16 exponent field by one
//   rotate, isolated by one AND), undone per accumulator row at the merge.
//
// CTA: 4 warps, one (batch, kv head, chunk). A warp owns 16 tokens of each
// 64-token tile: it scores them (16 lanes per token, 2 tokens per step), takes
// the online-softmax step (base-2 exponent; the log2(e) factor sits in the
// key tables) and issues the value / sign MMAs.

#include <cuda_fp16.h>

#include "tq_ptx.cuh"

namespace tq {
namespace {

constexpr int kWarps2 = 4;
constexpr int kTT = 64;     // tokens per tile
constexpr int kStages = 3;  // TMA pipeline depth (two CTAs per SM fit in shared memory)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

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
  // key table: positions per record (bytes, or 6-bit pair slots) and values per position
  static constexpr int kpos = (KB == 3) ? 64 : 16 * KB;
  static constexpr int kval = (KB == 3) ? 64 : 256;
  static constexpr int ktab = kpos * kval;                 // floats; row v holds kpos entries
  static constexpr int stab = KQJL ? 16 * 256 : 0;         // sign-byte table [256][16] (floats)
  static constexpr int vval = 1 << (2 * VB);               // values of one value pair field
  static constexpr int vlut = vval * 32;                   // half2 words, replicated per lane
  // shared-memory offsets (bytes from the dynamic base): value table first
  static constexpr int sm_ktab = vlut * 4;
  static constexpr int sm_stab = sm_ktab + ktab * 4;
  static constexpr int sm_stage = sm_stab + stab * 4;
  static constexpr int sm_bar = sm_stage + kStages * stage;
  static constexpr int sm_cnt = sm_bar + kStages * 8;
  static constexpr int sm_q = sm_cnt + 16;                 // [2][128] floats
  static constexpr int sm_m = sm_q + 2 * kD * 4;           // [warps] x 3 floats
  static constexpr int sm_acc = sm_m + 3 * kWarps2 * 4;    // [warps][128] floats, values
  static constexpr int sm_sacc = sm_acc + kWarps2 * kD * 4;  // [warps][128] floats, signs
  static constexpr int total = sm_sacc + kWarps2 * kD * 4;
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

__device__ __forceinline__ uint32_t rotr(uint32_t w, uint32_t r) { return __funnelshift_r(w, w, r); }

// coordinate of code offset o in the pair-slot order (coordinate 8n + 2t + e at 32t + 2n + e)
__device__ __forceinline__ int slot_coord(int o) {
  const int ps = o >> 1, e = o & 1;
  return 8 * (ps & 15) + 2 * (ps >> 4) + e;
}

// Lookup table T[v][pos] (row stride KPOS floats): the sum, over the CPP codes
// that value v packs at position pos (code offsets pos*CPP + j, CB bits each),
// of q[coord] * cb[code]. Built as lo[v & low bits] + hi[v >> LOB]: each
// thread owns one position and a slice of the high values. SIGN: cb = {-1, +1}.
template <int CB, int KPOS, int VBITS, bool SIGN>
__device__ __forceinline__ void build_lookup(float *T, const float *q, const float *cb_g, float scale, int tid) {
  constexpr int CPP = VBITS / CB;
  constexpr int LOB = (VBITS >= 8) ? 4 : 3;  // low-part bits (a whole number of codes)
  constexpr int HIB = VBITS - LOB;
  constexpr int NLO = 1 << LOB, PARTS = 128 / KPOS, NH = (1 << HIB) / PARTS;
  constexpr int M = (1 << CB) - 1;
  const int pos = tid % KPOS, part = tid / KPOS;
  float qv[CPP];
#pragma unroll
  for (int j = 0; j < CPP; ++j) qv[j] = q[slot_coord(pos * CPP + j)] * scale;
  float cb[M + 1];
#pragma unroll
  for (int c = 0; c <= M; ++c) cb[c] = SIGN ? (c ? 1.f : -1.f) : __ldg(cb_g + c);
  float lo[NLO];
#pragma unroll
  for (int x = 0; x < NLO; ++x) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < LOB / CB; ++j) acc = fmaf(qv[j], cb[(x >> (CB * j)) & M], acc);
    lo[x] = acc;
  }
#pragma unroll 1
  for (int yy = 0; yy < NH; ++yy) {
    const int y = part * NH + yy;
    float hi = 0.f;
#pragma unroll
    for (int j = 0; j < HIB / CB; ++j) {
      const int c = (y >> (CB * j)) & M;
      hi = fmaf(qv[LOB / CB + j], SIGN ? (c ? 1.f : -1.f) : __ldg(cb_g + c), hi);
    }
#pragma unroll
    for (int x = 0; x < NLO; ++x) T[((y << LOB) | x) * KPOS + pos] = lo[x] + hi;
  }
}

// landing bit (10..14) of sign bit k (0..15) of a half-word, and the rotation that takes it there
__host__ __device__ constexpr int sign_land(int k) { return k <= 4 ? k + 10 : (k <= 9 ? k + 5 : (k <= 14 ? k : 10)); }
__host__ __device__ constexpr int sign_rot(int k) { return k <= 4 ? 10 : (k <= 9 ? 5 : (k <= 14 ? 0 : 27)); }
// 1 / (fp16 value whose only set bit is bit L, 10 <= L <= 14): 2^(15 - 2^(L-10))
__device__ __forceinline__ float sign_unscale(int L) {
  return L == 10 ? 16384.f : (L == 11 ? 8192.f : (L == 12 ? 2048.f : (L == 13 ? 128.f : 0.5f)));
}

template <int KB, int VB, bool KQJL, bool VQJL>
__global__ void __launch_bounds__(kWarps2 * 32, 2) decode2_g1_kernel(Decode2Args a) {
  using Gm = Geo<KB, VB, KQJL, VQJL>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_vlut = smem;  // [vval][32] half2 words, at offset 0
  float *s_ktab = reinterpret_cast<float *>(smem + Gm::sm_ktab);
  float *s_stab = reinterpret_cast<float *>(smem + Gm::sm_stab);
  unsigned char *s_stage = smem + Gm::sm_stage;
  uint64_t *s_full = reinterpret_cast<uint64_t *>(smem + Gm::sm_bar);
  unsigned *s_cnt = reinterpret_cast<unsigned *>(smem + Gm::sm_cnt);
  float *s_q = reinterpret_cast<float *>(smem + Gm::sm_q);  // [128] q_rot / sqrt(d), [128] scaled S q
  float *s_m = reinterpret_cast<float *>(smem + Gm::sm_m);  // [warps] max, [warps] sum, [warps] sign weight sum
  float *s_acc = reinterpret_cast<float *>(smem + Gm::sm_acc);
  float *s_sacc = reinterpret_cast<float *>(smem + Gm::sm_sacc);

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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&s_full[s], 1);
      s_cnt[s] = 0;
    }
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

  // key tables carry log2(e) so that scores come out in base-2 units
  if constexpr (KB == 3) build_lookup<3, 64, 6, false>(s_ktab, s_q, a.k_centroids, kLog2e, tid);
  else build_lookup<KB, 16 * KB, 8, false>(s_ktab, s_q, a.k_centroids, kLog2e, tid);
  if constexpr (KQJL) build_lookup<1, 16, 8, true>(s_stab, s_q + kD, nullptr, kLog2e, tid);
  {
    // value pair table: field f -> half2(c[f & mask], c[f >> VB]), replicated for every lane
    const float *vcb = a.v_centroids;
    uint32_t *vl = reinterpret_cast<uint32_t *>(s_vlut);
    for (int e = tid; e < Gm::vlut; e += blockDim.x) {
      const int f = e >> 5;
      vl[e] = pack_half2(__ldg(vcb + (f & ((1 << VB) - 1))), __ldg(vcb + (f >> VB)));
    }
  }
  __syncthreads();

  // ---------------- per-lane constants
  const int half = lane >> 4, l = lane & 15;
  const int g = lane >> 2, t4 = lane & 3;
  // key lookups: byte offset into T from (record word, constant, selector / rotation)
  uint32_t kcon[4], ksel[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (KB == 4 || KB == 3) {
      const int kk = (k + (lane >> 3)) & 3;  // staggered so that the 32 lanes hit 32 banks
      kcon[k] = 4u * (4 * l + kk);
      ksel[k] = (KB == 4) ? (0x5504u | ((uint32_t)kk << 4)) : (uint32_t)((6 * kk - 8) & 31);
    } else if (KB == 2) {
      const int jj = (k + half) & 1, bpos = 2 * l + jj;
      kcon[k] = 4u * bpos;
      ksel[k] = (uint32_t)((8 * (bpos & 3) - 7) & 31);
    } else {
      kcon[k] = 4u * l;
      ksel[k] = (uint32_t)((8 * (l & 3) - 6) & 31);
    }
  }
  const uint32_t ssel = (uint32_t)((8 * (l & 3) - 6) & 31);  // key sign byte l -> row offset (64-byte rows)
  // reduce-scatter result: lane l (within its half) holds step sigma(l); token j = 2 sigma + half
  const int my_step = 4 * ((l >> 3) & 1) + 2 * ((l >> 2) & 1) + ((l >> 1) & 1);
  const int my_j = 2 * my_step + half;
  // B gather: token j of the warp sits on lanes 16(j&1) + 8((j>>3)&1) + 4((j>>2)&1) + 2((j>>1)&1) (+1);
  // the even lane carries p nu, the odd one p rho
  int bsrc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = 2 * t4 + (c & 1) + 8 * (c >> 1);
    bsrc[c] = 16 * (j & 1) + 8 * ((j >> 3) & 1) + 4 * ((j >> 2) & 1) + 2 * ((j >> 1) & 1) + ((g >> 1) & 1);
  }
  const uint32_t bsel = (g & 1) ? 0x7632u : 0x5410u;  // hi parts (even g) or lo parts (odd g)
  const bool bv_live = g < 2, bs_live = (g >> 1) == 1;
  const uint32_t lane4 = (uint32_t)lane << 2;
  // sign operands: this thread's rows are half (g & 1) of sign word (g >> 1)
  const uint32_t swsel = (g & 1) ? 0x7632u : 0x5410u;

  float m_run = -INFINITY, l_run = 0.f, w_run = 0.f;
  float acc[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[mb][j] = 0.f;

  // A wait that runs out of time (it never should) records TQ_ERR_TIMEOUT; the
  // warp then stops waiting and computing but keeps releasing its stages, so
  // no warp is left behind. The partial record is then meaningless, which the
  // error word reports.
  bool bad = false;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile % kStages;
    const uint32_t parity = (tile / kStages) & 1;
    if (!bad && !mbar_wait_bounded(&s_full[stage], parity, a.error)) bad = true;
    bad = __any_sync(kFull, bad);  // whole warps skip together (the body shuffles)
    const unsigned char *st = s_stage + stage * Gm::stage;
    const int t0 = t_begin + tile * kTT;
    const int wbase = warp * 16;  // this warp's first token within the tile
    if (!bad) {
      const float *kn = reinterpret_cast<const float *>(st + Gm::off_kn);
      const float *kr = reinterpret_cast<const float *>(st + Gm::off_kr);

      // ---- scores: 8 steps of 2 tokens, 16 lanes per token
      float part[8];
#pragma unroll
      for (int step = 0; step < 8; ++step) {
        const int lt = wbase + 2 * step + half;
        const uint32_t *rec = reinterpret_cast<const uint32_t *>(st + Gm::off_kc + lt * Gm::kc);
        const unsigned char *tb = reinterpret_cast<const unsigned char *>(s_ktab);
        float sum;
        if (KB == 4) {
          const uint32_t w = rec[l];
          float t[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) t[k] = *reinterpret_cast<const float *>(tb + __byte_perm(w, kcon[k], ksel[k]));
          sum = (t[0] + t[1]) + (t[2] + t[3]);
        } else if (KB == 3) {
          // lane l owns pair slots 4l..4l+3 (24 bits at bit 24 l)
          const int bit = 24 * l, wi = bit >> 5, off = bit & 31;
          const uint32_t f24 = __funnelshift_r(rec[wi], rec[(wi + 1 < 12) ? wi + 1 : wi], off);
          float t[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            t[k] = *reinterpret_cast<const float *>(tb + ((rotr(f24, ksel[k]) & 0x3F00u) | kcon[k]));
          sum = (t[0] + t[1]) + (t[2] + t[3]);
        } else if (KB == 2) {
          const uint32_t w = rec[l >> 1];
          float t[2];
#pragma unroll
          for (int k = 0; k < 2; ++k)
            t[k] = *reinterpret_cast<const float *>(tb + ((rotr(w, ksel[k]) & 0x7F80u) | kcon[k]));
          sum = t[0] + t[1];
        } else {
          const uint32_t w = rec[l >> 2];
          sum = *reinterpret_cast<const float *>(tb + ((rotr(w, ksel[0]) & 0x3FC0u) | kcon[0]));
        }
        if (KQJL) {
          const uint32_t *srec = reinterpret_cast<const uint32_t *>(st + Gm::off_ks + lt * 16);
          const uint32_t w = srec[l >> 2];
          const float ts = *reinterpret_cast<const float *>(reinterpret_cast<const unsigned char *>(s_stab) +
                                                            ((rotr(w, ssel) & 0x3FC0u) | (4u * l)));
          sum = fmaf(kr[lt], ts, kn[lt] * sum);
        }
        part[step] = sum;
      }
      // reduce-scatter 8 values over the 16 lanes of each half
      float sc;
      {
        float r4[4], r2[2];
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
        const bool hb1 = (l & 2) != 0;
        sc = (hb1 ? r2[1] : r2[0]) + __shfl_xor_sync(kFull, hb1 ? r2[0] : r2[1], 2);
        sc += __shfl_xor_sync(kFull, sc, 1);
      }
      const int tok = wbase + my_j;
      const bool valid = t0 + tok < t_end;
      if (!KQJL) sc *= kn[tok];
      sc = valid ? sc : -INFINITY;

      // ---- online softmax over the warp's 16 tokens (base 2)
      float tmax = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
      const float m_new = fmaxf(m_run, tmax);
      const float p = valid ? ex2_approx(sc - m_new) : 0.f;
      if (m_new != m_run) {  // warp-uniform: the running max moved (m_run = -inf scales zeros)
        const float scale = ex2_approx(m_run - m_new);
        l_run *= scale;
        w_run *= scale;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[mb][j] *= scale;
        m_run = m_new;
      }
      l_run += p;  // every token sits on two lanes: halved at the merge

      // ---- B operands: this lane's token weight (p nu on even lanes, p rho on odd ones)
      // as an fp16 hi/lo pair, gathered into column g of the MMA's B fragment
      uint32_t bv0, bv1, bs0 = 0, bs1 = 0;
      {
        const bool odd = VQJL && (lane & 1);
        const float *wsrc = reinterpret_cast<const float *>(st + (odd ? Gm::off_vr : Gm::off_vn));
        const float wv = valid ? p * wsrc[tok] : 0.f;
        w_run += wv;  // sum of p rho over the odd lanes (the even ones are ignored)
        const __half hh = __float2half_rn(wv);
        const float rem = wv - __half2float(hh);
        const uint32_t hl = (uint32_t)__half_as_ushort(hh) | ((uint32_t)__half_as_ushort(__float2half_rn(rem)) << 16);
        const uint32_t x0 = __shfl_sync(kFull, hl, bsrc[0]);
        const uint32_t x1 = __shfl_sync(kFull, hl, bsrc[1]);
        const uint32_t x2 = __shfl_sync(kFull, hl, bsrc[2]);
        const uint32_t x3 = __shfl_sync(kFull, hl, bsrc[3]);
        const uint32_t b0 = __byte_perm(x0, x1, bsel), b1 = __byte_perm(x2, x3, bsel);
        bv0 = bv_live ? b0 : 0u;
        bv1 = bv_live ? b1 : 0u;
        if (VQJL) {
          bs0 = bs_live ? b0 : 0u;
          bs1 = bs_live ? b1 : 0u;
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
        // field n of a span -> byte offset (field << 7) | (lane << 2) of the value table
        auto lut = [&](const uint32_t(&w)[VB], int n) -> uint32_t {
          constexpr int F = 2 * VB;
          constexpr uint32_t mask = ((1u << F) - 1u) << 7;
          const int bit = F * n, wi = bit >> 5, off = bit & 31;
          uint32_t x;
          if (off < 7) x = w[wi] << (7 - off);
          else x = __funnelshift_r(w[wi], w[(wi + 1 < VB) ? wi + 1 : wi], off - 7);
          return *reinterpret_cast<const uint32_t *>(s_vlut + ((x & mask) | lane4));
        };
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          const uint32_t x00 = movmatrix_t(lut(w0, 2 * mb));
          const uint32_t x01 = movmatrix_t(lut(w0, 2 * mb + 1));
          const uint32_t x10 = movmatrix_t(lut(w1, 2 * mb));
          const uint32_t x11 = movmatrix_t(lut(w1, 2 * mb + 1));
          mma_16816(acc[mb], x00, x01, x10, x11, bv0, bv1);
        }
      }

      // ---- QJL signs: rows of this thread = bits of half (g & 1) of sign word (g >> 1)
      if (VQJL) {
        const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + Gm::off_vs);
        const int wsel = g >> 1;
        const uint32_t wa0 = sw[(wbase + 2 * t4) * 4 + wsel], wb0 = sw[(wbase + 2 * t4 + 1) * 4 + wsel];
        const uint32_t wa1 = sw[(wbase + 2 * t4 + 8) * 4 + wsel], wb1 = sw[(wbase + 2 * t4 + 9) * 4 + wsel];
        // token 2t (8 + 2t) in bits 0..15, token 2t + 1 (9 + 2t) in bits 16..31
        const uint32_t s0 = __byte_perm(wa0, wb0, swsel), s1 = __byte_perm(wa1, wb1, swsel);
        const uint32_t s0r10 = rotr(s0, 22), s0r5 = rotr(s0, 27), s0r27 = rotr(s0, 5);
        const uint32_t s1r10 = rotr(s1, 22), s1r5 = rotr(s1, 27), s1r27 = rotr(s1, 5);
        auto pick = [&](int k, uint32_t r0, uint32_t r5, uint32_t r10, uint32_t r27) -> uint32_t {
          const uint32_t src = sign_rot(k) == 10 ? r10 : (sign_rot(k) == 5 ? r5 : (sign_rot(k) == 0 ? r0 : r27));
          return src & (0x00010001u << sign_land(k));
        };
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          const uint32_t a0 = pick(2 * mb, s0, s0r5, s0r10, s0r27);
          const uint32_t a1 = pick(2 * mb + 1, s0, s0r5, s0r10, s0r27);
          const uint32_t a2 = pick(2 * mb, s1, s1r5, s1r10, s1r27);
          const uint32_t a3 = pick(2 * mb + 1, s1, s1r5, s1r10, s1r27);
          mma_16816(acc[mb], a0, a1, a2, a3, bs0, bs1);
        }
      }
    }

    // release the stage: the last of the four warps refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const unsigned old = atomicAdd(&s_cnt[stage], 1u);
      if ((old & (kWarps2 - 1)) == kWarps2 - 1 && tile + kStages < ntiles) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_tile(tile + kStages);
      }
    }
  }

  // ---------------- merge the warps and write this chunk's partial record
  {
    float lw = l_run, ww = (lane & 1) ? w_run : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lw += __shfl_xor_sync(kFull, lw, o);
      ww += __shfl_xor_sync(kFull, ww, o);
    }
    if (lane == 0) {
      s_m[warp] = m_run;
      s_m[kWarps2 + warp] = 0.5f * lw;
      s_m[2 * kWarps2 + warp] = ww;
    }
  }
  if (t4 == 0) {  // columns 0/1: value sums of coordinates 16mb + g and 16mb + 8 + g
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      s_acc[warp * kD + 16 * mb + g] = acc[mb][0] + acc[mb][1];
      s_acc[warp * kD + 16 * mb + 8 + g] = acc[mb][2] + acc[mb][3];
    }
  } else if (VQJL && t4 == 1) {  // columns 2/3: sign sums; row (mb, r) is bit 2mb + r of half g&1 of word g>>1
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const int c0 = 64 * (g & 1) + 8 * mb + 2 * (g >> 1);
      s_sacc[warp * kD + c0] = (acc[mb][0] + acc[mb][1]) * sign_unscale(sign_land(2 * mb));
      s_sacc[warp * kD + c0 + 1] = (acc[mb][2] + acc[mb][3]) * sign_unscale(sign_land(2 * mb + 1));
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
    const float e = (s_m[w] == -INFINITY) ? 0.f : ex2_approx(s_m[w] - M);
    L += s_m[kWarps2 + w] * e;
    A += s_acc[w * kD + i] * e;
    // the sign MMA summed p rho b over bits b; sum p rho sigma = 2 sum p rho b - sum p rho
    if (VQJL) Sg += (2.f * s_sacc[w * kD + i] - s_m[2 * kWarps2 + w]) * e;
  }
  float *rec = a.partials + (((size_t)b * a.heads_q + hq) * a.splits + split) * kPartialFloats;
  if (i == 0) {
    rec[0] = M * kLn2;  // natural-log units for the combine step
    rec[1] = L;
  }
  rec[2 + i] = A;
  rec[2 + kD + i] = Sg;
}

template <int KB, int VB, bool KQJL, bool VQJL>
size_t smem_bytes() {
  return (size_t)Geo<KB, VB, KQJL, VQJL>::total;
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
