// Decode attention over the packed cache, one query head per KV head, as two
// kernels that share one tile body:
//
// * decode_persist_kernel -- persistent: one CTA of 16 warps per SM walks
//   contiguous slices of the flattened (batch, kv head, 64-token tile) space,
//   so every SM gets the same number of tiles whatever the sequence lengths;
//   key tables are rebuilt only where a slice crosses into the next head, and
//   the TMA ring (up to 16 stages, ~140 KB in flight) keeps streaming across
//   that boundary: each warp streams and refills its own quarter of a stage on
//   its own mbarrier. Each (CTA, head) segment ends in one partial softmax record.
// * decode2_g1_kernel -- split-K over a fixed (batch, head, chunk) grid, for
//   batches too large for the persistent kernel's shared-memory prefix table.
// * decode_persist_kernel<..., true> -- the persistent kernel as one decode step:
//   it also computes the lengths after the step's append and the tile prefix,
//   appends the new key and value of every head whose last tile its slice holds
//   (before its ring's first copy, with S^T bulk-copied into the key-table area),
//   and rotates its own queries.
//
// Both compute softmax(q K_hat^T / sqrt(d)) V_hat with keys read through
// logits and values through the p-weighted sum in the rotated domain
// ("HeadQ", 2.1-2.2; "Statistical Inference ... Inspired by TurboQuant",
// technical summary, "K-V asymmetry", "Main contribution 1"):
//
// * record tiles of 64 tokens stream into shared memory through 1-D TMA bulk
//   copies, each completing on an mbarrier (bounded waits); the last warp
//   done with a stage refills it, so warps never wait on one another inside
//   the token loop;
// * keys: a float32 table T[v][pos] = sum over the coordinates a code
//   position covers of q_rot[i] c[code_i(v)] turns each token's score into one
//   lookup per byte (or 6-bit slot) of its record -- fp32 throughout, so scores
//   keep full precision whatever the key scale. The table is built as an outer
//   sum of two per-position half tables, one add per entry;
// * values and QJL signs: the p-weighted sums over a warp's 16 tokens run on
//   the tensor cores (mma.sync m16n8k16, fp32 accumulate) into ONE accumulator:
//   B column 0/1 carry the fp16 hi/lo parts of p nu (values), columns 2/3 the
//   hi/lo parts of p rho (signs). Value codes are stored pair-interleaved (two
//   tokens' codes of one coordinate side by side), so one lookup in a per-lane
//   replicated table gives an A-fragment register directly; a sign bit
//   becomes a power of two (its bit moved into the fp16 exponent field by one
//   rotate, isolated by one AND), undone per accumulator row at the merge.
//
// A warp owns 16 tokens of each tile it takes: it scores them (16 lanes per
// token, 2 tokens per step), takes the online-softmax step (base-2 exponent;
// the log2(e) factor sits in the key tables) and issues the value / sign MMAs.

#include <cuda_fp16.h>

#include <algorithm>

#include "tq_ptx.cuh"

namespace tq {
namespace {

constexpr int kTT = kDecodeTile;  // tokens per tile (4 warps x 16)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxPersistBatch = 256;  // prefix table held in shared memory

template <int KB, int VB, bool KQJL, bool VQJL, int NW, int S>
struct Geo {
  static constexpr int kStages = S;
  // per-token record bytes of each plane
  static constexpr int kc = 16 * KB, vc = 16 * VB;
  // a stage is four 16-token blocks of the blocked record layout, copied as they are
  // stored; plane offsets inside a block (bytes, every plane 16-byte aligned)
  static constexpr int off_kc = 0;
  static constexpr int off_kn = off_kc + 16 * kc;
  static constexpr int off_ks = off_kn + 16 * 4;
  static constexpr int off_kr = off_ks + (KQJL ? 16 * 16 : 0);
  static constexpr int off_vc = off_kr + (KQJL ? 16 * 4 : 0);
  static constexpr int off_vn = off_vc + 16 * vc;
  static constexpr int off_vs = off_vn + 16 * 4;
  static constexpr int off_vr = off_vs + (VQJL ? 16 * 16 : 0);
  static constexpr int block = off_vr + (VQJL ? 16 * 4 : 0);
  static constexpr int stage = 4 * block;
  // key table: positions per record (bytes, or 6-bit pair slots) and values per position
  static constexpr int kpos = (KB == 3) ? 64 : 16 * KB;
  static constexpr int kval = (KB == 3) ? 64 : 256;
  static constexpr int ktab = kpos * kval;                 // floats; row v holds kpos entries
  static constexpr int stab = KQJL ? 16 * 256 : 0;         // sign-byte table [256][16] (floats)
  static constexpr int vval = 1 << (2 * VB);               // values of one value pair field
  static constexpr int vlut = vval * 32;                   // half2 words, replicated per lane
  // shared-memory offsets (bytes from the dynamic base): value table first
  static constexpr int ktab_region = (ktab > NW * kPartialFloats) ? ktab : NW * kPartialFloats;
  static constexpr int sm_ktab = vlut * 4;
  static constexpr int sm_stab = sm_ktab + ktab_region * 4;
  static constexpr int sm_stage = sm_stab + stab * 4;
  static constexpr int sm_bar = sm_stage + S * stage;
  static constexpr int sm_cnt = sm_bar + S * 4 * 8;                 // (persistent: 4 barriers per stage)
  static constexpr int sm_q = sm_cnt + 16 * ((S * 4 + 15) / 16);   // [2][128] floats
  static constexpr int sm_misc = sm_q + 2 * kD * 4;
  // per-warp partial states are parked in the key-table area at a flush
};

// stages of the persistent kernel's ring: as many as fit next to the tables in
// 227 KB, a multiple of the 4 warp groups, at most 16
template <int KB, int VB, bool KQJL, bool VQJL>
constexpr int persist_stages() {
  using G1 = Geo<KB, VB, KQJL, VQJL, 16, 1>;
  constexpr int fixed = G1::sm_stage + 16 * 4 * 8 + 16 * 4 + 2 * kD * 4 + 4 * (2 * 256 + 1) + 4 * kMaxLevels + 64;
  constexpr int n = (227 * 1024 - fixed) / G1::stage;
  return (n >= 16) ? 16 : (n / 4) * 4;
}

struct Decode2Args {
  const uint8_t *records;  // blocked records: [sequence-head][cap16 / 16] blocks of `bb` bytes (or a pool)
  int bb, cap16;
  int capacity, batch, heads_kv, heads_q, chunk, splits;
  const int32_t *seq_lens;
  const int32_t *tile_prefix;  // persistent kernel: [batch + 1] tiles before each batch
  const float *qprep;
  float *partials;
  const float *k_centroids;
  const float *v_centroids;
  int *error;
  // decode step (decode_persist_kernel<..., true>): the kernel appends one token per
  // sequence at slot seq_lens[b], attends over seq_lens[b] + 1 tokens and prepares
  // the queries itself
  const void *q_raw;          // [batch][heads_q][128]
  const void *k_new, *v_new;  // [batch][heads_kv][128]
  int q_bf16, kv_bf16, q_rotate;
  const float *diag;         // D as +/-1.0f
  const float *sketch_tp;    // permuted S^T (sketch_signs_warp)
  int32_t *tile_prefix_out;  // [batch + 1] tiles before each batch, for the combine
  WarpRole role[2];          // keys, values
  // paged caches: virtual block -> pool block (NULL: contiguous). Last in the struct: placed
  // after `records`, the shifted parameter offsets cost the contiguous token loop 5 %.
  const int32_t *btab;
  int pool_blocks;
  // an upper bound of the tiles the call covers (sizes the persistent grid; 0: one CTA per SM)
  long long tiles_max;
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
// of q[coord] * cb[code]. Built as lo[v & low bits] + hi[v >> LOB] by NT
// threads: each owns one position and a slice of the high values.
// SIGN: cb = {-1, +1}.
template <int CB, int KPOS, int VBITS, bool SIGN, int NT>
__device__ __forceinline__ void build_lookup(float *T, const float *q, const float *cb_g, float scale, int tid) {
  constexpr int CPP = VBITS / CB;
  constexpr int LOB = (VBITS >= 8) ? 4 : 3;  // low-part bits (a whole number of codes)
  constexpr int HIB = VBITS - LOB;
  constexpr int NLO = 1 << LOB;
  constexpr int PARTS = (NT / KPOS < (1 << HIB)) ? NT / KPOS : (1 << HIB), NH = (1 << HIB) / PARTS;
  static_assert(NH * PARTS == (1 << HIB) && PARTS * KPOS <= NT, "table build split");
  constexpr int M = (1 << CB) - 1;
  if (tid >= PARTS * KPOS) return;
  const int pos = tid % KPOS, part = tid / KPOS;
  float qv[CPP];
#pragma unroll
  for (int j = 0; j < CPP; ++j) qv[j] = q[slot_coord(pos * CPP + j)] * scale;
  float cb[M + 1];
#pragma unroll
  for (int c = 0; c <= M; ++c) cb[c] = SIGN ? (c ? 1.f : -1.f) : cb_g[c];
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
      hi = fmaf(qv[LOB / CB + j], SIGN ? (c ? 1.f : -1.f) : cb_g[c], hi);
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

// Key tables (with log2(e)) for one query head; `kc` may point to shared memory.
template <int KB, bool KQJL, int NT>
__device__ __forceinline__ void build_key_tables(unsigned char *smem, int sm_ktab, int sm_stab, const float *s_q,
                                                 const float *kc, int tid) {
  float *s_ktab = reinterpret_cast<float *>(smem + sm_ktab);
  if constexpr (KB == 3) build_lookup<3, 64, 6, false, NT>(s_ktab, s_q, kc, kLog2e, tid);
  else build_lookup<KB, 16 * KB, 8, false, NT>(s_ktab, s_q, kc, kLog2e, tid);
  if constexpr (KQJL)
    build_lookup<1, 16, 8, true, NT>(reinterpret_cast<float *>(smem + sm_stab), s_q + kD, nullptr, kLog2e, tid);
}

// Value pair table (head-independent): field f -> half2(c[f & mask], c[f >> VB]),
// replicated for every lane, at offset 0 of shared memory.
template <int VB, int NT>
__device__ __forceinline__ void build_value_table(unsigned char *smem, int vlut_words, const float *v_centroids,
                                                  int tid) {
  uint32_t *vl = reinterpret_cast<uint32_t *>(smem);
  for (int e = tid; e < vlut_words; e += NT) {
    const int f = e >> 5;
    vl[e] = pack_half2(__ldg(v_centroids + (f & ((1 << VB) - 1))), __ldg(v_centroids + (f >> VB)));
  }
}

// Lane-invariant constants of the tile body.
template <int KB>
struct LaneConsts {
  uint32_t kcon[4], ksel[4];  // key lookups: byte offset into T from (record word, constant, selector)
  uint32_t ssel;              // key sign byte -> row offset (64-byte rows)
  int my_j;                   // token (0..15 of the warp) this lane holds after the score reduction
  int bsrc[4];                // lanes that hold the tokens of this lane's B fragment
  uint32_t bsel, swsel, lane4;
  bool bv_live, bs_live;

  __device__ __forceinline__ explicit LaneConsts(int lane) {
    const int half = lane >> 4, l = lane & 15, g = lane >> 2, t4 = lane & 3;
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
    ssel = (uint32_t)((8 * (l & 3) - 6) & 31);
    // reduce-scatter result: lane l (within its half) holds step sigma(l); token j = 2 sigma + half
    const int my_step = 4 * ((l >> 3) & 1) + 2 * ((l >> 2) & 1) + ((l >> 1) & 1);
    my_j = 2 * my_step + half;
    // token j of the warp sits on lanes 16(j&1) + 8((j>>3)&1) + 4((j>>2)&1) + 2((j>>1)&1) (+1);
    // the even lane carries p nu, the odd one p rho
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 2 * t4 + (c & 1) + 8 * (c >> 1);
      bsrc[c] = 16 * (j & 1) + 8 * ((j >> 3) & 1) + 4 * ((j >> 2) & 1) + 2 * ((j >> 1) & 1) + ((g >> 1) & 1);
    }
    bsel = (g & 1) ? 0x7632u : 0x5410u;  // hi parts (even g) or lo parts (odd g)
    bv_live = g < 2;
    bs_live = (g >> 1) == 1;
    lane4 = (uint32_t)lane << 2;
    swsel = (g & 1) ? 0x7632u : 0x5410u;  // sign rows: half (g & 1) of sign word (g >> 1)
  }
};

// Online-softmax state of one warp (base-2 logits).
struct WarpState {
  float m, l, w;
  float acc[8][4];
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    l = 0.f;
    w = 0.f;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mb][j] = 0.f;
  }
};

// One warp's 16 tokens (wbase .. wbase + 15 of the tile at `st`, tile start t0,
// sequence end t_end): scores, online-softmax step, value and sign MMAs.
template <typename Gm, int KB, int VB, bool KQJL, bool VQJL>
__device__ __forceinline__ void tile_body(const unsigned char *st, const unsigned char *smem, int wtile, int t0,
                                          int t_end, int lane, const LaneConsts<KB> &lc, WarpState &ws) {
  const int half = lane >> 4, l = lane & 15, g = lane >> 2, t4 = lane & 3;
  // the warp's 16 tokens (wtile .. wtile + 15 of the tile) are one block of the stage:
  // addresses are taken inside that block, validity against the tile position
  st += (wtile >> 4) * Gm::block;
  constexpr int wbase = 0;
  const float *kn = reinterpret_cast<const float *>(st + Gm::off_kn);
  const float *kr = reinterpret_cast<const float *>(st + Gm::off_kr);
  const unsigned char *tb = smem + Gm::sm_ktab;

  // ---- scores: 8 steps of 2 tokens, 16 lanes per token
  float part[8];
#pragma unroll
  for (int step = 0; step < 8; ++step) {
    const int lt = wbase + 2 * step + half;
    const uint32_t *rec = reinterpret_cast<const uint32_t *>(st + Gm::off_kc + lt * Gm::kc);
    float sum;
    if (KB == 4) {
      const uint32_t w = rec[l];
      float t[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        t[k] = *reinterpret_cast<const float *>(tb + __byte_perm(w, lc.kcon[k], lc.ksel[k]));
      sum = (t[0] + t[1]) + (t[2] + t[3]);
    } else if (KB == 3) {
      // lane l owns pair slots 4l..4l+3 (24 bits at bit 24 l)
      const int bit = 24 * l, wi = bit >> 5, off = bit & 31;
      const uint32_t f24 = __funnelshift_r(rec[wi], rec[(wi + 1 < 12) ? wi + 1 : wi], off);
      float t[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        t[k] = *reinterpret_cast<const float *>(tb + ((rotr(f24, lc.ksel[k]) & 0x3F00u) | lc.kcon[k]));
      sum = (t[0] + t[1]) + (t[2] + t[3]);
    } else if (KB == 2) {
      const uint32_t w = rec[l >> 1];
      float t[2];
#pragma unroll
      for (int k = 0; k < 2; ++k)
        t[k] = *reinterpret_cast<const float *>(tb + ((rotr(w, lc.ksel[k]) & 0x7F80u) | lc.kcon[k]));
      sum = t[0] + t[1];
    } else {
      const uint32_t w = rec[l >> 2];
      sum = *reinterpret_cast<const float *>(tb + ((rotr(w, lc.ksel[0]) & 0x3FC0u) | lc.kcon[0]));
    }
    if (KQJL) {
      const uint32_t *srec = reinterpret_cast<const uint32_t *>(st + Gm::off_ks + lt * 16);
      const uint32_t w = srec[l >> 2];
      const float ts =
          *reinterpret_cast<const float *>(smem + Gm::sm_stab + ((rotr(w, lc.ssel) & 0x3FC0u) | (4u * l)));
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
  const int tok = wbase + lc.my_j;
  const bool valid = t0 + wtile + tok < t_end;
  if (!KQJL) sc *= kn[tok];
  sc = valid ? sc : -INFINITY;

  // ---- online softmax over the warp's 16 tokens (base 2)
  float tmax = sc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
  const float m_new = fmaxf(ws.m, tmax);
  const float p = valid ? ex2_approx(sc - m_new) : 0.f;
  if (m_new != ws.m) {  // warp-uniform: the running max moved (m = -inf scales zeros)
    const float scale = ex2_approx(ws.m - m_new);
    ws.l *= scale;
    ws.w *= scale;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int j = 0; j < 4; ++j) ws.acc[mb][j] *= scale;
    ws.m = m_new;
  }
  ws.l += p;  // every token sits on two lanes: halved at the flush

  // ---- B operands: this lane's token weight (p nu on even lanes, p rho on odd ones)
  // as an fp16 hi/lo pair, gathered into column g of the MMA's B fragment
  uint32_t bv0, bv1, bs0 = 0, bs1 = 0;
  {
    const bool odd = VQJL && (lane & 1);
    const float *wsrc = reinterpret_cast<const float *>(st + (odd ? Gm::off_vr : Gm::off_vn));
    const float wv = valid ? p * wsrc[tok] : 0.f;
    ws.w += wv;  // sum of p rho over the odd lanes (the even ones are ignored)
    const __half hh = __float2half_rn(wv);
    const float rem = wv - __half2float(hh);
    const uint32_t hl =
        (uint32_t)__half_as_ushort(hh) | ((uint32_t)__half_as_ushort(__float2half_rn(rem)) << 16);
    const uint32_t x0 = __shfl_sync(kFull, hl, lc.bsrc[0]);
    const uint32_t x1 = __shfl_sync(kFull, hl, lc.bsrc[1]);
    const uint32_t x2 = __shfl_sync(kFull, hl, lc.bsrc[2]);
    const uint32_t x3 = __shfl_sync(kFull, hl, lc.bsrc[3]);
    const uint32_t b0 = __byte_perm(x0, x1, lc.bsel), b1 = __byte_perm(x2, x3, lc.bsel);
    bv0 = lc.bv_live ? b0 : 0u;
    bv1 = lc.bv_live ? b1 : 0u;
    if (VQJL) {
      bs0 = lc.bs_live ? b0 : 0u;
      bs1 = lc.bs_live ? b1 : 0u;
    }
  }

  // ---- values: pair-table lookups give the A fragments (coordinates x token pairs), MMA
  {
    // pair-interleaved value codes: rows t4 and t4 + 4 (tokens 2t4, 2t4 + 1 and
    // 2t4 + 8, 2t4 + 9), the 16 fields of coordinates g (mod 8) at words VB g ..
    uint32_t w0[VB], w1[VB];
    const uint32_t *vrow = reinterpret_cast<const uint32_t *>(st + Gm::off_vc);
#pragma unroll
    for (int k = 0; k < VB; ++k) {
      w0[k] = vrow[VB * (8 * t4 + g) + k];
      w1[k] = vrow[VB * (8 * (t4 + 4) + g) + k];
    }
    // field n of a span -> byte offset (field << 7) | (lane << 2) of the value table
    auto lut = [&](const uint32_t(&w)[VB], int n) -> uint32_t {
      constexpr int F = 2 * VB;
      constexpr uint32_t mask = ((1u << F) - 1u) << 7;
      const int bit = F * n, wi = bit >> 5, off = bit & 31;
      uint32_t x;
      if (off < 7) x = w[wi] << (7 - off);
      else x = __funnelshift_r(w[wi], w[(wi + 1 < VB) ? wi + 1 : wi], off - 7);
      return *reinterpret_cast<const uint32_t *>(smem + ((x & mask) | lc.lane4));
    };
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      // A fragment: rows coordinates 16 mb + g, 16 mb + 8 + g; columns the token pairs
      mma_16816(ws.acc[mb], lut(w0, 2 * mb), lut(w0, 2 * mb + 1), lut(w1, 2 * mb), lut(w1, 2 * mb + 1), bv0, bv1);
    }
  }

  // ---- QJL signs: rows of this thread = bits of half (g & 1) of sign word (g >> 1)
  if (VQJL) {
    const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + Gm::off_vs);
    const int wsel = g >> 1;
    const uint32_t wa0 = sw[(wbase + 2 * t4) * 4 + wsel], wb0 = sw[(wbase + 2 * t4 + 1) * 4 + wsel];
    const uint32_t wa1 = sw[(wbase + 2 * t4 + 8) * 4 + wsel], wb1 = sw[(wbase + 2 * t4 + 9) * 4 + wsel];
    // token 2t (8 + 2t) in bits 0..15, token 2t + 1 (9 + 2t) in bits 16..31
    const uint32_t s0 = __byte_perm(wa0, wb0, lc.swsel), s1 = __byte_perm(wa1, wb1, lc.swsel);
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
      mma_16816(ws.acc[mb], a0, a1, a2, a3, bs0, bs1);
    }
  }
}

// Park one warp's state as [m, l, w, pad, values[128], signs[128]] (signs
// un-scaled, 2 sum p rho b - sum p rho not yet formed).
template <bool VQJL>
__device__ __forceinline__ void park_warp(float *dst, int lane, const WarpState &ws) {
  const int g = lane >> 2, t4 = lane & 3;
  float lw = ws.l, ww = (lane & 1) ? ws.w : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lw += __shfl_xor_sync(kFull, lw, o);
    ww += __shfl_xor_sync(kFull, ww, o);
  }
  if (lane == 0) {
    dst[0] = ws.m;
    dst[1] = 0.5f * lw;
    dst[2] = ww;
  }
  float *va = dst + 4, *sa = dst + 4 + kD;
  if (t4 == 0) {  // columns 0/1: value sums of coordinates 16mb + g and 16mb + 8 + g
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      va[16 * mb + g] = ws.acc[mb][0] + ws.acc[mb][1];
      va[16 * mb + 8 + g] = ws.acc[mb][2] + ws.acc[mb][3];
    }
  } else if (VQJL && t4 == 1) {  // columns 2/3: sign sums; row (mb, r) is bit 2mb + r of half g&1 of word g>>1
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const int c0 = 64 * (g & 1) + 8 * mb + 2 * (g >> 1);
      sa[c0] = (ws.acc[mb][0] + ws.acc[mb][1]) * sign_unscale(sign_land(2 * mb));
      sa[c0 + 1] = (ws.acc[mb][2] + ws.acc[mb][3]) * sign_unscale(sign_land(2 * mb + 1));
    }
  }
}

// Merge NWG parked warp states (stride kPartialFloats) into one partial record;
// thread i of 128 handles coordinate i.
template <int NWG, bool VQJL>
__device__ __forceinline__ void merge_parked(const float *src, int i, float *rec) {
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NWG; ++w) M = fmaxf(M, src[w * kPartialFloats]);
  float L = 0.f, A = 0.f, Sg = 0.f;
#pragma unroll
  for (int w = 0; w < NWG; ++w) {
    const float *p = src + w * kPartialFloats;
    const float e = (p[0] == -INFINITY) ? 0.f : ex2_approx(p[0] - M);
    L += p[1] * e;
    A += p[4 + i] * e;
    // the sign MMA summed p rho b over bits b; sum p rho sigma = 2 sum p rho b - sum p rho
    if (VQJL) Sg += (2.f * p[4 + kD + i] - p[2]) * e;
  }
  if (i == 0) {
    rec[0] = M * kLn2;  // natural-log units for the combine step
    rec[1] = L;
  }
  rec[2 + i] = A;
  rec[2 + kD + i] = Sg;
}

// The stored block holding virtual slot vslot (a multiple of 16): contiguous caches keep
// block vslot / 16 in place, paged ones at the pool block the table names; nullptr for an
// unmapped entry (recorded as TQ_ERR_ARG; the stage then keeps stale data and the output of
// that head is meaningless, which the error word reports).
template <int BLOCK>
__device__ __forceinline__ const uint8_t *block_src(const Decode2Args &a, long long vslot) {
  const long long p = phys_slot(a.btab, a.pool_blocks, vslot, a.error);
  return p < 0 ? nullptr : a.records + (p >> 4) * BLOCK;
}

// The stored block a prefetched table entry `pb` names (paged caches), or nullptr when it is
// outside the pool (recorded as TQ_ERR_ARG, as block_src does).
template <int BLOCK>
__device__ __forceinline__ const uint8_t *pool_block(const Decode2Args &a, int pb) {
  if (pb < 0 || pb >= a.pool_blocks) {
    set_error(a.error, TQ_ERR_ARG);
    return nullptr;
  }
  return a.records + (long long)pb * BLOCK;
}

// Copy the blocks holding tokens s0 .. s0 + n - 1 (s0 a multiple of 16) into a stage: one
// copy for contiguous blocks, one per block for a paged cache.
template <typename Gm>
__device__ __forceinline__ void issue_tile_to(unsigned char *st, uint64_t *bar, const Decode2Args &a, long long s0, int n) {
  const int nb = (n + 15) >> 4;
  if (a.btab == nullptr) {
    const uint32_t bytes = (uint32_t)(nb * Gm::block);
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_1d(st, a.records + (s0 >> 4) * Gm::block, bytes, bar);
    return;
  }
  const uint8_t *src[4];
  uint32_t bytes = 0;
  for (int j = 0; j < nb; ++j) {
    src[j] = block_src<Gm::block>(a, s0 + 16 * j);
    if (src[j]) bytes += Gm::block;
  }
  mbar_arrive_expect_tx(bar, bytes);
  for (int j = 0; j < nb; ++j)
    if (src[j]) tma_load_1d(st + j * Gm::block, src[j], (uint32_t)Gm::block, bar);
}

// ============================================================================
// split-K kernel: one CTA of 4 warps per (batch, kv head, chunk)
// ============================================================================
template <int KB, int VB, bool KQJL, bool VQJL>
__global__ void __launch_bounds__(128, 2) decode2_g1_kernel(Decode2Args a) {
  using Gm = Geo<KB, VB, KQJL, VQJL, 4, 3>;
  constexpr int S = Gm::kStages;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_stage = smem + Gm::sm_stage;
  uint64_t *s_full = reinterpret_cast<uint64_t *>(smem + Gm::sm_bar);
  unsigned *s_cnt = reinterpret_cast<unsigned *>(smem + Gm::sm_cnt);
  float *s_q = reinterpret_cast<float *>(smem + Gm::sm_q);

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();  // the prepared queries come from the kernel before
  const int len = min(max(__ldg(a.seq_lens + b), 0), a.capacity);
  const int t_begin = split * a.chunk;
  const int t_end = min(t_begin + a.chunk, len);
  const int ntiles = (t_end > t_begin) ? (t_end - t_begin + kTT - 1) / kTT : 0;
  const long long slot0 = ((long long)b * a.heads_kv + hk) * a.cap16;
  const int hq = hk;  // one query head per KV head

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&s_full[s], 1);
      s_cnt[s] = 0;
    }
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int tile) {
    const int t0 = t_begin + tile * kTT;
    issue_tile_to<Gm>(s_stage + (tile % S) * Gm::stage, &s_full[tile % S], a, slot0 + t0,
                                  min(kTT, t_end - t0));
  };
  if (tid == 0)
    for (int i = 0; i < S && i < ntiles; ++i) issue(i);

  // prepared query (already rotated and scaled by 1/sqrt(d); S q scaled by sqrt(pi/2)/m/sqrt(d))
  const float *qp = a.qprep + ((size_t)b * a.heads_q + hq) * 2 * kD;
  s_q[tid] = __ldg(qp + tid);
  if (KQJL) s_q[kD + tid] = __ldg(qp + kD + tid);
  __syncthreads();
  build_key_tables<KB, KQJL, 128>(smem, Gm::sm_ktab, Gm::sm_stab, s_q, a.k_centroids, tid);
  build_value_table<VB, 128>(smem, Gm::vlut, a.v_centroids, tid);
  __syncthreads();

  const LaneConsts<KB> lc(lane);
  WarpState ws;
  ws.reset();
  // A wait that runs out of time (it never should) records TQ_ERR_TIMEOUT; the
  // warp then stops waiting and computing but keeps releasing its stages, so
  // no warp is left behind. The partial record is then meaningless, which the
  // error word reports.
  bool bad = false;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile % S;
    if (!bad && !mbar_wait_bounded(&s_full[stage], (tile / S) & 1, a.error)) bad = true;
    bad = __any_sync(kFull, bad);  // whole warps skip together (the body shuffles)
    if (!bad)
      tile_body<Gm, KB, VB, KQJL, VQJL>(s_stage + stage * Gm::stage, smem, warp * 16, t_begin + tile * kTT, t_end,
                                        lane, lc, ws);
    // release the stage: the last of the four warps refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const unsigned old = atomicAdd(&s_cnt[stage], 1u);
      if ((old & 3u) == 3u && tile + S < ntiles) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(tile + S);
      }
    }
  }

  // merge the warps (parked in the key-table area) into this chunk's partial record
  __syncthreads();
  float *park = reinterpret_cast<float *>(smem + Gm::sm_ktab);
  park_warp<VQJL>(park + warp * kPartialFloats, lane, ws);
  __syncthreads();
  merge_parked<4, VQJL>(park, tid,
                        a.partials + (((size_t)b * a.heads_q + hq) * a.splits + split) * kPartialFloats);
}

// ============================================================================
// persistent kernel: one CTA of 16 warps per SM; warp group grp (4 warps)
// takes the CTA's tiles of local index = grp (mod 4), which live in the ring
// stages s = grp (mod 4). Each warp streams only its own 16-token quarter of
// a tile, on its own mbarrier, and refills that quarter as soon as it is done
// with it -- no warp ever waits for another inside a head.
// ============================================================================
constexpr int kPersistWarps = 16;  // four groups of four (kPersistGroups)

// Decode step: the lengths before the step (s_raw) and after the append (seq_lens + 1,
// clamped to [0, capacity]), the
// exclusive prefix over batches of their 64-token tile counts (batch <= 256: eight warp
// scans), and, by CTA 0, that prefix for the combine and the append's capacity errors.
__device__ __forceinline__ void step_lengths(const Decode2Args &a, int *s_pre, int *s_len, int *s_raw, int *s_scan,
                                             int tid) {
  const int B = a.batch, lane = tid & 31, warp = tid >> 5;
  int n = 0;
  if (tid < B) {
    const int len = __ldg(a.seq_lens + tid);
    const int dl = (len < 0) ? 0 : min(len, a.capacity - 1) + 1;
    s_len[tid] = dl;
    s_raw[tid] = len;
    n = (dl + kTT - 1) / kTT;
    if (blockIdx.x == 0 && (len < 0 || len >= a.capacity)) set_error(a.error, TQ_ERR_CAPACITY);
  }
  int v = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31 && warp < kMaxPersistBatch / 32) s_scan[warp] = v;
  __syncthreads();
  if (tid < B) {
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_scan[w];
    s_pre[tid + 1] = base + v;
  }
  if (tid == 0) s_pre[0] = 0;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = tid; i <= B; i += blockDim.x) a.tile_prefix_out[i] = s_pre[i];
}

// Raw query of row `row` (lane L: coordinates 4L..4L+3), copied asynchronously into 512
// bytes of shared memory by one warp and read back after cp_async_wait_all(), and its
// preparation as the query prep kernel does it: q_rot = H D q / sqrt(d) (orthonormal H),
// or q / sqrt(d) for unrotated keys.
__device__ __forceinline__ void stage_query(const Decode2Args &a, int row, int lane, float *raw) {
  if (a.q_bf16)
    cp_async_8(reinterpret_cast<uint16_t *>(raw) + 4 * lane,
               static_cast<const uint16_t *>(a.q_raw) + (size_t)row * kD + 4 * lane);
  else
    cp_async_16(raw + 4 * lane, static_cast<const float *>(a.q_raw) + (size_t)row * kD + 4 * lane);
  cp_async_commit();
}
__device__ __forceinline__ void staged_query(const Decode2Args &a, const float *raw, int lane, float (&v)[4]) {
  if (a.q_bf16) {
    const uint2 w = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(raw) + 4 * lane);
    v[0] = bf16_bits_to_float(w.x & 0xffffu);
    v[1] = bf16_bits_to_float(w.x >> 16);
    v[2] = bf16_bits_to_float(w.y & 0xffffu);
    v[3] = bf16_bits_to_float(w.y >> 16);
  } else {
    const float4 f = reinterpret_cast<const float4 *>(raw)[lane];
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
}
__device__ __forceinline__ void prep_query(const Decode2Args &a, int lane, float (&v)[4]) {
  if (a.q_rotate) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= __ldg(a.diag + 4 * lane + j);
    wht128(v, lane);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] *= kInvSqrtD;
}

// Append the new token (one role) of unit u = b * H + h at slot len (the sequence's
// length before the step, 0 <= len < capacity) by one warp. s_sk: the permuted S^T in
// shared memory. A paged cache's slot goes through the block table.
__device__ __forceinline__ void step_append(const Decode2Args &a, int u, int role, int len, int lane,
                                            const float *s_sk) {
  const long long slot = phys_slot(a.btab, a.pool_blocks, (long long)u * a.cap16 + len, a.error);
  if (slot < 0) return;  // an unmapped block: nothing appended (the error word says so)
  float x[4];
  load4(role ? a.v_new : a.k_new, (size_t)u * kD + 4 * lane, a.kv_bf16 != 0, x);
  const WarpRole &ro = a.role[role];
  float nu, rr, r[4];
  encode_vector_warp(ro, x, slot, a.bb, a.diag, lane, nu, r, rr);
  if (!ro.qjl) return;
  uint32_t w[4];
  sketch_signs_warp(s_sk, r, lane, w);
  float rho = nu * sqrtf(rr);
  if (nu == 0.f) {  // a zero vector: every sign set, rho = 0
    w[0] = w[1] = w[2] = w[3] = 0xffffffffu;
    rho = 0.f;
  }
  const uint32_t mine = lane == 0 ? w[0] : (lane == 1 ? w[1] : (lane == 2 ? w[2] : w[3]));
  if (lane < 4) reinterpret_cast<uint32_t *>(rec_at(ro.signs, slot, a.bb, kD / 8))[lane] = mine;
  if (lane == 0) {
    *rec_at(ro.norms, slot, a.bb, 4) = nu;
    *rec_at(ro.rnorms, slot, a.bb, 4) = rho;
  }
}

// shared-memory bytes of the persistent kernel: the layout of Geo, the batch prefix and
// lengths, the key centroids, one mbarrier (8-byte aligned) for the decode step's copy of
// the permuted S^T, and the decode step's lengths before the step
template <typename Gm>
constexpr int persist_sbar_offset() {
  return (Gm::sm_misc + 4 * (2 * kMaxPersistBatch + 1) + 4 * kMaxLevels + 7) & ~7;
}
template <typename Gm>
constexpr int persist_smem_bytes() {
  return persist_sbar_offset<Gm>() + 8 + 4 * kMaxPersistBatch;  // + the decode step's raw lengths
}

// One instantiation serves contiguous and paged caches: the layout only changes where each
// batch of copy sources is computed (measured: a separate contiguous instantiation ran its
// tile loop 3.7 % slower).
template <int KB, int VB, bool KQJL, bool VQJL, bool FUSED>
__global__ void __launch_bounds__(kPersistWarps * 32, 1) decode_persist_kernel(Decode2Args a) {
  static_assert(!(FUSED && KQJL), "the decode step prepares queries without a key sketch");
  constexpr int S = persist_stages<KB, VB, KQJL, VQJL>();
  static_assert(S >= 8 && S % kPersistGroups == 0, "ring stages");
  using Gm = Geo<KB, VB, KQJL, VQJL, kPersistWarps, S>;
  // the decode step's sketched values read S^T from the key-table area and, past it, the
  // first ring stages (contiguous when keys have no sketch table), until the ring starts
  constexpr bool kStepSketch = FUSED && VQJL;
  static_assert(!kStepSketch || Gm::sm_ktab + kD * kD * 4 <= Gm::sm_stage + S * Gm::stage, "S^T copy area");
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_stage = smem + Gm::sm_stage;
  uint64_t *s_full = reinterpret_cast<uint64_t *>(smem + Gm::sm_bar);  // [S][4 quarters]
  float *s_q = reinterpret_cast<float *>(smem + Gm::sm_q);
  int *s_pre = reinterpret_cast<int *>(smem + Gm::sm_misc);  // [batch + 1] tile prefix
  int *s_len = s_pre + kMaxPersistBatch + 1;                  // [batch] clamped lengths
  float *s_kc = reinterpret_cast<float *>(s_len + kMaxPersistBatch);  // [16] key centroids
  uint64_t *s_sbar = reinterpret_cast<uint64_t *>(smem + persist_sbar_offset<Gm>());
  int *s_raw = reinterpret_cast<int *>(smem + persist_sbar_offset<Gm>() + 8);  // [batch]
  const float *s_sk = reinterpret_cast<const float *>(smem + Gm::sm_ktab);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, grp = warp >> 2, qtr = warp & 3;
  const int B = a.batch, H = a.heads_kv;
  if constexpr (kStepSketch) {
    // S^T is a context constant: its copy overlaps the wait for the kernel before
    if (tid == 0) {
      mbar_init(s_sbar, 1);
      mbar_fence_init();
      mbar_arrive_expect_tx(s_sbar, kD * kD * sizeof(float));
      tma_load_1d(smem + Gm::sm_ktab, a.sketch_tp, kD * kD * sizeof(float), s_sbar);
    }
  }
  if (tid < kMaxLevels) s_kc[tid] = __ldg(a.k_centroids + tid);
  build_value_table<VB, kPersistWarps * 32>(smem, Gm::vlut, a.v_centroids, tid);
  // everything above reads context constants only; the query prep (tile prefix,
  // prepared queries) and the cache come from earlier kernels of the stream
  pdl_trigger();
  pdl_wait();
  if constexpr (FUSED) {
    // s_q is free until the first head's query is prepared
    step_lengths(a, s_pre, s_len, s_raw, reinterpret_cast<int *>(s_q), tid);
  } else {
    for (int i = tid; i <= B; i += blockDim.x) s_pre[i] = __ldg(a.tile_prefix + i);
    for (int i = tid; i < B; i += blockDim.x) s_len[i] = min(max(__ldg(a.seq_lens + i), 0), a.capacity);
  }
  if (tid < S * 4) mbar_init(&s_full[tid], 1);
  mbar_fence_init();
  __syncthreads();
  // slice of CTA c: [b(c), b(c + 1)) with b(c) = min(T, 4 floor(ceil(T / 4) c / C)), so
  // slices (and, when heads hold multiples of 4 tiles, head segments) split evenly
  // over the four warp groups
  const long long T = (long long)H * s_pre[B];
  const long long C = gridDim.x, c = blockIdx.x, T4 = (T + 3) / 4;
  const int g0 = (int)min(T, 4 * (T4 * c / C)), g1 = (int)min(T, 4 * (T4 * (c + 1) / C));
  if (g0 >= g1) {  // whole CTA: nothing to do (no record is read for it)
    if constexpr (kStepSketch) mbar_wait_bounded(s_sbar, 0, a.error);  // no copy outlives the CTA
    return;
  }
  const int nloc = g1 - g0;

  // batch of global tile g: the largest b with H * pre[b] <= g
  auto batch_of = [&](int g) -> int {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * s_pre[mid] <= g) lo = mid;
      else hi = mid;
    }
    return lo;
  };

  // the copies of this warp, in batches of 32 (lane j: the copy of local tile cur_i + 4 j as of
  // the batch's start): each lane works out its tile's head, token range and source block once
  // (for a paged cache through the block table), and each copy takes its source by a shuffle
  int cur_i = grp;
  const uint8_t *src_lane = nullptr;
  int src_next = 32;
  auto refill_sources = [&]() {
    const int li = cur_i + kPersistGroups * lane;
    const uint8_t *p = nullptr;
    if (li < nloc) {
      const int g = g0 + li;
      const int bq = batch_of(g);
      const int nb = s_pre[bq + 1] - s_pre[bq];
      const int r = g - H * s_pre[bq];
      const int hq = r / nb, tq_ = r - hq * nb;
      const int t0 = tq_ * kTT + 16 * qtr;
      if (t0 < s_len[bq]) {  // this quarter holds tokens: its stored block
        const long long vslot = ((long long)bq * H + hq) * a.cap16 + t0;
        if (a.btab) p = pool_block<Gm::block>(a, __ldg(a.btab + (vslot >> 4)));
        else p = a.records + (vslot >> 4) * Gm::block;
      }
    }
    src_lane = p;
    src_next = 0;
  };
  // issue this warp's quarter of local tile cur_i (whole warp), then step to the group's next tile
  auto issue_next = [&]() {
    const int st = cur_i % S;
    uint64_t *bar = &s_full[st * 4 + qtr];
    if (src_next == 32) refill_sources();
    const uint8_t *src = reinterpret_cast<const uint8_t *>(
        __shfl_sync(kFull, reinterpret_cast<unsigned long long>(src_lane), src_next++));
    if (lane == 0) {  // the quarter is one stored block: one bulk copy
      mbar_arrive_expect_tx(bar, src ? (uint32_t)Gm::block : 0u);
      if (src) tma_load_1d(s_stage + st * Gm::stage + qtr * Gm::block, src, (uint32_t)Gm::block, bar);
    }
    cur_i += kPersistGroups;
  };
  // query row (= unit: one query head per KV head) of the segment starting at tile g
  auto unit_of = [&](int g) -> int {
    const int bb = batch_of(g);
    const int nb = s_pre[bb + 1] - s_pre[bb];
    return bb * H + (g - H * s_pre[bb]) / nb;
  };
  // decode step: the CTA holding a head's last tile appends that head's new token (keys
  // and values, one warp each) before any tile is copied (appends issued while the ring's
  // copies stream would queue their loads and stores behind them); meanwhile the first
  // head's query is copied into the upper half of s_q
  if constexpr (FUSED) {
    if (warp == kPersistWarps - 1) stage_query(a, unit_of(g0), lane, s_q + kD);
    if constexpr (kStepSketch) mbar_wait_bounded(s_sbar, 0, a.error);
    const int ua = unit_of(g0), ub = unit_of(g1 - 1);
    for (int j = warp; j < 2 * (ub - ua + 1); j += kPersistWarps) {
      const int u = ua + (j >> 1);
      const int bq = u / H, hq = u - bq * H;
      const int nb = s_pre[bq + 1] - s_pre[bq];
      const int gl = H * s_pre[bq] + (hq + 1) * nb - 1;  // the head's last tile
      const int len = s_raw[bq];
      if (nb == 0 || gl < g0 || gl >= g1 || len < 0 || len >= a.capacity) continue;
      step_append(a, u, j & 1, len, lane, s_sk);
      fence_proxy_async_global();  // the records written above, before their bulk copies
    }
    if constexpr (kStepSketch) fence_proxy_async_shared();  // S^T read above, before the ring overwrites it
    __syncthreads();
  }
  for (int k = 0; k < S / kPersistGroups && cur_i < nloc; ++k) issue_next();

  const LaneConsts<KB> lc(lane);
  WarpState ws;
  bool bad = false;
  float *park = reinterpret_cast<float *>(smem + Gm::sm_ktab);
  if constexpr (FUSED) {
    if (warp == kPersistWarps - 1) {
      cp_async_wait_all();
      __syncwarp();
      float v[4];
      staged_query(a, s_q + kD, lane, v);
      prep_query(a, lane, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) s_q[4 * lane + j] = v[j];
    }
  } else {
    if (tid < 2 * kD) s_q[tid] = __ldg(a.qprep + (size_t)unit_of(g0) * 2 * kD + tid);
  }
  __syncthreads();
  int g = g0;
  while (g < g1) {  // one segment per (batch, kv head) the slice touches
    const int bb = batch_of(g);
    const int nb = s_pre[bb + 1] - s_pre[bb];
    const int ubase = H * s_pre[bb];
    const int h = (g - ubase) / nb;
    const int us = ubase + h * nb;
    const int se = min(us + nb, g1);
    const int len = s_len[bb];
    const int u = bb * H + h;

    // key tables for this head (s_q holds its query; the previous segment's
    // readers of the table area passed the barrier that closed its flush)
    build_key_tables<KB, KQJL, kPersistWarps * 32>(smem, Gm::sm_ktab, Gm::sm_stab, s_q, s_kc, tid);
    __syncthreads();
    // the next segment's query, fetched while this one streams (decode step: its raw
    // values copied into the upper half of s_q, which keys without a sketch leave unused,
    // by the last warp, which takes no part in the merge below)
    float q_next = 0.f;
    if constexpr (FUSED) {
      if (se < g1 && warp == kPersistWarps - 1) stage_query(a, unit_of(se), lane, s_q + kD);
    } else {
      if (se < g1 && tid < 2 * kD) q_next = __ldg(a.qprep + (size_t)unit_of(se) * 2 * kD + tid);
    }

    ws.reset();
    // this group's tiles: local index i = t - g0 with i % 4 == grp
    for (int t = g + ((grp - ((g - g0) & 3)) & 3); t < se; t += kPersistGroups) {
      const int i = t - g0;
      const int stage = i % S;
      if (!bad && !mbar_wait_bounded(&s_full[stage * 4 + qtr], (uint32_t)((i / S) & 1), a.error)) bad = true;
      bad = __any_sync(kFull, bad);
      if (!bad)
        tile_body<Gm, KB, VB, KQJL, VQJL>(s_stage + stage * Gm::stage, smem, qtr * 16, (t - us) * kTT, len, lane,
                                          lc, ws);
      // this warp is done with its quarter of the stage: refill it
      __syncwarp();
      if (cur_i < nloc) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_next();
      }
    }

    // flush: every group is done with this head; park the warps in the table area
    __syncthreads();
    park_warp<VQJL>(park + warp * kPartialFloats, lane, ws);
    __syncthreads();
    if constexpr (FUSED) {
      if (warp == kPersistWarps - 1 && se < g1) {
        cp_async_wait_all();
        __syncwarp();
        float qn4[4];
        staged_query(a, s_q + kD, lane, qn4);
        prep_query(a, lane, qn4);
#pragma unroll
        for (int j = 0; j < 4; ++j) s_q[4 * lane + j] = qn4[j];
      }
    } else {
      if (tid < 2 * kD) s_q[tid] = q_next;
    }
    // one record per (CTA, head): all 16 warps merged
    if (tid < kD) merge_parked<kPersistWarps, VQJL>(park, tid, a.partials + (size_t)(c + u) * kPartialFloats);
    __syncthreads();  // the table area is rebuilt next
    g = se;
  }
}

// ============================================================================
// GQA: G query heads per KV head (G = 2 or 4), persistent like the kernel
// above. Keys become the MMA's A operand: a lane-replicated table maps each
// pair field of a key record to (hi, lo) fp16 pairs of the two centroids, and
// the pair-slot layout makes the MMA's K index natural coordinate order, so B
// holds the G rotated queries' fp16 hi / lo parts as columns 2h, 2h + 1. Two
// MMAs per 16 coordinates (A hi, A lo) score 16 tokens for all G heads with
// all four hi / lo products. A lane (g, t) then owns head t: the scores of
// tokens g and g + 8, that head's softmax state and accumulator columns.
// ============================================================================
template <int KB, int VB, bool VQJL, int G>
struct GeoQ {
  using Gs = Geo<KB, VB, false, VQJL, kPersistWarps, 1>;  // stage layout
  static constexpr int kval = 1 << (2 * KB);
  static constexpr int vlut = Gs::vlut;                  // words
  static constexpr int sm_klut = vlut * 4;               // [kval][32 lanes] x (hi, lo) half2 pairs
  static constexpr int sm_park = sm_klut + kval * 256;   // [4 warps][G][kPartialFloats]
  static constexpr int sm_stage0 = sm_park + 4 * G * kPartialFloats * 4;
  static constexpr int fixed = sm_stage0 + 16 * 4 * 8 + G * kD * 4 + 4 * (2 * kMaxPersistBatch + 1) + 64;
  static constexpr int S = ((227 * 1024 - fixed) / Gs::stage >= 16) ? 16 : (((227 * 1024 - fixed) / Gs::stage) / 4) * 4;
  static constexpr int stage = Gs::stage;
  static constexpr int off_kc = Gs::off_kc, off_kn = Gs::off_kn, off_vc = Gs::off_vc, off_vn = Gs::off_vn;
  static constexpr int off_vs = Gs::off_vs, off_vr = Gs::off_vr, kc = Gs::kc, vc = Gs::vc;
  static constexpr int block = Gs::block;
  static constexpr int sm_bar = sm_stage0 + S * stage;
  static constexpr int sm_q = sm_bar + S * 4 * 8;                  // [G][128]
  static constexpr int sm_misc = sm_q + G * kD * 4;
  static constexpr int total = sm_misc + 4 * (2 * kMaxPersistBatch + 1);
};

// one warp's 16 tokens for all G heads of its KV head
template <typename Q, int KB, int VB, bool VQJL, int G>
__device__ __forceinline__ void tile_body_gqa(const unsigned char *st, const unsigned char *smem, int wtile, int t0,
                                              int t_end, int lane, const uint32_t (&bk)[8][2], float &m_run,
                                              float &l_run, float &w_run, float (&acc)[8][4]) {
  const int g = lane >> 2, t4 = lane & 3, h = g >> 1;
  st += (wtile >> 4) * Q::block;  // the warp's block of the stage (see tile_body)
  constexpr int wbase = 0;
  const uint32_t lane8 = (uint32_t)lane << 3, lane4 = (uint32_t)lane << 2;
  const float *kn = reinterpret_cast<const float *>(st + Q::off_kn);
  // ---- scores of tokens g and g + 8 for head t4: S = K_hat (A) x [q_hi, q_lo] (B)
  float sk[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint32_t w0[KB], w1[KB];
    const uint32_t *r0 = reinterpret_cast<const uint32_t *>(st + Q::off_kc + (wbase + g) * Q::kc);
    const uint32_t *r1 = reinterpret_cast<const uint32_t *>(st + Q::off_kc + (wbase + 8 + g) * Q::kc);
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      w0[k] = r0[KB * t4 + k];
      w1[k] = r1[KB * t4 + k];
    }
    // field n of a span -> (hi, lo) pair of the key table at (field << 8) | (lane << 3)
    auto klut = [&](const uint32_t(&w)[KB], int n) -> uint2 {
      constexpr int F = 2 * KB;
      constexpr uint32_t mask = ((1u << F) - 1u) << 8;
      const int bit = F * n, wi = bit >> 5, off = bit & 31;
      uint32_t x;
      if (off < 8) x = w[wi] << (8 - off);
      else x = __funnelshift_r(w[wi], w[(wi + 1 < KB) ? wi + 1 : wi], off - 8);
      return *reinterpret_cast<const uint2 *>(smem + Q::sm_klut + ((x & mask) | lane8));
    };
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const uint2 a0 = klut(w0, 2 * kb), a1 = klut(w1, 2 * kb), a2 = klut(w0, 2 * kb + 1), a3 = klut(w1, 2 * kb + 1);
      mma_16816(sk, a0.x, a1.x, a2.x, a3.x, bk[kb][0], bk[kb][1]);
      mma_16816(sk, a0.y, a1.y, a2.y, a3.y, bk[kb][0], bk[kb][1]);
    }
  }
  const int tok0 = wbase + g, tok1 = wbase + 8 + g;
  const bool v0 = t0 + wtile + tok0 < t_end, v1 = t0 + wtile + tok1 < t_end;
  float s0 = v0 ? (sk[0] + sk[1]) * kn[tok0] : -INFINITY;
  float s1 = v1 ? (sk[2] + sk[3]) * kn[tok1] : -INFINITY;
  // ---- online softmax of head t4 over the warp's 16 tokens (the 8 lanes g share t4)
  float tmax = fmaxf(s0, s1);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
  const float m_new = fmaxf(m_run, tmax);
  const float p0 = v0 ? ex2_approx(s0 - m_new) : 0.f, p1 = v1 ? ex2_approx(s1 - m_new) : 0.f;
  if (m_new != m_run) {  // per head (lane-divergent; no shuffles inside)
    const float scale = ex2_approx(m_run - m_new);
    l_run *= scale;
    w_run *= scale;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mb][j] *= scale;
    m_run = m_new;
  }
  l_run += p0 + p1;
  // ---- B operands, column g of lane (g, t), tokens 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1); token j
  // of head h sits on lane 4 (j % 8) + h. Without signs: column 2h + part = the hi / lo part of
  // head h's weights p nu, one MMA per 16 coordinates. With signs: column 2h = head h's values,
  // 2h + 1 its signs, each filled by two MMAs (hi, then lo parts of p nu or p rho) into one
  // accumulator -- twice the MMAs of two hi / lo accumulators, half their registers.
  auto hl2 = [](float a, float b, uint32_t &hi, uint32_t &lo) {
    const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
    hi = (uint32_t)__half_as_ushort(ha) | ((uint32_t)__half_as_ushort(hb) << 16);
    lo = (uint32_t)__half_as_ushort(__float2half_rn(a - __half2float(ha))) |
         ((uint32_t)__half_as_ushort(__float2half_rn(b - __half2float(hb))) << 16);
  };
  const int src0 = 4 * (2 * t4) + h, src1 = 4 * (2 * t4 + 1) + h;
  const bool live = g < 2 * G, odd = (g & 1) != 0;
  // the hi and lo fragments of one weight kind; `mine`: this lane's column takes that kind
  auto gather = [&](uint32_t xh, uint32_t xl, bool mine, uint32_t (&bh)[2], uint32_t (&bl)[2]) {
    const uint32_t a_h = __shfl_sync(kFull, xh, src0), a_l = __shfl_sync(kFull, xl, src0);
    const uint32_t c_h = __shfl_sync(kFull, xh, src1), c_l = __shfl_sync(kFull, xl, src1);
    bh[0] = mine ? __byte_perm(a_h, c_h, 0x5410u) : 0u;  // tokens 2t, 2t+1
    bh[1] = mine ? __byte_perm(a_h, c_h, 0x7632u) : 0u;  // tokens 2t+8, 2t+9
    bl[0] = mine ? __byte_perm(a_l, c_l, 0x5410u) : 0u;
    bl[1] = mine ? __byte_perm(a_l, c_l, 0x7632u) : 0u;
  };
  uint32_t bvh[2], bvl[2], bsh[2] = {0u, 0u}, bsl[2] = {0u, 0u};
  uint32_t bv0, bv1;
  {
    const float *vn = reinterpret_cast<const float *>(st + Q::off_vn);
    uint32_t xh, xl;
    hl2(v0 ? p0 * vn[tok0] : 0.f, v1 ? p1 * vn[tok1] : 0.f, xh, xl);
    gather(xh, xl, live && (VQJL ? !odd : true), bvh, bvl);
    bv0 = odd ? bvl[0] : bvh[0];  // without signs: hi / lo by column parity
    bv1 = odd ? bvl[1] : bvh[1];
    if (VQJL) {
      const float *vr = reinterpret_cast<const float *>(st + Q::off_vr);
      const float r0 = v0 ? p0 * vr[tok0] : 0.f, r1 = v1 ? p1 * vr[tok1] : 0.f;
      w_run += r0 + r1;
      hl2(r0, r1, xh, xl);
      gather(xh, xl, live && odd, bsh, bsl);
    }
  }
  // ---- values: as in the one-head body (pair-table A fragments), G heads in the columns
  {
    // pair-interleaved value codes: rows t4 and t4 + 4 (tokens 2t4, 2t4 + 1 and
    // 2t4 + 8, 2t4 + 9), the 16 fields of coordinates g (mod 8) at words VB g ..
    uint32_t w0[VB], w1[VB];
    const uint32_t *vrow = reinterpret_cast<const uint32_t *>(st + Q::off_vc);
#pragma unroll
    for (int k = 0; k < VB; ++k) {
      w0[k] = vrow[VB * (8 * t4 + g) + k];
      w1[k] = vrow[VB * (8 * (t4 + 4) + g) + k];
    }
    auto lut = [&](const uint32_t(&w)[VB], int n) -> uint32_t {
      constexpr int F = 2 * VB;
      constexpr uint32_t mask = ((1u << F) - 1u) << 7;
      const int bit = F * n, wi = bit >> 5, off = bit & 31;
      uint32_t x;
      if (off < 7) x = w[wi] << (7 - off);
      else x = __funnelshift_r(w[wi], w[(wi + 1 < VB) ? wi + 1 : wi], off - 7);
      return *reinterpret_cast<const uint32_t *>(smem + ((x & mask) | lane4));
    };
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      // A fragment: rows coordinates 16 mb + g, 16 mb + 8 + g; columns the token pairs
      const uint32_t a0 = lut(w0, 2 * mb), a1 = lut(w0, 2 * mb + 1), a2 = lut(w1, 2 * mb), a3 = lut(w1, 2 * mb + 1);
      if (VQJL) {
        mma_16816(acc[mb], a0, a1, a2, a3, bvh[0], bvh[1]);
        mma_16816(acc[mb], a0, a1, a2, a3, bvl[0], bvl[1]);
      } else {
        mma_16816(acc[mb], a0, a1, a2, a3, bv0, bv1);
      }
    }
  }
  // ---- QJL signs (same operands as the one-head body), separate accumulator
  if (VQJL) {
    const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + Q::off_vs);
    const int wsel = g >> 1;
    const uint32_t swsel = (g & 1) ? 0x7632u : 0x5410u;
    const uint32_t wa0 = sw[(wbase + 2 * t4) * 4 + wsel], wb0 = sw[(wbase + 2 * t4 + 1) * 4 + wsel];
    const uint32_t wa1 = sw[(wbase + 2 * t4 + 8) * 4 + wsel], wb1 = sw[(wbase + 2 * t4 + 9) * 4 + wsel];
    const uint32_t sa = __byte_perm(wa0, wb0, swsel), sb = __byte_perm(wa1, wb1, swsel);
    const uint32_t sar10 = rotr(sa, 22), sar5 = rotr(sa, 27), sar27 = rotr(sa, 5);
    const uint32_t sbr10 = rotr(sb, 22), sbr5 = rotr(sb, 27), sbr27 = rotr(sb, 5);
    auto pick = [&](int k, uint32_t r0, uint32_t r5, uint32_t r10, uint32_t r27) -> uint32_t {
      const uint32_t src = sign_rot(k) == 10 ? r10 : (sign_rot(k) == 5 ? r5 : (sign_rot(k) == 0 ? r0 : r27));
      return src & (0x00010001u << sign_land(k));
    };
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const uint32_t a0 = pick(2 * mb, sa, sar5, sar10, sar27);
      const uint32_t a1 = pick(2 * mb + 1, sa, sar5, sar10, sar27);
      const uint32_t a2 = pick(2 * mb, sb, sbr5, sbr10, sbr27);
      const uint32_t a3 = pick(2 * mb + 1, sb, sbr5, sbr10, sbr27);
      mma_16816(acc[mb], a0, a1, a2, a3, bsh[0], bsh[1]);
      mma_16816(acc[mb], a0, a1, a2, a3, bsl[0], bsl[1]);
    }
  }
}

template <int KB, int VB, bool VQJL, int G>
__global__ void __launch_bounds__(kPersistWarps * 32, 1) decode_persist_gqa_kernel(Decode2Args a) {
  using Q = GeoQ<KB, VB, VQJL, G>;
  constexpr int S = Q::S;
  static_assert(S >= 4 && S % kPersistGroups == 0, "ring stages");
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_stage = smem + Q::sm_stage0;
  uint64_t *s_full = reinterpret_cast<uint64_t *>(smem + Q::sm_bar);  // [S][4 quarters]
  float *s_q = reinterpret_cast<float *>(smem + Q::sm_q);              // [G][128]
  int *s_pre = reinterpret_cast<int *>(smem + Q::sm_misc);
  int *s_len = s_pre + kMaxPersistBatch + 1;
  float *park = reinterpret_cast<float *>(smem + Q::sm_park);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, grp = warp >> 2, qtr = warp & 3;
  const int g = lane >> 2, t4 = lane & 3;
  const int B = a.batch, H = a.heads_kv;
  // head-independent tables: value pairs, and key pairs as (hi, lo) fp16 of the centroids
  build_value_table<VB, kPersistWarps * 32>(smem, Q::vlut, a.v_centroids, tid);
  {
    uint2 *kl = reinterpret_cast<uint2 *>(smem + Q::sm_klut);
    constexpr int M = (1 << KB) - 1;
    for (int e = tid; e < Q::kval * 32; e += blockDim.x) {
      const int f = e >> 5;
      const float c0 = __ldg(a.k_centroids + (f & M)), c1 = __ldg(a.k_centroids + (f >> KB));
      const __half h0 = __float2half_rn(c0), h1 = __float2half_rn(c1);
      const __half l0 = __float2half_rn(c0 - __half2float(h0)), l1 = __float2half_rn(c1 - __half2float(h1));
      kl[e] = make_uint2((uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16),
                         (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16));
    }
  }
  pdl_trigger();  // the tables above read context constants only
  pdl_wait();
  for (int i = tid; i <= B; i += blockDim.x) s_pre[i] = __ldg(a.tile_prefix + i);
  for (int i = tid; i < B; i += blockDim.x) s_len[i] = min(max(__ldg(a.seq_lens + i), 0), a.capacity);
  if (tid < S * 4) mbar_init(&s_full[tid], 1);
  mbar_fence_init();
  __syncthreads();
  const long long T = (long long)H * s_pre[B];
  const long long C = gridDim.x, c = blockIdx.x, T4 = (T + 3) / 4;
  const int g0 = (int)min(T, 4 * (T4 * c / C)), g1 = (int)min(T, 4 * (T4 * (c + 1) / C));
  if (g0 >= g1) return;
  const int nloc = g1 - g0;
  auto batch_of = [&](int gg) -> int {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * s_pre[mid] <= gg) lo = mid;
      else hi = mid;
    }
    return lo;
  };
  using Gs = typename Q::Gs;
  // this warp's copies in batches of 32 sources, one per lane, as in the one-head kernel
  int cur_i = grp;
  const uint8_t *src_lane = nullptr;
  int src_next = 32;
  auto refill_sources = [&]() {
    const int li = cur_i + kPersistGroups * lane;
    const uint8_t *p = nullptr;
    if (li < nloc) {
      const int gq = g0 + li;
      const int bq = batch_of(gq);
      const int nb = s_pre[bq + 1] - s_pre[bq];
      const int r = gq - H * s_pre[bq];
      const int hq = r / nb, tq_ = r - hq * nb;
      const int t0 = tq_ * kTT + 16 * qtr;
      if (t0 < s_len[bq]) {
        const long long vslot = ((long long)bq * H + hq) * a.cap16 + t0;
        if (a.btab) p = pool_block<Q::block>(a, __ldg(a.btab + (vslot >> 4)));
        else p = a.records + (vslot >> 4) * Q::block;
      }
    }
    src_lane = p;
    src_next = 0;
  };
  auto issue_next = [&]() {
    const int stn = cur_i % S;
    uint64_t *bar = &s_full[stn * 4 + qtr];
    if (src_next == 32) refill_sources();
    const uint8_t *src = reinterpret_cast<const uint8_t *>(
        __shfl_sync(kFull, reinterpret_cast<unsigned long long>(src_lane), src_next++));
    if (lane == 0) {  // the quarter is one stored block: one bulk copy
      mbar_arrive_expect_tx(bar, src ? (uint32_t)Q::block : 0u);
      if (src) tma_load_1d(s_stage + stn * Q::stage + qtr * Q::block, src, (uint32_t)Q::block, bar);
    }
    cur_i += kPersistGroups;
  };
  for (int k = 0; k < S / kPersistGroups && cur_i < nloc; ++k) issue_next();

  // queries of unit u (= batch b, kv head hk): query rows (b, hk G + h), h < G
  auto unit_of = [&](int gg) -> int {
    const int bb = batch_of(gg);
    const int nb = s_pre[bb + 1] - s_pre[bb];
    return bb * H + (gg - H * s_pre[bb]) / nb;
  };
  for (int e = tid; e < G * kD; e += blockDim.x) s_q[e] = __ldg(a.qprep + (size_t)unit_of(g0) * G * 2 * kD +
                                                              (size_t)(e / kD) * 2 * kD + (e % kD));
  __syncthreads();
  bool bad = false;
  int gseg = g0;
  while (gseg < g1) {
    const int bb = batch_of(gseg);
    const int nb = s_pre[bb + 1] - s_pre[bb];
    const int ubase = H * s_pre[bb];
    const int hk = (gseg - ubase) / nb;
    const int us = ubase + hk * nb;
    const int se = min(us + nb, g1);
    const int len = s_len[bb];
    const int u = bb * H + hk;
    // B fragments of the key MMA: column 2h + part = hi / lo of query h (log2 e folded in);
    // rows k = 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1) of block kb are coordinates 16 kb + k
    uint32_t bk[8][2];
    {
      const int hh = g >> 1;
      const bool lop = (g & 1) != 0, live = g < 2 * G;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int k0 = 16 * kb + 2 * t4 + 8 * r;
          const float q0 = live ? s_q[hh * kD + k0] * kLog2e : 0.f, q1 = live ? s_q[hh * kD + k0 + 1] * kLog2e : 0.f;
          const __half h0 = __float2half_rn(q0), h1 = __float2half_rn(q1);
          const __half e0 = lop ? __float2half_rn(q0 - __half2float(h0)) : h0;
          const __half e1 = lop ? __float2half_rn(q1 - __half2float(h1)) : h1;
          bk[kb][r] = (uint32_t)__half_as_ushort(e0) | ((uint32_t)__half_as_ushort(e1) << 16);
        }
    }
    __syncthreads();  // every warp has its fragments: s_q may take the next head's queries
    if (se < g1)
      for (int e = tid; e < G * kD; e += blockDim.x)
        s_q[e] = __ldg(a.qprep + (size_t)unit_of(se) * G * 2 * kD + (size_t)(e / kD) * 2 * kD + (e % kD));

    float m_run = -INFINITY, l_run = 0.f, w_run = 0.f;
    float acc[8][4];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mb][j] = 0.f;
    for (int t = gseg + ((grp - ((gseg - g0) & 3)) & 3); t < se; t += kPersistGroups) {
      const int i = t - g0;
      const int stage = i % S;
      if (!bad && !mbar_wait_bounded(&s_full[stage * 4 + qtr], (uint32_t)((i / S) & 1), a.error)) bad = true;
      bad = __any_sync(kFull, bad);
      if (!bad)
        tile_body_gqa<Q, KB, VB, VQJL, G>(s_stage + stage * Q::stage, smem, qtr * 16, (t - us) * kTT, len, lane,
                                          bk, m_run, l_run, w_run, acc);
      __syncwarp();
      if (cur_i < nloc) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_next();
      }
    }

    // flush, one warp group at a time through the park area [4 warps][G][260]:
    // lane (g, t) parks head t of its warp (value rows 16mb + g, 16mb + 8 + g)
    float lsum = l_run, wsum = w_run;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lsum += __shfl_xor_sync(kFull, lsum, o);
      wsum += __shfl_xor_sync(kFull, wsum, o);
    }
    for (int gr = 0; gr < kPersistGroups; ++gr) {
      __syncthreads();
      if (grp == gr && t4 < G) {
        float *dst = park + (qtr * G + t4) * kPartialFloats;
        if (g == 0) {
          dst[0] = m_run;
          dst[1] = lsum;
          dst[2] = wsum;
        }
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          if (VQJL) {  // columns 2t (values) and 2t + 1 (signs, rows in the sign MMA's order)
            dst[4 + 16 * mb + g] = acc[mb][0];
            dst[4 + 16 * mb + 8 + g] = acc[mb][2];
            const int c0 = 64 * (g & 1) + 8 * mb + 2 * (g >> 1);
            dst[4 + kD + c0] = acc[mb][1] * sign_unscale(sign_land(2 * mb));
            dst[4 + kD + c0 + 1] = acc[mb][3] * sign_unscale(sign_land(2 * mb + 1));
          } else {  // columns 2t, 2t + 1: hi and lo parts of the values
            dst[4 + 16 * mb + g] = acc[mb][0] + acc[mb][1];
            dst[4 + 16 * mb + 8 + g] = acc[mb][2] + acc[mb][3];
          }
        }
      }
      __syncthreads();
      if (tid < G * kD) {
        const int hh = tid / kD, i = tid % kD;
        // the four warps' records of head hh sit at stride G records
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, park[(w * G + hh) * kPartialFloats]);
        float L = 0.f, A = 0.f, Sg = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float *p = park + (w * G + hh) * kPartialFloats;
          const float e = (p[0] == -INFINITY) ? 0.f : ex2_approx(p[0] - M);
          L += p[1] * e;
          A += p[4 + i] * e;
          if (VQJL) Sg += (2.f * p[4 + kD + i] - p[2]) * e;
        }
        float *rec = a.partials + (((size_t)(c + u) * kPersistGroups + gr) * G + hh) * kPartialFloats;
        if (i == 0) {
          rec[0] = M * kLn2;
          rec[1] = L;
        }
        rec[2 + i] = A;
        rec[2 + kD + i] = Sg;
      }
    }
    __syncthreads();
    gseg = se;
  }
}

template <int KB, int VB, bool KQJL, bool VQJL>
int launch_split(const Decode2Args &k, dim3 grid, cudaStream_t st) {
  using Gm = Geo<KB, VB, KQJL, VQJL, 4, 3>;
  if (k.bb != Gm::block) return TQ_ERR_UNSUPPORTED;  // the context's record layout is this stage layout
  const size_t smem = Gm::sm_misc;
  auto fn = decode2_g1_kernel<KB, VB, KQJL, VQJL>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  return launch_overlapped(true, fn, grid, dim3(128), smem, st, k) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// persistent grid: one CTA per SM, or one per 4 tiles when the call has fewer (slices start
// at multiples of 4 tiles, so further CTAs would get nothing and only lengthen the combine)
inline int persist_grid(const Decode2Args &k, int num_sms) {
  if (k.tiles_max <= 0) return num_sms;
  return (int)std::max(1LL, std::min((long long)num_sms, (k.tiles_max + 3) / 4));
}

// persistent launch: at most one CTA per SM (the workspace's record count assumes no more)
template <int KB, int VB, bool KQJL, bool VQJL, bool FUSED = false>
int launch_persist(const Decode2Args &k, int num_sms, int *ctas, cudaStream_t st) {
  constexpr int S = persist_stages<KB, VB, KQJL, VQJL>();
  using Gm = Geo<KB, VB, KQJL, VQJL, kPersistWarps, S>;
  if (k.bb != Gm::block) return TQ_ERR_UNSUPPORTED;
  const size_t smem = persist_smem_bytes<Gm>();
  auto fn = decode_persist_kernel<KB, VB, KQJL, VQJL, FUSED>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  *ctas = persist_grid(k, num_sms);
  return launch_overlapped(true, fn, dim3(*ctas), dim3(kPersistWarps * 32), smem, st, k) == cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

template <int KB, int VB, bool VQJL, int G>
int launch_persist_gqa(const Decode2Args &k, int num_sms, int *ctas, cudaStream_t st) {
  using Q = GeoQ<KB, VB, VQJL, G>;
  if (k.bb != Q::block) return TQ_ERR_UNSUPPORTED;
  const size_t smem = Q::total;
  auto fn = decode_persist_gqa_kernel<KB, VB, VQJL, G>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  *ctas = persist_grid(k, num_sms);
  return launch_overlapped(true, fn, dim3(*ctas), dim3(kPersistWarps * 32), smem, st, k) == cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

template <int KB, int VB, bool VQJL>
int launch_gqa_g(const Decode2Args &k, int G, int num_sms, int *ctas, cudaStream_t st) {
  if (G == 2) return launch_persist_gqa<KB, VB, VQJL, 2>(k, num_sms, ctas, st);
  if (G == 4) return launch_persist_gqa<KB, VB, VQJL, 4>(k, num_sms, ctas, st);
  return TQ_ERR_UNSUPPORTED;
}

template <int KB, int VB, bool KQJL, bool VQJL>
int launch_variant(const Decode2Args &k, bool persist, int num_sms, int *ctas, cudaStream_t st) {
  if (persist) return launch_persist<KB, VB, KQJL, VQJL>(k, num_sms, ctas, st);
  *ctas = 0;
  return launch_split<KB, VB, KQJL, VQJL>(k, dim3(k.splits, k.heads_kv, k.batch), st);
}

// tiles of a call whose lengths are at most max_len (+ 1 for a decode step's append)
long long tiles_bound(const DecodeArgs &a) {
  const long long len = std::min<long long>((long long)a.max_len + 1, a.cache->capacity);
  return (long long)a.batch * a.heads_kv * ((len + kTT - 1) / kTT);
}

// Common arguments of the persistent and split-K launches.
Decode2Args decode2_args(const DecodeArgs &a) {
  const tq_ctx *ctx = a.ctx;
  const tq_cache *c = a.cache;
  Decode2Args k{};
  k.records = c->records;
  k.bb = ctx->lay.bb;
  k.cap16 = cap16_of(c->capacity);
  k.btab = c->block_table;
  k.pool_blocks = c->pool_blocks;
  k.capacity = c->capacity;
  k.batch = a.batch;
  k.heads_kv = a.heads_kv;
  k.heads_q = a.heads_q;
  k.chunk = a.chunk;
  k.splits = a.splits;
  k.seq_lens = a.seq_lens;
  k.tile_prefix = a.tile_prefix;
  k.qprep = a.qprep;
  k.partials = a.partials;
  k.k_centroids = ctx->dparams->k_centroids;
  k.v_centroids = ctx->dparams->v_centroids;
  k.error = &ctx->dparams->error;
  k.tiles_max = tiles_bound(a);
  return k;
}

}  // namespace

// The decode step on the persistent kernel (one query head per KV head, keys without a
// sketch, batch <= 256); TQ_ERR_UNSUPPORTED otherwise. The kernel writes the tile prefix
// to a.tile_prefix for the combine.
int launch_decode2_step(const DecodeArgs &a, const StepArgs &s, int *persist_ctas, void *stream) {
  const tq_ctx *ctx = a.ctx;
  *persist_ctas = 0;
  if (a.heads_q != a.heads_kv || a.batch > kMaxPersistBatch || ctx->num_sms <= 0 || !a.tile_prefix)
    return TQ_ERR_UNSUPPORTED;
  if (ctx->scheme != TQ_SCHEME_KV && ctx->scheme != TQ_SCHEME_KQV) return TQ_ERR_UNSUPPORTED;
  // the fused kernel rotates queries and new tokens with the Walsh-Hadamard transform
  if (ctx->scheme == TQ_SCHEME_KQV && ctx->rotation != TQ_ROTATION_WHT) return TQ_ERR_UNSUPPORTED;
  if (ctx->side_rank) return TQ_ERR_UNSUPPORTED;  // key side codes: the general path
  Decode2Args k = decode2_args(a);
  k.tile_prefix = nullptr;
  k.tile_prefix_out = a.tile_prefix;
  k.q_raw = a.q;
  k.q_bf16 = a.q_dtype == TQ_BF16;
  k.q_rotate = ctx->k.rotate ? 1 : 0;
  k.k_new = s.k_new;
  k.v_new = s.v_new;
  k.kv_bf16 = s.kv_dtype == TQ_BF16;
  k.diag = ctx->dparams->diag;
  k.sketch_tp = ctx->dparams->sketch_tp;
  for (int r = 0; r < 2; ++r) {
    WarpRole &o = k.role[r];
    const Role &role = r ? ctx->v : ctx->k;
    const int p0 = r ? TQ_PLANE_V_CODES : TQ_PLANE_K_CODES;
    auto at = [&](int p) -> uint8_t * { return ctx->lay.tok[p] ? a.cache->records + ctx->lay.off[p] : nullptr; };
    o.codes = at(p0);
    o.norms = reinterpret_cast<float *>(at(p0 + 1));
    o.signs = at(p0 + 2);
    o.rnorms = reinterpret_cast<float *>(at(p0 + 3));
    o.bits = role.bits;
    o.rotate = role.rotate ? 1 : 0;
    o.qjl = role.qjl ? 1 : 0;
    o.vt = r;  // value codes are stored pair-interleaved
    const float *bounds = r ? ctx->v_bounds : ctx->k_bounds;
    const float *cents = r ? ctx->v_centroids : ctx->k_centroids;
    const int L = 1 << role.bits;
    for (int i = 0; i < kMaxLevels; ++i) {
      o.bounds[i] = (i < L - 1) ? bounds[i] : __builtin_huge_valf();
      o.centroids[i] = (i < L) ? cents[i] : 0.f;
    }
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int kb = ctx->k.bits, ns = ctx->num_sms;
  if (ctx->scheme == TQ_SCHEME_KV) {
    if (kb == 2) return launch_persist<2, 2, false, false, true>(k, ns, persist_ctas, st);
    if (kb == 3) return launch_persist<3, 3, false, false, true>(k, ns, persist_ctas, st);
    if (kb == 4) return launch_persist<4, 4, false, false, true>(k, ns, persist_ctas, st);
  } else {
    if (kb == 2) return launch_persist<2, 1, false, true, true>(k, ns, persist_ctas, st);
    if (kb == 3) return launch_persist<3, 2, false, true, true>(k, ns, persist_ctas, st);
    if (kb == 4) return launch_persist<4, 3, false, true, true>(k, ns, persist_ctas, st);
  }
  return TQ_ERR_UNSUPPORTED;
}

// Returns TQ_ERR_UNSUPPORTED when this path does not cover the request (the
// caller then uses the general kernel). *persist_ctas receives the persistent
// grid size, or 0 when the split-K kernel ran (partials laid out per split).
int launch_decode2_g1(const DecodeArgs &a, int *persist_ctas, void *stream) {
  const tq_ctx *ctx = a.ctx;
  *persist_ctas = 0;
  const int G = a.heads_q / a.heads_kv;
  if (G != 1) {
    // GQA groups of 2 or 4 query heads, keys without a sketch, on the persistent tensor-core kernel
    if ((G != 2 && G != 4) || ctx->scheme == TQ_SCHEME_QKQV || !a.tile_prefix || a.batch > kMaxPersistBatch ||
        ctx->num_sms <= 0)
      return TQ_ERR_UNSUPPORTED;
    const Decode2Args k = decode2_args(a);
    cudaStream_t st = (cudaStream_t)stream;
    const int kb = ctx->k.bits, ns = ctx->num_sms;
    if (ctx->scheme == TQ_SCHEME_KV) {
      if (kb == 2) return launch_gqa_g<2, 2, false>(k, G, ns, persist_ctas, st);
      if (kb == 3) return launch_gqa_g<3, 3, false>(k, G, ns, persist_ctas, st);
      if (kb == 4) return launch_gqa_g<4, 4, false>(k, G, ns, persist_ctas, st);
    } else if (ctx->scheme == TQ_SCHEME_KQV) {
      if (kb == 2) return launch_gqa_g<2, 1, true>(k, G, ns, persist_ctas, st);
      if (kb == 3) return launch_gqa_g<3, 2, true>(k, G, ns, persist_ctas, st);
      if (kb == 4) return launch_gqa_g<4, 3, true>(k, G, ns, persist_ctas, st);
    }
    return TQ_ERR_UNSUPPORTED;
  }
  // tiles (persistent) and chunks (split-K) start at multiples of 16 tokens, i.e. at
  // whole blocks of the records, which are 16-byte aligned
  const bool persist = a.tile_prefix != nullptr && a.batch <= kMaxPersistBatch && ctx->num_sms > 0;
  if (!persist && a.chunk % kBlockTokens) return TQ_ERR_UNSUPPORTED;
  const Decode2Args k = decode2_args(a);
  cudaStream_t st = (cudaStream_t)stream;
  const int kb = ctx->k.bits, ns = ctx->num_sms;
  int *pc = persist_ctas;
  switch (ctx->scheme) {
    case TQ_SCHEME_KV:
      if (kb == 2) return launch_variant<2, 2, false, false>(k, persist, ns, pc, st);
      if (kb == 3) return launch_variant<3, 3, false, false>(k, persist, ns, pc, st);
      if (kb == 4) return launch_variant<4, 4, false, false>(k, persist, ns, pc, st);
      break;
    case TQ_SCHEME_KQV:
      if (kb == 2) return launch_variant<2, 1, false, true>(k, persist, ns, pc, st);
      if (kb == 3) return launch_variant<3, 2, false, true>(k, persist, ns, pc, st);
      if (kb == 4) return launch_variant<4, 3, false, true>(k, persist, ns, pc, st);
      break;
    case TQ_SCHEME_QKQV:
      if (kb == 1) return launch_variant<1, 1, true, true>(k, persist, ns, pc, st);
      if (kb == 2) return launch_variant<2, 2, true, true>(k, persist, ns, pc, st);
      if (kb == 3) return launch_variant<3, 3, true, true>(k, persist, ns, pc, st);
      break;
    default: break;
  }
  return TQ_ERR_UNSUPPORTED;
}

}  // namespace tq
