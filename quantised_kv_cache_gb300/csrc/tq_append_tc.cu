// Append-quantise for rotated vectors (keys and values of KQV and QKQV), one
// thread per vector, with the rotation and the QJL sketch on tcgen05 tensor
// cores.
//
// "Statistical Inference ... Inspired by TurboQuant", technical summary,
// "Quantisation schemes" and "Main contribution 1": normalise, rotate with the
// randomised WHT, code each coordinate with the Lloyd-Max codebook; sketched
// vectors also keep sign(S r) and rho = ||x|| ||r|| of the unit-domain
// residual r = y - c[code]. "KVQuant++", "Fast codebook lookup": a code is a
// count of boundaries, found by binary search.
//
// A CTA of 128 threads handles 128 vectors per pass (thread t <-> vector t <->
// TMEM lane t), in phases:
// 1. load x, nu = ||x||; x' = x 2^-floor(log2 nu) split into fp16 hi + lo is
//    stored to tensor memory as the A operand (the hi / lo split is exact to
//    about 2^-22, the power of two keeps fp16 in range);
// 2. y' = H D x' on the tensor cores: B = the Hadamard matrix times the seeded
//    diagonal (entries +-1, exact in fp16; prepared once per context) with its
//    rows in code-storage order, so accumulator column n is
//    the coordinate stored at code offset n (pair-slot order); two passes
//    (hi, lo), fp32 accumulate;
// 3. in four 32-column chunks read back with tcgen05.ld: codes against the
//    boundaries scaled to the vector (nu sqrt(d) b_j 2^-floor(log2 nu), so no
//    division), stored chunk by chunk; for sketched vectors the residual
//    r = y / (nu sqrt(d)) - c[code], scaled by 2^10 and split into fp16 hi +
//    lo, becomes the next A operand;
// 4. sketched vectors: z = S r on the tensor cores (S as fp16 hi + lo with both
//    its rows and its columns in the same storage order; three passes hi x hi,
//    lo x hi, hi x lo), column n = sign offset n of the stored record; signs
//    come out 32 at a time. Any |z| within a bound on the dropped terms and the
//    accumulation error is recomputed in fp32 from the residual rebuilt from
//    its hi + lo parts (2^-22 relative), so a sign can differ from exact
//    arithmetic only where |z| is about 1e-6 or less.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_ptx.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

struct TcArgs {
  const void *x;
  int batch, heads, n_new, capacity, cap16, bb;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  int vt;  // value role: codes in the pair-interleaved layout
  const int32_t *seq_lens;
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  const float *sketch;          // S, fp32 [128][128] row-major (rare-path exact signs)
  const uint16_t *bh;           // B operand of the rotation (DevParams::hadamard_b, or the dense hi part)
  const uint16_t *bm_lo;        // dense rotation: the lo part of sqrt(d) M (nullptr: Walsh-Hadamard)
  const uint16_t *bs;           // B operand of the sketch, hi then lo (DevParams::sketch_hl)
  float sketch_rowmax;
  int *error;
  // key side codes (side_rank > 0): plane base and the bases in code-storage order
  int side_rank;
  uint16_t *side;
  const float *side_urs;
  float bounds[kMaxLevels];     // 2^BITS - 1 used
  float centroids[kMaxLevels];  // 2^BITS used
};

constexpr int kQV = 128;               // vectors per pass = MMA M
constexpr uint32_t kTmemCols = 256;    // D [0, 128) | A hi [128, 192) | A lo [192, 256)
constexpr int kOpBytes = kD * kD * 2;  // one fp16 128 x 128 operand
constexpr float kSqrtD = 11.313708498984761f;
constexpr float kRScale = 1024.f;      // residual scale for the fp16 split (|r| < 2)

// coordinate stored at code (or sign) offset n: n = 32t + 2m + e holds 8m + 2t + e
__host__ __device__ __forceinline__ int slot_coord_tc(int n) {
  const int ps = n >> 1, e = n & 1;
  return 8 * (ps & 15) + 2 * (ps >> 4) + e;
}

// byte offset of element (row n, K index k) of a K-major core-matrix operand
__device__ __forceinline__ int core_off(int n, int k) {
  return (n >> 3) * 2048 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}

template <int H>
__device__ __forceinline__ int count_pos(float a, const float (&P)[H > 0 ? H : 1]) {
  if constexpr (H == 0) {
    return 0;
  } else if constexpr (H == 1) {
    return a >= P[0] ? 1 : 0;
  } else if constexpr (H == 3) {
    int m = a >= P[1] ? 2 : 0;
    const float c = m ? P[2] : P[0];
    return m + (a >= c ? 1 : 0);
  } else {  // H == 7
    int m = a >= P[3] ? 4 : 0;
    const float c2 = m ? P[5] : P[1];
    m += a >= c2 ? 2 : 0;
    const float c1 = (m & 4) ? ((m & 2) ? P[6] : P[4]) : ((m & 2) ? P[2] : P[0]);
    return m + (a >= c1 ? 1 : 0);
  }
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};\n\ttcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// (a, b) -> fp16x2 hi = rn(a, b) and lo = rn(a - hi, b - hi), packed (lower element low)
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Rare path, entered by whole warps (tcgen05.ld is warp-collective): rebuild each
// thread's residual (storage order, hi + lo) from TMEM and take its flagged signs
// from an fp32 S r. Column c of the residual is coordinate slot_coord_tc(c).
__device__ __noinline__ void certify_signs_tc(uint32_t tlane_a, const float *sketch, uint32_t (&flag)[4],
                                              uint32_t (&sw)[4]) {
  float r[kD];
#pragma unroll
  for (int chunk = 0; chunk < 2; ++chunk) {
    uint32_t hi[32], lo[32];
    tmem_ld_x32(tlane_a + 32 * chunk, hi);
    tmem_ld_x32(tlane_a + 64 + 32 * chunk, lo);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int k = 2 * (32 * chunk + c);
      r[k] = (__half2float(__ushort_as_half((unsigned short)(hi[c] & 0xffffu))) +
              __half2float(__ushort_as_half((unsigned short)(lo[c] & 0xffffu)))) * (1.f / kRScale);
      r[k + 1] = (__half2float(__ushort_as_half((unsigned short)(hi[c] >> 16))) +
                  __half2float(__ushort_as_half((unsigned short)(lo[c] >> 16)))) * (1.f / kRScale);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    while (flag[q]) {
      const int bit = __ffs(flag[q]) - 1;
      flag[q] &= flag[q] - 1u;
      const float *row = sketch + (size_t)slot_coord_tc(32 * q + bit) * kD;
      float zz = 0.f;
#pragma unroll
      for (int c = 0; c < kD; ++c) zz = fmaf(__ldg(row + slot_coord_tc(c)), r[c], zz);
      sw[q] = (sw[q] & ~(1u << bit)) | ((zz >= 0.f ? 1u : 0u) << bit);
    }
  }
}

template <int BITS, bool QJL, bool BF16>
__global__ void __launch_bounds__(kQV, 2) append_tc_kernel(const __grid_constant__ TcArgs a) {
  constexpr int L = 1 << BITS, H = L / 2 - 1;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_bh = smem;                 // rotation B operand
  unsigned char *s_bs = smem + kOpBytes;      // sketch B operand, hi then lo (QJL)
  constexpr int kOps = QJL ? 3 : 1;
  const bool dense = a.bm_lo != nullptr;      // dense rotation: a lo part follows the others
  unsigned char *s_bl = smem + kOps * kOpBytes;
  const int nops = kOps + (dense ? 1 : 0);
  uint64_t *s_bar = reinterpret_cast<uint64_t *>(smem + nops * kOpBytes);
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(smem + nops * kOpBytes + 8);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(s_bar, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(s_bar, nops * kOpBytes);
    tma_load_1d(s_bh, a.bh, kOpBytes, s_bar);
    if (QJL) {
      tma_load_1d(s_bs, a.bs, kOpBytes, s_bar);
      tma_load_1d(s_bs + kOpBytes, a.bs + kD * kD, kOpBytes, s_bar);
    }
    if (dense) tma_load_1d(s_bl, a.bm_lo, kOpBytes, s_bar);
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(smem_u32(s_taddr), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  bool bad = !mbar_wait_bounded(s_bar, 0, a.error);  // phase 0: the operand copies
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *s_taddr;
  const uint32_t tlane = tbase + ((uint32_t)(warp * 32) << 16);  // this warp's TMEM lanes
  const uint32_t sa_h = smem_u32(s_bh), sa_s = smem_u32(s_bs), sa_l = smem_u32(s_bl);
  constexpr uint32_t idesc = tc_idesc_f16_f32(128, 128);
  const float smax = a.sketch_rowmax;
  float P[H > 0 ? H : 1], CP[H + 1];
#pragma unroll
  for (int k = 0; k <= H; ++k) CP[k] = a.centroids[L / 2 + k];

  const long long total = (long long)a.batch * a.heads * a.n_new;
  bad = __syncthreads_or(bad);
  uint32_t phase = 1;  // mbarrier phase 0 was the operand copies
  for (long long base = (long long)blockIdx.x * kQV; base < total && !bad;
       base += (long long)gridDim.x * kQV) {
    // ---------------- 1. load, norm, A = D x 2^-e as fp16 hi + lo
    const long long vec = base + tid;
    long long slot = -1;
    int head = 0;
    if (vec < total) {
      const int t = (int)(vec % a.n_new);
      const long long bh = vec / a.n_new;
      head = (int)(bh % a.heads);
      const int b = (int)(bh / a.heads);
      const int len = __ldg(a.seq_lens + b);
      if (len >= 0 && len + a.n_new <= a.capacity) slot = phys_slot(a.btab, a.pool_blocks, bh * a.cap16 + len + t, a.error);
      else if (t == 0) set_error(a.error, TQ_ERR_CAPACITY);  // the sequence is skipped whole
    }
    float nu, xs;
    {
      float x[kD];
      if (slot >= 0) {
        if (BF16) {
          const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + vec * kD);
#pragma unroll
          for (int k = 0; k < kD / 8; ++k) {
            const uint4 w = __ldg(src + k);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              x[8 * k + 2 * j] = __uint_as_float(ww[j] << 16);
              x[8 * k + 2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
            }
          }
        } else {
          const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + vec * kD);
#pragma unroll
          for (int k = 0; k < kD / 4; ++k) {
            const float4 f = __ldg(src + k);
            x[4 * k] = f.x;
            x[4 * k + 1] = f.y;
            x[4 * k + 2] = f.z;
            x[4 * k + 3] = f.w;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < kD; ++i) x[i] = 0.f;
      }
      float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kD; ++i) sq[i & 3] = fmaf(x[i], x[i], sq[i & 3]);
      nu = sqrtf((sq[0] + sq[1]) + (sq[2] + sq[3]));
      // 2^-floor(log2 nu): |x_i| 2^-e < 2, well inside fp16
      xs = (nu > 0.f) ? __int_as_float((254 - ((__float_as_int(nu) >> 23) & 0xff)) << 23) : 1.f;
      // (the diagonal D sits in the rotation operand's columns)
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        uint32_t wh[32], wl[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k = 2 * (32 * chunk + c);
          split_pair(x[k] * xs, x[k + 1] * xs, wh[c], wl[c]);
        }
        __syncwarp();
        tmem_st_x32(tlane + 128 + 32 * chunk, wh);
        tmem_st_x32(tlane + 192 + 32 * chunk, wl);
      }
    }
    tc_fence_before_sync();
    __syncthreads();

    // ---------------- 2. y' = H x' (columns in code-storage order); a dense rotation
    // sqrt(d) M = B_hi + B_lo adds the pass x'_hi B_lo (x'_lo B_lo, about 2^-44, is dropped)
    if (tid == 0) {
      tc_fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t db = tc_sdesc_kmajor(sa_h + 256 * ks, 128, 2048);
        tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, db, idesc, ks > 0);
        tc_mma_f16_ts(tbase, tbase + 192 + 8 * ks, db, idesc, true);
        if (dense) tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, tc_sdesc_kmajor(sa_l + 256 * ks, 128, 2048), idesc, true);
      }
      tc_commit(smem_u32(s_bar));
    }
    if (!mbar_wait_bounded(s_bar, phase & 1, a.error)) bad = true;
    else ++phase;
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
    tc_fence_after_sync();

    // ---------------- 3. codes (and residuals) 32 storage offsets at a time
    const float sv = (nu > 0.f) ? nu * kSqrtD * xs : 1.f;  // boundary scale
    const float inv = (nu > 0.f) ? kRScale / (nu * kSqrtD * xs) : 0.f;
#pragma unroll
    for (int k = 0; k < H; ++k) P[k] = a.bounds[L / 2 + k] * sv;
    float rr = 0.f;
    uint32_t *crec = reinterpret_cast<uint32_t *>(rec_at(a.codes, slot >= 0 ? slot : 0, a.bb, BITS * kD / 8));
    // value codes: is the other token of this token's pair (slot ^ 1) the neighbouring lane's?
    const long long pslot = ((long long)__shfl_xor_sync(kFull, (int)(slot >> 32), 1) << 32) |
                            (uint32_t)__shfl_xor_sync(kFull, (int)(uint32_t)slot, 1);
    const bool paired = slot >= 0 && pslot >= 0 && pslot == (slot ^ 1);
    const int half = (int)(slot & 1);
    // side code of an unsketched key: z_k = nu sum_n U[n][k] (y_n / ||y|| - c[code_n]) over
    // the storage offsets n (the basis stored in the same order)
    const int srank = QJL ? 0 : a.side_rank;
    const float *su = srank ? a.side_urs + (size_t)head * kD * srank : nullptr;
    const float inv_unit = (nu > 0.f) ? 1.f / (nu * kSqrtD * xs) : 0.f;
    float zs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t yz[32];
      __syncwarp();  // tcgen05.ld / st are warp-collective
      tmem_ld_x32(tlane + 32 * q, yz);
      // key records: BITS words per chunk in code-offset order; value codes: the chunk's 32
      // fields of the pair row (2 BITS words), this token's half
      uint32_t word[2 * BITS], vw[2 * BITS];
#pragma unroll
      for (int w = 0; w < 2 * BITS; ++w) word[w] = vw[w] = 0u;
      uint32_t rh[16], rl[16];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float y = __uint_as_float(yz[j]);
        const int m = count_pos<H>(fabsf(y), P);
        const int code = (y >= 0.f) ? (L / 2 + m) : (L / 2 - 1 - m);
        const int off = BITS * j;
        word[off >> 5] |= (uint32_t)code << (off & 31);
        if ((off & 31) + BITS > 32) word[(off >> 5) + 1] |= (uint32_t)code >> (32 - (off & 31));
        const int voff = 2 * BITS * (16 * (j & 1) + (j >> 1));
        vw[voff >> 5] |= (uint32_t)code << (voff & 31);
        if ((voff & 31) + BITS > 32) vw[(voff >> 5) + 1] |= (uint32_t)code >> (32 - (voff & 31));
        if (QJL) {
          float cm = CP[0];
#pragma unroll
          for (int k = 1; k <= H; ++k) cm = (m == k) ? CP[k] : cm;
          // r 2^10 = y' inv - c 2^10
          const float r = fmaf(y, inv, (y >= 0.f) ? -cm * kRScale : cm * kRScale);
          rr = fmaf(r, r, rr);
          yz[j] = __float_as_uint(r);
        } else if (srank) {
          float cm = CP[0];
#pragma unroll
          for (int k = 1; k <= H; ++k) cm = (m == k) ? CP[k] : cm;
          const float r = fmaf(y, inv_unit, (y >= 0.f) ? -cm : cm);
          const float *un = su + (32 * q + j) * srank;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (k < srank) zs[k] = fmaf(__ldg(un + k), r, zs[k]);
        }
      }
      if (a.vt) {  // warp-uniform
        if (half) {
#pragma unroll
          for (int i = 2 * BITS - 1; i > 0; --i) vw[i] = (vw[i] << BITS) | (vw[i - 1] >> (32 - BITS));
          vw[0] <<= BITS;
        }
        vt_store_chunk<BITS>(vt_row<BITS>(a.codes, slot >= 0 ? slot : 0, a.bb), q, vw, half, paired, slot >= 0);
      } else if (slot >= 0) {
#pragma unroll
        for (int w = 0; w < BITS; ++w) crec[BITS * q + w] = word[w];
      }
      if (QJL) {
#pragma unroll
        for (int p = 0; p < 16; ++p) split_pair(__uint_as_float(yz[2 * p]), __uint_as_float(yz[2 * p + 1]), rh[p], rl[p]);
        __syncwarp();
        tmem_st_x16(tlane + 128 + 16 * q, rh);
        tmem_st_x16(tlane + 192 + 16 * q, rl);
      }
    }
    if (slot >= 0) *rec_at(a.norms, slot, a.bb, 4) = nu;
    if (srank && slot >= 0) {
      uint16_t *zp = rec_at(a.side, slot, a.bb, 2 * srank);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < srank) zp[k] = __half_as_ushort(__float2half_rn(zs[k] * nu));
    }

    if constexpr (QJL) {
      tc_fence_before_sync();
      __syncthreads();
      // ---------------- 4. z = S r (rows and columns in storage order)
      if (tid == 0) {
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t dh = tc_sdesc_kmajor(sa_s + 256 * ks, 128, 2048);
          const uint64_t dl = tc_sdesc_kmajor(sa_s + kOpBytes + 256 * ks, 128, 2048);
          tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, dh, idesc, ks > 0);
          tc_mma_f16_ts(tbase, tbase + 192 + 8 * ks, dh, idesc, true);
          tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, dl, idesc, true);
        }
        tc_commit(smem_u32(s_bar));
      }
      if (!mbar_wait_bounded(s_bar, phase & 1, a.error)) bad = true;
      else ++phase;
      if (__syncthreads_or(bad)) {
        bad = true;
        break;
      }
      tc_fence_after_sync();
      // dropped terms + accumulation error of z' = 2^10 S r (see the file comment)
      const float E = 0x1p-16f * smax * sqrtf(rr) + 0x1p-20f * smax;
      uint32_t sw[4], flag[4];
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t z[32];
        __syncwarp();
        tmem_ld_x32(tlane + 32 * q, z);
        uint32_t wv = 0u, fv = 0u;
#pragma unroll
        for (int bit = 0; bit < 32; ++bit) {
          const float zf = __uint_as_float(z[bit]);
          wv |= (zf >= 0.f ? 1u : 0u) << bit;
          fv |= (fabsf(zf) <= E ? 1u : 0u) << bit;
        }
        // q is dynamic here: keep the words in a fixed register order
        sw[0] = (q == 0) ? wv : sw[0];
        sw[1] = (q == 1) ? wv : sw[1];
        sw[2] = (q == 2) ? wv : sw[2];
        sw[3] = (q == 3) ? wv : sw[3];
        flag[0] = (q == 0) ? fv : flag[0];
        flag[1] = (q == 1) ? fv : flag[1];
        flag[2] = (q == 2) ? fv : flag[2];
        flag[3] = (q == 3) ? fv : flag[3];
      }
      if (__any_sync(kFull, (flag[0] | flag[1] | flag[2] | flag[3]) != 0u)) {
        __syncwarp();
        certify_signs_tc(tlane + 128, a.sketch, flag, sw);
      }
      if (slot >= 0) {
        float rho = nu * sqrtf(rr) * (1.f / kRScale);
        if (nu == 0.f) {  // a zero vector: every sign set, rho = 0
          sw[0] = sw[1] = sw[2] = sw[3] = 0xffffffffu;
          rho = 0.f;
        }
        *reinterpret_cast<uint4 *>(rec_at(a.signs, slot, a.bb, kD / 8)) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
        *rec_at(a.rnorms, slot, a.bb, 4) = rho;
      }
    }
    // the next pass overwrites A and D only after every thread passed its barrier
    tc_fence_before_sync();
  }

  // ---------------- teardown: no tensor-core work in flight, then free TMEM
  if (bad) mbar_wait_bounded(s_bar, phase & 1, a.error);  // the stuck phase, bounded: a last chance
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// B operands, once per context: the rotation H D (rows in storage order) and S split
// into fp16 hi + lo (rows and columns in storage order), K-major core matrices
__global__ void __launch_bounds__(128) operand_prep_kernel(DevParams *dp) {
  const int n = threadIdx.x;
  unsigned char *bh = reinterpret_cast<unsigned char *>(dp->hadamard_b);
  unsigned char *shi = reinterpret_cast<unsigned char *>(dp->sketch_hl);
  unsigned char *slo = shi + kOpBytes;
  const int i = slot_coord_tc(n);  // the coordinate (or sketch row) of storage offset n
  for (int k = 0; k < kD; ++k) {
    const float h = ((__popc(i & k) & 1) ? -1.f : 1.f) * dp->diag[k];  // (H D)[i][k]
    *reinterpret_cast<__half *>(bh + core_off(n, k)) = __float2half_rn(h);
    *reinterpret_cast<__nv_bfloat16 *>(reinterpret_cast<unsigned char *>(dp->hadamard_bf) + core_off(n, k)) =
        __float2bfloat16_rn(h);
    const float s = dp->sketch[i * kD + slot_coord_tc(k)];
    dp->sketch_perm[n * kD + k] = s;
    const __half sh = __float2half_rn(s);
    *reinterpret_cast<__half *>(shi + core_off(n, k)) = sh;
    *reinterpret_cast<__half *>(slo + core_off(n, k)) = __float2half_rn(s - __half2float(sh));
  }
}

// The dense rotation's B operands, once per context: sqrt(d) M (rows in storage order)
// split into fp16 hi + lo, K-major core matrices as for H D above.
__global__ void __launch_bounds__(128) rotation_prep_kernel(DevParams *dp) {
  const int n = threadIdx.x;
  unsigned char *hi = reinterpret_cast<unsigned char *>(dp->rot_hl);
  unsigned char *lo = hi + kOpBytes;
  const int i = slot_coord_tc(n);
  for (int k = 0; k < kD; ++k) {
    const float v = dp->rot[i * kD + k] * kSqrtD;
    const __half h = __float2half_rn(v);
    *reinterpret_cast<__half *>(hi + core_off(n, k)) = h;
    *reinterpret_cast<__half *>(lo + core_off(n, k)) = __float2half_rn(v - __half2float(h));
  }
}

int g_sms_tc = 0;

template <int BITS, bool QJL, bool BF16>
int go(const TcArgs &k, long long total, cudaStream_t st) {
  if (g_sms_tc == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_tc, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms_tc <= 0) g_sms_tc = 152;
  }
  // shared memory sized so that at most two CTAs share an SM (their TMEM totals 512 columns);
  // a dense rotation's extra operand leaves sketched roles at one CTA per SM
  constexpr int smem_max = QJL ? 4 * kOpBytes + 64 : 80 * 1024;
  const int smem = QJL ? (k.bm_lo ? 4 : 3) * kOpBytes + 64 : 80 * 1024;
  auto fn = append_tc_kernel<BITS, QJL, BF16>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  long long blocks = (total + kQV - 1) / kQV;
  const long long cap = 2LL * g_sms_tc;  // persistent: two CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fn<<<(unsigned)blocks, kQV, smem, st>>>(k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <bool QJL, bool BF16>
int dispatch(int bits, const TcArgs &k, long long total, cudaStream_t st) {
  switch (bits) {
    case 1: return go<1, QJL, BF16>(k, total, st);
    case 2: return go<2, QJL, BF16>(k, total, st);
    case 3: return go<3, QJL, BF16>(k, total, st);
    case 4: return go<4, QJL, BF16>(k, total, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_rotation_prep(DevParams *dp, void *stream) {
  rotation_prep_kernel<<<1, kD, 0, (cudaStream_t)stream>>>(dp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

int launch_operand_prep(DevParams *dp, void *stream) {
  operand_prep_kernel<<<1, kD, 0, (cudaStream_t)stream>>>(dp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Tensor-core append for rotated vectors; TQ_ERR_UNSUPPORTED otherwise.
int launch_append_tc(const AppendArgs &a, const tq_ctx *ctx, void *stream) {
  if (!a.role.rotate || a.role.bits < 1 || a.role.bits > 4 || (a.role.qjl && a.role.bits > 3))
    return TQ_ERR_UNSUPPORTED;
  TcArgs k{};
  k.x = a.x;
  k.batch = a.batch;
  k.heads = a.heads;
  k.n_new = a.n_new;
  k.capacity = a.capacity;
  k.cap16 = a.cap16;
  k.bb = a.bb;
  k.btab = a.btab;
  k.pool_blocks = a.pool_blocks;
  k.vt = a.vt;
  k.seq_lens = a.seq_lens;
  k.codes = a.codes;
  k.norms = a.norms;
  k.signs = a.signs;
  k.rnorms = a.rnorms;
  k.sketch = ctx->dparams->sketch;
  const bool dense = ctx->rotation == TQ_ROTATION_DENSE;
  k.bh = dense ? ctx->dparams->rot_hl : ctx->dparams->hadamard_b;
  k.bm_lo = dense ? ctx->dparams->rot_hl + kD * kD : nullptr;
  k.bs = ctx->dparams->sketch_hl;
  k.sketch_rowmax = ctx->sketch_rowmax;
  k.error = a.error;
  k.side_rank = a.side_rank;
  k.side = a.side;
  k.side_urs = a.side_urs;
  const bool is_k = a.centroids == ctx->dparams->k_centroids;
  const float *bsrc = is_k ? ctx->k_bounds : ctx->v_bounds;
  const float *csrc = is_k ? ctx->k_centroids : ctx->v_centroids;
  for (int i = 0; i < (1 << a.role.bits) - 1; ++i) k.bounds[i] = bsrc[i];
  for (int i = 0; i < (1 << a.role.bits); ++i) k.centroids[i] = csrc[i];
  const long long total = (long long)a.batch * a.heads * a.n_new;
  cudaStream_t st = (cudaStream_t)stream;
  const bool bf16 = a.dtype == TQ_BF16;
  if (a.role.qjl) return bf16 ? dispatch<true, true>(a.role.bits, k, total, st)
                              : dispatch<true, false>(a.role.bits, k, total, st);
  return bf16 ? dispatch<false, true>(a.role.bits, k, total, st) : dispatch<false, false>(a.role.bits, k, total, st);
}

}  // namespace tq
