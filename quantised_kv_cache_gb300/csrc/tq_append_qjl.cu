// Append-quantise for vectors that carry a QJL sketch (the values of KQV and
// QKQV, the keys of QKQV), one thread per vector, with the sketch on the
// tensor cores.
//
// "Statistical Inference ... Inspired by TurboQuant", technical summary,
// "Quantisation schemes" and "Main contribution 1": normalise, rotate with the
// randomised WHT, code each coordinate with the Lloyd-Max codebook, and keep
// sign(S r) and rho = ||x|| ||r|| of the unit-domain residual r = y - c[code].
//
// A CTA of 128 threads quantises 128 vectors per pass (thread t <-> vector t
// <-> TMEM lane t). The residuals, scaled by a power of two and split into
// fp16 hi + lo parts, are stored into tensor memory as the A operand of
// tcgen05.mma (M = N = 128, K = 128); S, split the same way, sits in shared
// memory as B. Three passes (hi x hi, lo x hi, hi x lo) accumulate z = S r in
// fp32 in TMEM, and thread t reads back row t: its own 128 sketch values.
//
// Signs are certified: the dropped terms and the accumulation error are bounded
// by 2^-16 max_j ||S_j|| ||r'|| + 2^-20 max_j ||S_j||; any |z| within that bound
// (about 2% of vectors have one) is recomputed in fp32 from the fp32 row of S
// and the residual rebuilt from its hi + lo parts (2^-22 relative), so a sign
// can differ from an exact evaluation only where |z| is about 1e-6 or less.

#include <cuda_fp16.h>

#include "tq_ptx.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

struct QjlArgs {
  const void *x;
  int batch, heads, n_new, capacity;
  const int32_t *seq_lens;
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  const float *sketch;  // S, fp32 [128][128] row-major
  const uint16_t *sketch_hl;  // S fp16 hi + lo in the core-matrix layout (DevParams)
  float sketch_rowmax;
  int *error;
  float diag[kD];
  float bounds[kMaxLevels];     // 2^BITS - 1 used
  float centroids[kMaxLevels];  // 2^BITS used
};

constexpr int kQV = 128;                // vectors per pass = MMA M
constexpr uint32_t kTmemCols = 256;     // D [0, 128) | A hi [128, 192) | A lo [192, 256)
constexpr int kSBytes = kD * kD * 2;    // one fp16 copy of S
constexpr int kSmemQjl = 80 * 1024;     // 2 x 32 KB of S + control; sized so that at most
                                        // two CTAs share an SM (their TMEM totals 512 columns)
constexpr float kSqrtD = 11.313708498984761f;

// sketch row that MMA column n (= sign offset n of the stored record) uses
__device__ __forceinline__ int sketch_row(int n) {
  const int ps = n >> 1, e = n & 1;
  return 8 * (ps & 15) + 2 * (ps >> 4) + e;
}

// count of positive boundaries P[0..H-1] (ascending) at or below a >= 0, and the
// positive centroid cp[m] of that count
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

// Load vector `vec` (zeros when !live), quantise it and leave the unit-domain
// residual r = y / (nu sqrt(128)) - c[code] in x; codes (pair-slot order) in word.
template <int BITS, bool BF16>
__device__ __forceinline__ void quantise_residual(const QjlArgs &a, long long vec, bool live, float (&x)[kD],
                                                  float &nu, float &rr, float &mx, uint32_t (&word)[4 * BITS]) {
  constexpr int L = 1 << BITS, H = L / 2 - 1;
    if (live) {
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
    // squared norm: four interleaved fp32 chains, then their sum
    {
      float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kD; ++i) sq[i & 3] = fmaf(x[i], x[i], sq[i & 3]);
      nu = sqrtf((sq[0] + sq[1]) + (sq[2] + sq[3]));
    }
    // y = H D x, unnormalised (entries +/-1)
#pragma unroll
    for (int i = 0; i < kD; ++i) x[i] *= a.diag[i];
#pragma unroll
    for (int hs = 1; hs < kD; hs <<= 1)
#pragma unroll
      for (int i = 0; i < kD; ++i)
        if ((i & hs) == 0) {
          const float u = x[i], v = x[i + hs];
          x[i] = u + v;
          x[i + hs] = u - v;
        }
    // codes against the boundaries scaled to this vector (nu sqrt(128) b_j); the
    // residual in the unit domain, r = y / (nu sqrt(128)) - c[code], replaces y
    const float s = (nu > 0.f) ? nu * kSqrtD : 1.f;
    const float inv = (nu > 0.f) ? 1.f / (nu * kSqrtD) : 0.f;
    float P[H > 0 ? H : 1], CP[H + 1];
#pragma unroll
    for (int k = 0; k < H; ++k) P[k] = a.bounds[L / 2 + k] * s;
#pragma unroll
    for (int k = 0; k <= H; ++k) CP[k] = a.centroids[L / 2 + k];
#pragma unroll
    for (int w = 0; w < 4 * BITS; ++w) word[w] = 0u;
    rr = 0.f;
    mx = 0.f;
#pragma unroll
    for (int i = 0; i < kD; ++i) {
      const float y = x[i];
      const int m = count_pos<H>(fabsf(y), P);
      const int code = (y >= 0.f) ? (L / 2 + m) : (L / 2 - 1 - m);
      // slot order: coordinate i = 8n + 2t + e at code offset 32t + 2n + e
      const int n = i >> 3, tt = (i >> 1) & 3, e = i & 1;
      const int off = BITS * (32 * tt + 2 * n + e);
      word[off >> 5] |= (uint32_t)code << (off & 31);
      if ((off & 31) + BITS > 32) word[(off >> 5) + 1] |= (uint32_t)code >> (32 - (off & 31));
      float cm = CP[0];
#pragma unroll
      for (int k = 1; k <= H; ++k) cm = (m == k) ? CP[k] : cm;
      const float r = fmaf(y, inv, (y >= 0.f) ? -cm : cm);
      x[i] = r;
      rr = fmaf(r, r, rr);
      mx = fmaxf(mx, fabsf(r));
    }
}

// Rare path, entered by whole warps (tcgen05.ld is warp-collective): rebuild each
// thread's residual r = (hi + lo) / sc from the A operand still in TMEM and take
// its flagged signs from an fp32 S r. The rebuilt r agrees
// with the fp32 residual to about 2^-22 relative, so these signs can differ from
// an exact evaluation only where |z| is far below the coding tolerance.
__device__ __noinline__ void certify_signs(uint32_t tlane_a, float inv_sc, const float *sketch, uint32_t (&flag)[4],
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
              __half2float(__ushort_as_half((unsigned short)(lo[c] & 0xffffu)))) * inv_sc;
      r[k + 1] = (__half2float(__ushort_as_half((unsigned short)(hi[c] >> 16))) +
                  __half2float(__ushort_as_half((unsigned short)(lo[c] >> 16)))) * inv_sc;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    while (flag[q]) {
      const int bit = __ffs(flag[q]) - 1;
      flag[q] &= flag[q] - 1u;
      const float4 *row = reinterpret_cast<const float4 *>(sketch + (size_t)sketch_row(32 * q + bit) * kD);
      float zz = 0.f;
#pragma unroll
      for (int k = 0; k < kD / 4; ++k) {
        const float4 f = __ldg(row + k);
        zz = fmaf(f.x, r[4 * k], zz);
        zz = fmaf(f.y, r[4 * k + 1], zz);
        zz = fmaf(f.z, r[4 * k + 2], zz);
        zz = fmaf(f.w, r[4 * k + 3], zz);
      }
      sw[q] = (sw[q] & ~(1u << bit)) | ((zz >= 0.f ? 1u : 0u) << bit);
    }
  }
}

template <int BITS, bool BF16>
__global__ void __launch_bounds__(kQV, 2) append_qjl_kernel(const __grid_constant__ QjlArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *s_hi = smem, *s_lo = smem + kSBytes;
  uint64_t *s_bar = reinterpret_cast<uint64_t *>(smem + 2 * kSBytes);
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(smem + 2 * kSBytes + 8);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(s_bar, 1);
    mbar_fence_init();
    // B operand: S hi + lo, prepared once per context in the core-matrix layout
    mbar_arrive_expect_tx(s_bar, 2 * kSBytes);
    tma_load_1d(s_hi, a.sketch_hl, kSBytes, s_bar);
    tma_load_1d(s_lo, a.sketch_hl + kD * kD, kSBytes, s_bar);
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(smem_u32(s_taddr), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  bool bad = !mbar_wait_bounded(s_bar, 0, a.error);  // phase 0: the sketch copy
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *s_taddr;
  const float smax = a.sketch_rowmax;
  const uint32_t tlane = tbase + ((uint32_t)(warp * 32) << 16);  // this warp's TMEM lanes
  const uint32_t sa_hi = smem_u32(s_hi), sa_lo = smem_u32(s_lo);
  constexpr uint32_t idesc = tc_idesc_f16_f32(128, 128);

  const long long total = (long long)a.batch * a.heads * a.n_new;
  bad = __syncthreads_or(bad);
  int it = 1;  // mbarrier phase 0 was the sketch copy
  for (long long base = (long long)blockIdx.x * kQV; base < total; base += (long long)gridDim.x * kQV, ++it) {
    // ---------------- quantise: thread tid owns vector base + tid
    const long long vec = base + tid;
    long long slot = -1;
    if (vec < total) {
      const int t = (int)(vec % a.n_new);
      const long long bh = vec / a.n_new;
      const int b = (int)(bh / a.heads);
      const int len = __ldg(a.seq_lens + b);
      if (len >= 0 && len + a.n_new <= a.capacity) slot = bh * a.capacity + len + t;
      else if (t == 0) set_error(a.error, TQ_ERR_CAPACITY);  // the sequence is skipped whole
    }
    float x[kD];
    float nu, rr, mx;
    uint32_t word[4 * BITS];
    quantise_residual<BITS, BF16>(a, vec, slot >= 0, x, nu, rr, mx, word);
    if (slot >= 0) {
      uint4 *dst = reinterpret_cast<uint4 *>(a.codes + slot * (BITS * kD / 8));
#pragma unroll
      for (int k = 0; k < BITS; ++k)
        dst[k] = make_uint4(word[4 * k], word[4 * k + 1], word[4 * k + 2], word[4 * k + 3]);
      a.norms[slot] = nu;
    }

    // ---------------- A operand: r' = r 2^-floor(log2 max|r|) as fp16 hi + lo in TMEM
    __syncwarp();  // the TMEM moves below are warp-collective
    const float sc = (mx > 0.f) ? __int_as_float((254 - ((__float_as_int(mx) >> 23) & 0xff)) << 23) : 1.f;
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int chunk = 0; chunk < 2; ++chunk) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k = 2 * (32 * chunk + c);
          const float v0 = x[k] * sc, v1 = x[k + 1] * sc;
          const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
          __half o0 = h0, o1 = h1;
          if (part == 1) {
            o0 = __float2half_rn(v0 - __half2float(h0));
            o1 = __float2half_rn(v1 - __half2float(h1));
          }
          w[c] = (uint32_t)__half_as_ushort(o0) | ((uint32_t)__half_as_ushort(o1) << 16);
        }
        tmem_st_x32(tlane + 128 + 64 * part + 32 * chunk, w);
      }
    tc_fence_before_sync();
    __syncthreads();

    // ---------------- z' = S r' on the tensor cores: hi x hi + lo x hi + hi x lo
    if (tid == 0) {
      tc_fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t dh = tc_sdesc_kmajor(sa_hi + 256 * ks, 128, 2048);
        const uint64_t dl = tc_sdesc_kmajor(sa_lo + 256 * ks, 128, 2048);
        tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, dh, idesc, ks > 0);
        tc_mma_f16_ts(tbase, tbase + 192 + 8 * ks, dh, idesc, true);
        tc_mma_f16_ts(tbase, tbase + 128 + 8 * ks, dl, idesc, true);
      }
      tc_commit(smem_u32(s_bar));
    }
    if (!bad && !mbar_wait_bounded(s_bar, (uint32_t)(it & 1), a.error)) bad = true;
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
    tc_fence_after_sync();

    // ---------------- signs of this thread's row; certify those too close to zero
    const float E = 0x1p-16f * smax * sc * sqrtf(rr) + 0x1p-20f * smax;
    uint32_t sw[4], flag[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t z[32];
      tmem_ld_x32(tlane + 32 * q, z);
      uint32_t wv = 0u, fv = 0u;
#pragma unroll
      for (int bit = 0; bit < 32; ++bit) {
        const float zf = __uint_as_float(z[bit]);
        wv |= (zf >= 0.f ? 1u : 0u) << bit;
        fv |= (fabsf(zf) <= E ? 1u : 0u) << bit;
      }
      sw[q] = wv;
      flag[q] = fv;
    }
    // tcgen05.ld is warp-collective: the whole warp enters when any lane has a flag
    if (__any_sync(kFull, (flag[0] | flag[1] | flag[2] | flag[3]) != 0u)) {
      __syncwarp();
      certify_signs(tlane + 128, 1.f / sc, a.sketch, flag, sw);
    }
    if (slot >= 0) {
      float rho = nu * sqrtf(rr);
      if (nu == 0.f) {  // a zero vector: every sign set, rho = 0
        sw[0] = sw[1] = sw[2] = sw[3] = 0xffffffffu;
        rho = 0.f;
      }
      *reinterpret_cast<uint4 *>(a.signs + slot * (kD / 8)) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
      a.rnorms[slot] = rho;
    }
    // the next pass overwrites A and D only after every thread passed its barrier
    tc_fence_before_sync();
  }

  // ---------------- teardown: no tensor-core work in flight, then free TMEM
  if (bad) mbar_wait_bounded(s_bar, (uint32_t)(it & 1), a.error);  // bounded: give the MMAs a last chance
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// S -> fp16 hi + lo, row n of the operand = S row sketch_row(n), K-major core
// matrices: core (n / 8, k / 8) at byte 2048 (n / 8) + 128 (k / 8), row n % 8 at 16 (n % 8)
__global__ void __launch_bounds__(128) sketch_prep_kernel(DevParams *dp) {
  const int n = threadIdx.x;
  const float *row = dp->sketch + (size_t)sketch_row(n) * kD;
  unsigned char *hi = reinterpret_cast<unsigned char *>(dp->sketch_hl);
  unsigned char *lo = hi + kSBytes;
  for (int kb = 0; kb < kD / 8; ++kb) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float v0 = row[8 * kb + 2 * p], v1 = row[8 * kb + 2 * p + 1];
      const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
      const __half l0 = __float2half_rn(v0 - __half2float(h0)), l1 = __float2half_rn(v1 - __half2float(h1));
      h[p] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      l[p] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
    const int off = (n >> 3) * 2048 + kb * 128 + (n & 7) * 16;
    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

int g_sms_qjl = 0;

template <int BITS, bool BF16>
int go(const QjlArgs &k, long long total, cudaStream_t st) {
  if (g_sms_qjl == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_qjl, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms_qjl <= 0) g_sms_qjl = 152;
  }
  auto fn = append_qjl_kernel<BITS, BF16>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQjl) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  long long blocks = (total + kQV - 1) / kQV;
  const long long cap = 2LL * g_sms_qjl;  // persistent: two CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fn<<<(unsigned)blocks, kQV, kSmemQjl, st>>>(k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <bool BF16>
int dispatch(int bits, const QjlArgs &k, long long total, cudaStream_t st) {
  switch (bits) {
    case 1: return go<1, BF16>(k, total, st);
    case 2: return go<2, BF16>(k, total, st);
    case 3: return go<3, BF16>(k, total, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_sketch_prep(DevParams *dp, void *stream) {
  sketch_prep_kernel<<<1, kD, 0, (cudaStream_t)stream>>>(dp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Tensor-core append for sketched, rotated vectors; TQ_ERR_UNSUPPORTED otherwise.
int launch_append_qjl(const AppendArgs &a, const tq_ctx *ctx, void *stream) {
  if (!a.role.qjl || !a.role.rotate || a.role.bits < 1 || a.role.bits > 3) return TQ_ERR_UNSUPPORTED;
  QjlArgs k{};
  k.x = a.x;
  k.batch = a.batch;
  k.heads = a.heads;
  k.n_new = a.n_new;
  k.capacity = a.capacity;
  k.seq_lens = a.seq_lens;
  k.codes = a.codes;
  k.norms = a.norms;
  k.signs = a.signs;
  k.rnorms = a.rnorms;
  k.sketch = ctx->dparams->sketch;
  k.sketch_hl = ctx->dparams->sketch_hl;
  k.sketch_rowmax = ctx->sketch_rowmax;
  k.error = a.error;
  for (int i = 0; i < kD; ++i) k.diag[i] = (float)ctx->diag[i];
  const bool is_k = a.centroids == ctx->dparams->k_centroids;
  const float *bsrc = is_k ? ctx->k_bounds : ctx->v_bounds;
  const float *csrc = is_k ? ctx->k_centroids : ctx->v_centroids;
  for (int i = 0; i < (1 << a.role.bits) - 1; ++i) k.bounds[i] = bsrc[i];
  for (int i = 0; i < (1 << a.role.bits); ++i) k.centroids[i] = csrc[i];
  const long long total = (long long)a.batch * a.heads * a.n_new;
  cudaStream_t st = (cudaStream_t)stream;
  return a.dtype == TQ_BF16 ? dispatch<true>(a.role.bits, k, total, st) : dispatch<false>(a.role.bits, k, total, st);
}

}  // namespace tq
