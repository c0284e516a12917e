// Append-quantise of unrotated vectors (the KV scheme's keys and values) with one
// thread per vector.
//
// "Statistical Inference ... Inspired by TurboQuant", technical summary,
// "Quantisation schemes": the KV scheme codes each coordinate of the normalised
// vector with the Lloyd-Max codebook, without rotation; "KVQuant++", "Fast
// codebook lookup": the code is a boundary count, found by binary search.
//
// A thread holds its whole 128-coordinate vector in registers and does not divide
// it by its norm: it compares against its own scaled boundaries nu * b_j, which
// decides every code exactly as x / nu against b_j would. The boundaries are
// symmetric about 0, so a code is the sign of x plus a binary search of |x| over
// the positive boundaries. (Rotated roles take the tensor-core kernels.)

#include "tq_device.cuh"

namespace tq {
namespace {

struct Append2Args {
  const void *x;
  int batch, heads, n_new, capacity, cap16, bb;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  int vt;  // value role: codes in the pair-interleaved layout (merged atomically)
  const int32_t *seq_lens;
  uint8_t *codes;
  float *norms;
  int *error;
  // key side codes (side_rank > 0): plane base and bases [heads][d][rank] (natural order)
  int side_rank;
  uint16_t *side;
  const float *side_ur;
  float bounds[kMaxLevels];     // 2^BITS - 1 used
  float centroids[kMaxLevels];  // 2^BITS used (side codes)
};


// count of positive boundaries P[0..H-1] (ascending) at or below a >= 0
template <int H>
__device__ __forceinline__ int count_pos(float a, const float (&P)[H]) {
  if (H == 1) {
    return a >= P[0] ? 1 : 0;
  } else if (H == 3) {
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

template <int BITS, bool BF16>
__global__ void __launch_bounds__(128) append2_kernel(const __grid_constant__ Append2Args a) {
  constexpr int L = 1 << BITS, H = L / 2 - 1;
  const long long total = (long long)a.batch * a.heads * a.n_new;
  for (long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x; vec < total;
       vec += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(vec % a.n_new);
    const long long bh = vec / a.n_new;
    const int b = (int)(bh / a.heads);
    const int len = __ldg(a.seq_lens + b);
    const bool ok = len >= 0 && len + a.n_new <= a.capacity;  // a sequence that would not fit is skipped whole
    if (!ok) {
      if (t == 0) set_error(a.error, TQ_ERR_CAPACITY);
      continue;
    }
    const long long slot = phys_slot(a.btab, a.pool_blocks, bh * a.cap16 + len + t, a.error);
    if (slot < 0) continue;
    const int head = (int)(bh % a.heads);

    float x[kD];
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
    // squared norm by a pairwise tree (matches the warp design's rounding order closely)
    float sq[kD / 2];
#pragma unroll
    for (int i = 0; i < kD / 2; ++i) sq[i] = fmaf(x[2 * i], x[2 * i], x[2 * i + 1] * x[2 * i + 1]);
#pragma unroll
    for (int w = kD / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) sq[i] = sq[i] + sq[i + w];
    const float nu = sqrtf(sq[0]);

    // positive boundaries scaled to this vector: b_{L/2 + k} * nu; a zero vector keeps the
    // unit boundaries so that y = 0 codes to L/2 as the format requires
    const float s = (nu > 0.f) ? nu : 1.f;
    float P[H];
#pragma unroll
    for (int k = 0; k < H; ++k) P[k] = a.bounds[L / 2 + k] * s;

    // code i: sign half plus the count of positive boundaries below |y|; nu = 0 gives y = 0 -> L/2
    uint32_t word[4 * BITS];
#pragma unroll
    for (int w = 0; w < 4 * BITS; ++w) word[w] = 0u;
    // side code of an unsketched key: z_k = nu sum_i U[i][k] (x_i / nu - c[code_i])
    const int srank = a.side_rank;
    const float *su = srank ? a.side_ur + (size_t)head * kD * srank : nullptr;
    const float inv_nu = (nu > 0.f) ? 1.f / nu : 0.f;
    float zs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kD; ++i) {
      const float y = x[i];
      const int m = count_pos<H>(fabsf(y), P);
      const int code = (y >= 0.f) ? (L / 2 + m) : (L / 2 - 1 - m);
      if (srank) {
        const float r = fmaf(y, inv_nu, -a.centroids[code]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < srank) zs[k] = fmaf(__ldg(su + i * srank + k), r, zs[k]);
      }
      // slot order: coordinate i = 8n + 2t + e at code offset 32t + 2n + e
      const int n = i >> 3, tt = (i >> 1) & 3, e = i & 1;
      const int off = BITS * (32 * tt + 2 * n + e);
      word[off >> 5] |= (uint32_t)code << (off & 31);
      if ((off & 31) + BITS > 32) word[(off >> 5) + 1] |= (uint32_t)code >> (32 - (off & 31));
    }
    if (a.vt) {
      // this token's half of every field of its pair row: code offset n = 32 q + 2 m + e
      // holds coordinate 8 m + 2 q + e, whose field is vt_field() = 32 q + 16 e + m
      uint32_t *row = vt_row<BITS>(a.codes, slot, a.bb);
      const int half = (int)(slot & 1);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t cw[32], w[2 * BITS], ones[32], own[2 * BITS];
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          const int off = BITS * (32 * q + n);
          uint32_t v = word[off >> 5] >> (off & 31);
          if ((off & 31) + BITS > 32) v |= word[(off >> 5) + 1] << (32 - (off & 31));
          cw[n] = v & ((1u << BITS) - 1u);
          ones[n] = (1u << BITS) - 1u;
        }
        vt_spread<BITS>(cw, half, w);
        vt_spread<BITS>(ones, half, own);
#pragma unroll
        for (int i = 0; i < 2 * BITS; ++i) {
          atomicAnd(row + 2 * BITS * q + i, ~own[i]);
          atomicOr(row + 2 * BITS * q + i, w[i]);
        }
      }
    } else {
      uint4 *dst = reinterpret_cast<uint4 *>(rec_at(a.codes, slot, a.bb, BITS * kD / 8));
#pragma unroll
      for (int k = 0; k < BITS; ++k) dst[k] = make_uint4(word[4 * k], word[4 * k + 1], word[4 * k + 2], word[4 * k + 3]);
    }
    *rec_at(a.norms, slot, a.bb, 4) = nu;
    if (srank) {
      uint16_t *zp = rec_at(a.side, slot, a.bb, 2 * srank);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < srank) zp[k] = __half_as_ushort(__float2half_rn(zs[k] * nu));
    }
  }
}

int g_sms2 = 0;

template <int BITS, bool BF16>
int go(const Append2Args &k, long long total, cudaStream_t st) {
  if (g_sms2 == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms2, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms2 <= 0) g_sms2 = 152;
  }
  long long blocks = (total + 127) / 128;
  const long long cap = 4LL * g_sms2;  // enough resident threads to cover memory latency
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  append2_kernel<BITS, BF16><<<(unsigned)blocks, 128, 0, st>>>(k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <bool BF16>
int dispatch(int bits, const Append2Args &k, long long total, cudaStream_t st) {
  switch (bits) {
    case 2: return go<2, BF16>(k, total, st);
    case 3: return go<3, BF16>(k, total, st);
    case 4: return go<4, BF16>(k, total, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

}  // namespace

// Thread-per-vector append for vectors without a sketch; TQ_ERR_UNSUPPORTED otherwise.
int launch_append2(const AppendArgs &a, const tq_ctx *ctx, void *stream) {
  if (a.role.qjl || a.role.rotate || a.role.bits < 2) return TQ_ERR_UNSUPPORTED;
  Append2Args k{};
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
  k.error = a.error;
  const bool is_k = a.centroids == ctx->dparams->k_centroids;
  const float *src = is_k ? ctx->k_bounds : ctx->v_bounds;
  const float *csrc = is_k ? ctx->k_centroids : ctx->v_centroids;
  for (int i = 0; i < (1 << a.role.bits) - 1; ++i) k.bounds[i] = src[i];
  for (int i = 0; i < (1 << a.role.bits); ++i) k.centroids[i] = csrc[i];
  k.side_rank = a.side_rank;
  k.side = a.side;
  k.side_ur = a.side_ur;
  const long long total = (long long)a.batch * a.heads * a.n_new;
  cudaStream_t st = (cudaStream_t)stream;
  const bool bf16 = a.dtype == TQ_BF16;
  return bf16 ? dispatch<true>(a.role.bits, k, total, st) : dispatch<false>(a.role.bits, k, total, st);
}

}  // namespace tq
