// Append-quantise of unrotated vectors (the KV scheme's keys and values), one warp per two
// token pairs.
//
// "Statistical Inference ... Inspired by TurboQuant", technical summary,
// "Quantisation schemes": the KV scheme codes each coordinate of the normalised
// vector with the Lloyd-Max codebook, without rotation; "KVQuant++", "Fast
// codebook lookup": the code is a boundary count, found by binary search.
//
// A warp takes two consecutive stored pairs of a sequence-head (slots 2j and 2j + 1 are the
// unit the value layout interleaves) and the tokens of them that this append writes; lane L
// holds coordinates 4L..4L+3 of each, every row loaded (coalesced) before any is coded. The
// vector is not divided by its norm: each coordinate is compared against the scaled
// boundaries nu * b_j, which decides every code exactly as x / nu against b_j would. The
// boundaries are symmetric about 0, so a code is the sign of x plus a binary search of |x|
// over the positive boundaries. Key records and value rows are assembled from the lanes'
// codes by shuffles and written as whole words; a value row whose other token is not part of
// this append keeps that token's bits (the warp is the row's only writer in the launch).
// (Rotated roles take the tensor-core kernels.)

#include "tq_device.cuh"

namespace tq {
namespace {

struct Append2Args {
  const void *x;
  int batch, heads, n_new, capacity, cap16, bb;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  int vt;  // value role: codes in the pair-interleaved layout
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
  FastDiv div_pairs, div_heads;  // by the warps (groups of token pairs) per sequence-head, and by heads
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

// the bits of word `lane` of a pair row that belong to token half h (VB ones per field)
template <int VB>
__device__ __forceinline__ uint32_t vt_row_half_mask(int h, int lane) {
  constexpr int F = 2 * VB;
  constexpr int K = (32 + F - 1) / F + 1;
  const int first = (32 * lane) / F;
  const uint32_t f = ((1u << VB) - 1u) << (VB * h);
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const int o = first + i;
    const int shift = F * o - 32 * lane;
    if (o < 128 && shift > -F && shift < 32) word |= (shift >= 0) ? (f << shift) : (f >> (-shift));
  }
  return word;
}

// kPairs consecutive pairs of one sequence-head per warp, all rows loaded before any is coded
constexpr int kPairs = 2;

// Records and pair rows are assembled from the lanes' codes by shuffles. Every lane packs its
// two pair fields (key records: pair 2L low, pair 2L + 1 high) or its four coordinate fields
// (value rows: coordinate 4L + k at field k) into one word, 2 BITS bits a field. Key record
// slot s (pair p = 4n + t at slot 16t + n) is lane 2 (s mod 16) + (s / 32) mod 2's field
// (s / 16) mod 2; value row field o = vt_field(c) is lane 2 (o mod 16) + o / 64's field
// (o / 16) mod 4. When a field's 2 BITS bits divide 32 (BITS = 2, 4), a word holds
// n = 16 / BITS whole fields, all at one position of their lanes, from n lanes two apart, so
// each field costs a shuffle, a shift and an add.
// Key record word w (lanes < 4 BITS): slots n w + i, i < n.
template <int BITS>
__device__ __forceinline__ uint32_t key_word_even(uint32_t both, int lane) {
  constexpr int F = 2 * BITS, N = 32 / F;
  const int s = N * lane;
  const int src = 2 * (s & 15) + ((s >> 5) & 1);
  const int sh = F * ((s >> 4) & 1);
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t v = __shfl_sync(kFull, both, (src + 2 * i) & 31);
    word += ((v >> sh) & ((1u << F) - 1u)) << (F * i);
  }
  return word;
}
// Value row word w (lanes < 8 BITS): fields o = n w + i, from lane 2 (o mod 16) + o / 64,
// position (o / 16) mod 4 of that lane's four fields.
template <int BITS>
__device__ __forceinline__ uint32_t vt_word_even(uint32_t both, int lane) {
  constexpr int F = 2 * BITS, N = 32 / F;
  const int o = N * lane;
  const int src = 2 * (o & 15) + ((o >> 6) & 1);
  const int sh = F * ((o >> 4) & 3);
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t v = __shfl_sync(kFull, both, (src + 2 * i) & 31);
    word += ((v >> sh) & ((1u << F) - 1u)) << (F * i);
  }
  return word;
}

// 3-bit codes (6-bit fields): 16 consecutive fields fill exactly three words, so word j of such
// a group takes fields i0 = 32 j / 6 .. i0 + 5 (from lanes src0 + 2 i, at shift sh of their
// packed fields), gathered in 64 bits and shifted right by 32 j - 6 i0.
__device__ __forceinline__ uint32_t word6(uint32_t both, int src0, int sh, int j) {
  const int i0 = (32 * j) / 6;
  uint64_t acc = 0;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const uint32_t v = __shfl_sync(kFull, both, (src0 + 2 * (i0 + k)) & 31);
    acc |= (uint64_t)((v >> sh) & 63u) << (6 * k);
  }
  return (uint32_t)(acc >> (32 * j - 6 * i0));
}
// key record word w (lanes < 12): group G = w / 3 of 16 slots (a fields of even lanes, b of
// even, a of odd, b of odd)
__device__ __forceinline__ uint32_t key_word6(uint32_t both, int lane) {
  const int G = lane / 3, j = lane - 3 * (lane / 3);
  return word6(both, (G >> 1) & 1, 6 * (G & 1), j);
}
// value row word w (lanes < 24): fields o = 16 m + i, m = w / 3, from lanes 2 i + m / 4,
// position m mod 4
__device__ __forceinline__ uint32_t vt_word6(uint32_t both, int lane) {
  const int m = lane / 3, j = lane - 3 * (lane / 3);
  return word6(both, (m >> 2) & 1, 6 * (m & 3), j);
}

template <int BITS, bool BF16>
__global__ void __launch_bounds__(256) append2_kernel(const __grid_constant__ Append2Args a) {
  constexpr int L = 1 << BITS, H = L / 2 - 1;
  const int lane = threadIdx.x & 31;
  const uint32_t unit = blockIdx.x * 8u + (threadIdx.x >> 5);
  const uint32_t bh = fast_div(unit, a.div_pairs);
  if (bh >= (uint32_t)(a.batch * a.heads)) return;
  const uint32_t b = fast_div(bh, a.div_heads);
  const int head = (int)(bh - b * (uint32_t)a.heads);
  const int group = (int)(unit - bh * a.div_pairs.d);
  const int len = __ldg(a.seq_lens + b);
  if (len < 0 || len + a.n_new > a.capacity) {  // a sequence that would not fit is skipped whole
    if (group == 0 && lane == 0) set_error(a.error, TQ_ERR_CAPACITY);
    return;
  }
  // the group's slots from s0 = (len rounded down to even) + 2 kPairs group; the append
  // writes slots [len, len + n_new)
  const int s0 = (len & ~1) + 2 * kPairs * group;
  const int s_end = len + a.n_new;
  if (s0 >= s_end) return;
  float x[2 * kPairs][4];
#pragma unroll
  for (int i = 0; i < 2 * kPairs; ++i) {
    const int s = s0 + i;
    const long long t = (long long)bh * a.n_new + (s - len);  // input row
    if (s >= len && s < s_end) {
      if (BF16) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.x) + t * kD) + lane);
        x[i][0] = __uint_as_float(w.x << 16);
        x[i][1] = __uint_as_float(w.x & 0xffff0000u);
        x[i][2] = __uint_as_float(w.y << 16);
        x[i][3] = __uint_as_float(w.y & 0xffff0000u);
      } else {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + t * kD) + lane);
        x[i][0] = f.x;
        x[i][1] = f.y;
        x[i][2] = f.z;
        x[i][3] = f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) x[i][j] = 0.f;
    }
  }
#pragma unroll
  for (int p = 0; p < kPairs; ++p) {
    const int sp = s0 + 2 * p;
    if (sp >= s_end) break;  // warp-uniform
    const long long vs = (long long)bh * a.cap16 + sp;
    long long slot[2];
    int code[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool has = sp + h >= len && sp + h < s_end;
      slot[h] = has ? phys_slot(a.btab, a.pool_blocks, vs + h, a.error) : -1;
      const float (&xv)[4] = x[2 * p + h];
      const float nu = sqrtf(warp_sum(xv[0] * xv[0] + xv[1] * xv[1] + xv[2] * xv[2] + xv[3] * xv[3]));
      // positive boundaries scaled to this vector: b_{L/2 + k} * nu; a zero vector keeps the
      // unit boundaries so that x = 0 codes to L/2 as the format requires
      const float sc = (nu > 0.f) ? nu : 1.f;
      float P[H];
#pragma unroll
      for (int k = 0; k < H; ++k) P[k] = a.bounds[L / 2 + k] * sc;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y = xv[j];
        const int m = count_pos<H>(fabsf(y), P);
        code[h][j] = (y >= 0.f) ? (L / 2 + m) : (L / 2 - 1 - m);
      }
      if (!a.vt) {  // key record of this token
        const uint32_t fa = (uint32_t)code[h][0] | ((uint32_t)code[h][1] << BITS);
        const uint32_t fb = (uint32_t)code[h][2] | ((uint32_t)code[h][3] << BITS);
        uint32_t word;  // every lane takes part
        if constexpr (32 % (2 * BITS) == 0) word = key_word_even<BITS>(fa | (fb << (2 * BITS)), lane);
        else word = key_word6(fa | (fb << (2 * BITS)), lane);
        if (slot[h] >= 0 && lane < 4 * BITS)
          reinterpret_cast<uint32_t *>(rec_at(a.codes, slot[h], a.bb, BITS * kD / 8))[lane] = word;
      }
      if (slot[h] >= 0 && lane == 0) *rec_at(a.norms, slot[h], a.bb, 4) = nu;
      if (a.side_rank) {  // warp-uniform
        const float inv_nu = (nu > 0.f) ? 1.f / nu : 0.f;
        float r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = fmaf(xv[j], inv_nu, -a.centroids[code[h][j]]);
        side_code_warp(a.side_ur + (size_t)head * kD * a.side_rank, a.side_rank, nu, r, a.side, slot[h], a.bb, lane);
      }
    }
    if (a.vt) {
      // the pair row: both tokens' codes, this lane's four fields packed
      uint32_t both = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        both |= ((uint32_t)code[0][j] | ((uint32_t)code[1][j] << BITS)) << (2 * BITS * j);
      uint32_t word;  // every lane takes part
      if constexpr (32 % (2 * BITS) == 0) word = vt_word_even<BITS>(both, lane);
      else word = vt_word6(both, lane);
      const long long any = slot[0] >= 0 ? slot[0] : slot[1];
      if (any >= 0 && lane < 8 * BITS) {
        uint32_t *row = vt_row<BITS>(a.codes, any, a.bb);
        if (slot[0] >= 0 && slot[1] >= 0) {
          row[lane] = word;
        } else {  // one token of the pair: keep the other token's bits
          const uint32_t mine = vt_row_half_mask<BITS>(slot[0] >= 0 ? 0 : 1, lane);
          row[lane] = (row[lane] & ~mine) | (word & mine);
        }
      }
    }
  }
}

template <int BITS, bool BF16>
int go(const Append2Args &k, long long warps, cudaStream_t st) {
  append2_kernel<BITS, BF16><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(k);
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

// Warp-per-pair append for unrotated vectors without a sketch; TQ_ERR_UNSUPPORTED otherwise.
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
  // pairs of slots touched per sequence-head: [len rounded down to even, len + n_new), in
  // groups of kPairs per warp
  const int pairs = a.n_new / 2 + 1;
  const int groups = (pairs + kPairs - 1) / kPairs;
  const long long warps = (long long)a.batch * a.heads * groups;
  if (warps >= 0xffffffffLL - 8) return TQ_ERR_ARG;  // warp indices are 32-bit
  k.div_pairs = make_fastdiv((uint32_t)groups);
  k.div_heads = make_fastdiv((uint32_t)a.heads);
  cudaStream_t st = (cudaStream_t)stream;
  const bool bf16 = a.dtype == TQ_BF16;
  return bf16 ? dispatch<true>(a.role.bits, k, warps, st) : dispatch<false>(a.role.bits, k, warps, st);
}

}  // namespace tq
