// Low-latency append for calls that quantise few vectors (a decode step appends
// one token per sequence and head): one warp per vector, keys and values of the
// call in a single launch (blockIdx.y is the role), nothing staged per block.
//
// "Statistical Inference and Quality Measures of KV Cache Quantisations
// Inspired by TurboQuant", technical summary, "Quantisation schemes" (norm,
// seeded +/-1 diagonal and Walsh-Hadamard rotation, scalar Lloyd-Max codes;
// the (n-1)-bit vectors keep a 1-bit QJL sketch of their residual) and "Main
// contribution 1" (the sketch stores sign(S r) and rho = ||x|| ||r||).
// "KVQuant++", "Fast codebook lookup": a code is the count of boundaries at or
// below the coordinate.
//
// Lane L holds coordinates 4L..4L+3. The rotation is the warp's in-register /
// shuffle WHT; codes are counted against the context's boundaries. For
// sketched vectors a transposed, permuted copy of S (prepared once per
// context; column 4L + m is the sketch row whose sign is bit L of sign word m)
// is bulk-copied into shared memory while the vectors are coded, and the
// block's threads then form S r for all of its vectors at once, each S entry
// read from shared memory once per half-warp and used for four vectors.

#include "tq_device.cuh"
#include "tq_ptx.cuh"

namespace tq {
namespace {

constexpr int kSmallWarps = 8;  // vectors per block
// S^T, residuals, sign words, mbarrier
constexpr int kRS = kD + 4;  // residual row stride (floats): the two vector groups of a warp hit different banks
constexpr size_t kSmallSmem = sizeof(float) * (kD * kD + kSmallWarps * kRS) + sizeof(uint32_t) * kSmallWarps * 4 + 16;

struct SmallRole {
  const void *x;  // [batch][heads][n_new][d]
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  int bits, rotate, qjl, vt;
  float bounds[kMaxLevels];  // 2^bits - 1 used, +inf after
  float centroids[kMaxLevels];
};

struct SmallArgs {
  SmallRole role[2];  // keys, values (plane bases in the blocked records)
  int batch, heads, n_new, capacity, cap16, bb;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  const int32_t *seq_lens;
  const float *diag;       // D as +/-1.0f
  const float *rot_t;      // dense rotation M^T, or nullptr (Walsh-Hadamard)
  uint16_t *k_side;        // key side codes (side_rank > 0): plane base, bases [heads][d][rank]
  const float *side_ur;
  int side_rank;
  const float *sketch_tp;  // entry (i, 4L + m) = S[8(L/2) + 2m + (L&1)][i]
  int *error;
};

template <bool BF16>
__global__ void __launch_bounds__(kSmallWarps * 32, 1) append_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  float *s_st = reinterpret_cast<float *>(smem);            // S^T, permuted [128][128] (sketched role)
  float *s_r = s_st + kD * kD;                               // residuals [vector][kRS]
  uint32_t *s_sw = reinterpret_cast<uint32_t *>(s_r + kSmallWarps * kRS);  // sign words [vector][4]
  uint64_t *s_bar = reinterpret_cast<uint64_t *>(s_sw + kSmallWarps * 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SmallRole &ro = a.role[blockIdx.y];
  const bool qjl = ro.qjl != 0;  // block-uniform
  if (qjl) {
    // S^T streams in while the vectors are normalised, rotated and coded
    if (tid == 0) {
      mbar_init(s_bar, 1);
      mbar_fence_init();
      mbar_arrive_expect_tx(s_bar, kD * kD * sizeof(float));
      tma_load_1d(s_st, a.sketch_tp, kD * kD * sizeof(float), s_bar);
    }
    if (tid < kSmallWarps * 4) s_sw[tid] = 0u;
  }
  // the inputs and the cache may be written by the kernel before (a launch with programmatic
  // serialization starts before it ends); everything above reads context constants only
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)a.batch * a.heads * a.n_new;
  const long long vec = (long long)blockIdx.x * kSmallWarps + warp;
  const bool live = vec < total;  // warp-uniform

  long long slot = -1;
  float nu = 0.f, rr = 0.f;
  if (live) {
    const int t = (int)(vec % a.n_new);
    const long long bh = vec / a.n_new;
    const int b = (int)(bh / a.heads);
    const int len = __ldg(a.seq_lens + b);
    // a sequence whose new tokens would not all fit is skipped whole
    const bool ok = len >= 0 && len + a.n_new <= a.capacity;
    if (!ok && t == 0 && lane == 0 && blockIdx.y == 0) set_error(a.error, TQ_ERR_CAPACITY);
    slot = ok ? phys_slot(a.btab, a.pool_blocks, bh * a.cap16 + len + t, a.error) : -1;

    float x[4];
    load4(ro.x, (size_t)vec * kD + 4 * lane, BF16, x);
    float r[4];
    const bool side = a.side_rank > 0 && blockIdx.y == 0;  // keys with side codes
    encode_vector_warp_general(ro, x, slot, a.bb, a.diag, lane, nu, r, rr, a.rot_t, side);
    if (side)
      side_code_warp(a.side_ur + (size_t)(bh % a.heads) * kD * a.side_rank, a.side_rank, nu, r, a.k_side, slot,
                     a.bb, lane);
    if (qjl) reinterpret_cast<float4 *>(s_r + warp * kRS)[lane] = make_float4(r[0], r[1], r[2], r[3]);
  } else if (qjl) {
    reinterpret_cast<float4 *>(s_r + warp * kRS)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (!qjl) return;

  // z = S r for the block's vectors, S read once per block: thread (warp w, lane l) forms
  // sketch column c = 16 w + (l & 15) (the row whose sign is bit c / 4 of word c % 4) for
  // vectors 4 (l >> 4) .. 4 (l >> 4) + 3, summing over i in order
  __syncthreads();
  const bool have_s = mbar_wait_bounded(s_bar, 0, a.error);
  const int c = 16 * warp + (lane & 15), v0 = 4 * (lane >> 4);
  float z[4] = {0.f, 0.f, 0.f, 0.f};
  if (have_s) {
#pragma unroll 4
    for (int i4 = 0; i4 < kD / 4; ++i4) {
      float4 rv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) rv[k] = reinterpret_cast<const float4 *>(s_r + (v0 + k) * kRS)[i4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float sv = s_st[(4 * i4 + ii) * kD + c];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float ri = ii == 0 ? rv[k].x : ii == 1 ? rv[k].y : ii == 2 ? rv[k].z : rv[k].w;
          z[k] = fmaf(sv, ri, z[k]);
        }
      }
    }
  }
  // bit t of a half-warp's ballot is column 16 w + t = sign bit 4 w + t / 4 of word t % 4
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t bal = __ballot_sync(kFull, z[k] >= 0.f);
    if (lane < 8) {
      const int h = lane >> 2, m = lane & 3;
      const uint32_t x = bal >> (16 * h);
      const uint32_t nib = ((x >> m) & 1u) | ((x >> (m + 3)) & 2u) | ((x >> (m + 6)) & 4u) | ((x >> (m + 9)) & 8u);
      atomicOr(&s_sw[(4 * h + k) * 4 + m], nib << (4 * warp));
    }
  }
  __syncthreads();
  if (slot < 0) return;
  float rho = nu * sqrtf(rr);
  uint32_t w = s_sw[warp * 4 + (lane & 3)];
  if (nu == 0.f) {  // a zero vector: every sign set, rho = 0
    w = 0xffffffffu;
    rho = 0.f;
  }
  if (lane < 4) reinterpret_cast<uint32_t *>(rec_at(ro.signs, slot, a.bb, kD / 8))[lane] = w;
  if (lane == 0) {
    *rec_at(ro.norms, slot, a.bb, 4) = nu;
    *rec_at(ro.rnorms, slot, a.bb, 4) = rho;
  }
}

void fill_role(SmallRole &r, const Role &role, const float *bounds, const float *centroids) {
  r.bits = role.bits;
  r.rotate = role.rotate ? 1 : 0;
  r.qjl = role.qjl ? 1 : 0;
  const int L = 1 << role.bits;
  for (int i = 0; i < kMaxLevels; ++i) {
    r.bounds[i] = (i < L - 1) ? bounds[i] : __builtin_huge_valf();
    r.centroids[i] = (i < L) ? centroids[i] : 0.f;
  }
}

__global__ void sketch_transpose_kernel(DevParams *dp) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < kD * kD; e += gridDim.x * blockDim.x) {
    const int i = e >> 7, col = e & 127, l = col >> 2, m = col & 3;
    dp->sketch_tp[e] = dp->sketch[(8 * (l >> 1) + 2 * m + (l & 1)) * kD + i];
  }
}

}  // namespace

int launch_sketch_transpose(DevParams *dp, void *stream) {
  sketch_transpose_kernel<<<16, 256, 0, (cudaStream_t)stream>>>(dp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

bool append_small_fits(const tq_ctx *ctx, long long vectors) {
  return vectors > 0 && vectors <= kSmallAppendMax && ctx->k.bits >= 1 && ctx->k.bits <= 4 && ctx->v.bits >= 1 &&
         ctx->v.bits <= 4;
}

int launch_append_small(const AppendArgs &k, const AppendArgs &v, const tq_ctx *ctx, void *stream) {
  SmallArgs s{};
  const AppendArgs *src[2] = {&k, &v};
  for (int r = 0; r < 2; ++r) {
    const AppendArgs &x = *src[r];
    SmallRole &o = s.role[r];
    o.x = x.x;
    o.codes = x.codes;
    o.norms = x.norms;
    o.signs = x.signs;
    o.rnorms = x.rnorms;
    o.vt = x.vt;
    fill_role(o, x.role, r == 0 ? ctx->k_bounds : ctx->v_bounds, r == 0 ? ctx->k_centroids : ctx->v_centroids);
  }
  s.batch = k.batch;
  s.heads = k.heads;
  s.n_new = k.n_new;
  s.capacity = k.capacity;
  s.cap16 = k.cap16;
  s.bb = k.bb;
  s.btab = k.btab;
  s.pool_blocks = k.pool_blocks;
  s.seq_lens = k.seq_lens;
  s.diag = ctx->dparams->diag;
  s.rot_t = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot_t : nullptr;
  s.k_side = k.side;
  s.side_ur = k.side_ur;
  s.side_rank = k.side_rank;
  s.sketch_tp = ctx->dparams->sketch_tp;
  s.error = k.error;
  const long long total = (long long)k.batch * k.heads * k.n_new;
  if (!append_small_fits(ctx, total)) return TQ_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)((total + kSmallWarps - 1) / kSmallWarps), 2);
  cudaStream_t st = (cudaStream_t)stream;
  auto fn = k.dtype == TQ_BF16 ? append_small_kernel<true> : append_small_kernel<false>;
  static bool attr_done[2] = {false, false};
  bool &done = attr_done[k.dtype == TQ_BF16 ? 1 : 0];
  if (!done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallSmem) != cudaSuccess)
      return TQ_ERR_CUDA;
    done = true;
  }
  return launch_overlapped(true, fn, grid, dim3(kSmallWarps * 32), kSmallSmem, st, s) == cudaSuccess ? TQ_OK
                                                                                                 : TQ_ERR_CUDA;
}

}  // namespace tq
