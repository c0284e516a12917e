// Decode attention read straight from the compressed cache.
//
//   o = softmax(q K_hat^T / sqrt(d)) V_hat
// with K_hat and V_hat never materialised: keys are read through logits
// ("HeadQ", 2.1: a key enters attention only through q^T k / sqrt(d)) and
// values through the p-weighted sum, which is linear ("HeadQ", 2.2; "Statistical
// Inference ... Inspired by TurboQuant", technical summary, "K-V asymmetry").
// Linearity lets the value side stay in the rotated, unit-codebook domain:
//   sum_j p_j v_hat_j = D H ( sum_j p_j nu_j c[idx_j]
//                             + sqrt(pi/2)/m S^T sum_j p_j rho_j sigma_j ),
// so each head needs one S^T matvec and one inverse WHT after the token loop.
// For sketched keys (QKQV) the score adds the QJL correction
//   rho_j sqrt(pi/2)/m <S q_rot, sigma_j>  ("Main contribution 1").
//
// Three launches, stream-ordered:
//   qprep   -- q_rot = H D q / sqrt(d) (and S q_rot for sketched keys)
//   decode  -- one CTA per (batch, kv head, token chunk): online softmax over
//              the chunk, partial (m, l, sum p nu c, sum p rho sigma)
//   combine -- merge the chunks of each query head, S^T, inverse WHT.

#include <cuda_fp16.h>

#include <type_traits>

#include "tq_device.cuh"
#include "tq_ptx.cuh"

namespace tq {
namespace {

constexpr int kDecodeWarps = 4;
constexpr int kTile = 8;  // tokens per warp step

struct PrepArgs {
  const void *q;
  int bf16, batch, heads_q, rotate, sketch_k;
  const float *diag;
  const float *sketch;
  float *qprep;  // [batch*heads_q][2][128]
  // optional: tiles of kDecodeTile tokens before each batch, [batch + 1]
  const int32_t *seq_lens;
  int capacity;
  int32_t *tile_prefix;
  const float *rot_t = nullptr;  // dense rotation M^T (q_rot = M q), or nullptr (Walsh-Hadamard)
  // key side codes: w = U_rot^T q_rot / sqrt(d) for the row's KV head (rows / heads_q / G),
  // written to the second half of the row's record (unsketched keys leave it free)
  const float *side_ur = nullptr;
  int side_rank = 0, group = 1;
  // S transposed and permuted: entry (i, 4L + m) = S[8 (L / 2) + 2 m + (L & 1)][i], so that
  // lane L reads its four sketch rows' column i as one coalesced float4
  const float *sketch_tp = nullptr;
};

// Exclusive prefix over batches of ceil(clamped length / kDecodeTile), by one
// block of 128 threads (any batch count: chunks of 128 with a running carry).
__device__ void tile_prefix_block(const PrepArgs &a) {
  __shared__ int s_scan[128];
  __shared__ int s_carry;
  const int t = threadIdx.x;
  if (t == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < a.batch; base += 128) {
    const int b = base + t;
    const int len = (b < a.batch) ? min(max(__ldg(a.seq_lens + b), 0), a.capacity) : 0;
    const int n = (len + kDecodeTile - 1) / kDecodeTile;
    s_scan[t] = n;
    __syncthreads();
    for (int o = 1; o < 128; o <<= 1) {  // inclusive Hillis-Steele scan
      const int v = (t >= o) ? s_scan[t - o] : 0;
      __syncthreads();
      s_scan[t] += v;
      __syncthreads();
    }
    const int carry = s_carry;
    if (b < a.batch) a.tile_prefix[b] = carry + s_scan[t] - n;
    __syncthreads();
    if (t == 127) s_carry = carry + s_scan[127];
    __syncthreads();
  }
  if (t == 0) a.tile_prefix[a.batch] = s_carry;
}

// one warp per (batch, query head)
__global__ void __launch_bounds__(128) qprep_kernel(PrepArgs a) {
  __shared__ float s_q[4][kD];
  pdl_trigger();  // the decode kernel may start its prologue now
  pdl_wait();     // the queries and lengths may come from the kernel before (e.g. the step's append)
  if (a.tile_prefix && blockIdx.x == 0) tile_prefix_block(a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  const bool live = row < a.batch * a.heads_q;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (live) load4(a.q, (size_t)row * kD + 4 * lane, a.bf16 != 0, v);
  if (a.rotate && a.rot_t) {
    matvec_t_warp(a.rot_t, v, lane);
  } else if (a.rotate) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= __ldg(a.diag + 4 * lane + j);
    wht128(v, lane);
  }
  if (live) {
    float4 o = make_float4(v[0] * kInvSqrtD, v[1] * kInvSqrtD, v[2] * kInvSqrtD, v[3] * kInvSqrtD);
    reinterpret_cast<float4 *>(a.qprep + (size_t)row * 2 * kD)[lane] = o;
  }
  if (a.side_rank && live) {  // warp-uniform
    const int hk = (row % a.heads_q) / a.group;
    const float *U = a.side_ur + (size_t)hk * kD * a.side_rank;
    for (int k = 0; k < a.side_rank; ++k) {
      float p = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) p = fmaf(__ldg(U + (4 * lane + j) * a.side_rank + k), v[j], p);
      p = warp_sum(p);
      if (lane == 0) a.qprep[(size_t)row * 2 * kD + kD + k] = p * kInvSqrtD;
    }
  }
  if (!a.sketch_k) return;  // (uniform over the grid)
#pragma unroll
  for (int j = 0; j < 4; ++j) s_q[warp][4 * lane + j] = v[j];
  __syncthreads();
  // (S q_rot)_k for the four sketch rows k = 8 (lane / 2) + 2 m + (lane & 1) of the block's four
  // query rows: warp w sums columns i in [32 w, 32 w + 32), each column read from the transposed
  // copy in one coalesced 512-byte line, and the four warps' partial sums meet in shared memory
  // (a warp streaming all 128 lines for one row kept too few loads in flight)
  __shared__ __align__(16) float s_part[4][4][kD];  // [warp][row][lane-ordered outputs]
  float acc[4][4] = {};
#pragma unroll 8
  for (int ii = 0; ii < 32; ++ii) {
    const int i = 32 * warp + ii;
    const float4 s4 = __ldg(reinterpret_cast<const float4 *>(a.sketch_tp + (size_t)i * kD) + lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float qi = s_q[r][i];
      acc[r][0] = fmaf(s4.x, qi, acc[r][0]);
      acc[r][1] = fmaf(s4.y, qi, acc[r][1]);
      acc[r][2] = fmaf(s4.z, qi, acc[r][2]);
      acc[r][3] = fmaf(s4.w, qi, acc[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
    reinterpret_cast<float4 *>(s_part[warp][r])[lane] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  __syncthreads();
  if (live) {  // warp w finishes row w of the block
    const float c = kSqrtHalfPi / kD * kInvSqrtD;
    float4 t = reinterpret_cast<const float4 *>(s_part[0][warp])[lane];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      const float4 u = reinterpret_cast<const float4 *>(s_part[w][warp])[lane];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float o[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int m = 0; m < 4; ++m)
      a.qprep[(size_t)row * 2 * kD + kD + 8 * (lane >> 1) + 2 * m + (lane & 1)] = o[m] * c;
  }
}

struct DecodeKernelArgs {
  const uint8_t *k_codes;
  const float *k_norm;
  const uint8_t *k_signs;
  const float *k_rnorm;
  const uint8_t *v_codes;
  const float *v_norm;
  const uint8_t *v_signs;
  const float *v_rnorm;
  int bb, cap16;  // blocked records (plane pointers are the block-0 bases)
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  int *error;
  int capacity, heads_kv, heads_q, chunk, splits;
  const int32_t *seq_lens;
  const float *qprep;
  float *partials;
  const float *k_centroids;
  const float *v_centroids;
  const uint16_t *k_side;  // key side codes (side_rank > 0): plane base
  int side_rank;
};

// lane -> token (0..7) after the 8-way reduce-scatter below, and back
__device__ __forceinline__ int tile_token_of_lane(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}
__device__ __forceinline__ int lane_of_tile_token(int jj) {
  return ((jj >> 2) & 1) * 16 + ((jj >> 1) & 1) * 8 + (jj & 1) * 4;
}

// Sum eight per-lane partials over the warp; lane ends with the sum for token
// tile_token_of_lane(lane). 9 shuffles instead of 40 for eight full reductions.
__device__ __forceinline__ float reduce8(const float (&p)[kTile], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float k1[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = b4 ? p[k] : p[k + 4];
    const float keep = b4 ? p[k + 4] : p[k];
    k1[k] = keep + __shfl_xor_sync(kFull, send, 16);
  }
  float k2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = b3 ? k1[k] : k1[k + 2];
    const float keep = b3 ? k1[k + 2] : k1[k];
    k2[k] = keep + __shfl_xor_sync(kFull, send, 8);
  }
  const float send = b2 ? k2[0] : k2[1];
  float s = (b2 ? k2[1] : k2[0]) + __shfl_xor_sync(kFull, send, 4);
  s += __shfl_xor_sync(kFull, s, 2);
  s += __shfl_xor_sync(kFull, s, 1);
  return s;
}

template <int KB, int VB, bool KQJL, bool VQJL, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_tq_kernel(DecodeKernelArgs a) {
  __shared__ float s_cb[32];  // [0,16) K centroids, [16,32) V centroids
  __shared__ float s_m[kDecodeWarps][G], s_l[kDecodeWarps][G];
  __shared__ float s_acc[kDecodeWarps][G][kD];
  __shared__ float s_sacc[VQJL ? kDecodeWarps : 1][G][VQJL ? kD : 1];

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 16) s_cb[tid] = a.k_centroids[tid];
  else if (tid < 32) s_cb[tid] = a.v_centroids[tid - 16];

  const int len = min(max(__ldg(a.seq_lens + b), 0), a.capacity);
  const int t_begin = split * a.chunk;
  const int t_end = min(t_begin + a.chunk, len);

  float qv[G][4], sq[G][4], wz[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float *qp = a.qprep + ((size_t)b * a.heads_q + hk * G + g) * 2 * kD;
#pragma unroll
    for (int k = 0; k < 8; ++k) wz[g][k] = (k < a.side_rank) ? __ldg(qp + kD + k) : 0.f;
    const float4 q4 = __ldg(reinterpret_cast<const float4 *>(qp) + lane);
    qv[g][0] = q4.x; qv[g][1] = q4.y; qv[g][2] = q4.z; qv[g][3] = q4.w;
    if (KQJL) {
      const float4 s4 = __ldg(reinterpret_cast<const float4 *>(qp + kD) + lane);
      sq[g][0] = s4.x; sq[g][1] = s4.y; sq[g][2] = s4.z; sq[g][3] = s4.w;
    }
  }
  __syncthreads();

  float m[G], l[G], acc[G][4], sacc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[g][j] = sacc[g][j] = 0.f;
  }

  const long long slot0 = ((long long)b * a.heads_kv + hk) * a.cap16;
  // token t's physical slot (an unmapped block of a paged cache reads block 0; the error
  // word reports it)
  auto ps = [&](int t) -> long long {
    const long long p = phys_slot(a.btab, a.pool_blocks, slot0 + t, a.error);
    return p < 0 ? 0 : p;
  };
  auto rec32 = [&](const uint8_t *plane, long long slot, int tok) {
    return reinterpret_cast<const uint32_t *>(rec_at(plane, slot, a.bb, tok));
  };
  auto recf = [&](const float *plane, long long slot) { return __ldg(rec_at(plane, slot, a.bb, 4)); };
  const int my_tok = tile_token_of_lane(lane);

  for (int tile = t_begin + warp * kTile; tile < t_end; tile += kDecodeWarps * kTile) {
    // ---- scores for 8 tokens
    float part[G][kTile];
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      const long long sl = ps(min(tile + jj, t_end - 1));
      uint32_t code[4];
      lane_codes<KB>(rec32(a.k_codes, sl, KB * 16), lane, code);
      float c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = s_cb[code[j]];
      const float nu = recf(a.k_norm, sl);
      float sg[4];
      float rk = 0.f;
      if (KQJL) {
        uint32_t sb[4];
        lane_signs(rec32(a.k_signs, sl, 16), lane, sb);
#pragma unroll
        for (int j = 0; j < 4; ++j) sg[j] = sb[j] ? 1.f : -1.f;
        rk = recf(a.k_rnorm, sl);
      }
      // side code (lane 0 adds the key's correction w . z_hat once to the lanes' partial sums)
      float zt[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (a.side_rank && lane == 0) {
        const uint16_t *zp = rec_at(a.k_side, sl, a.bb, 2 * a.side_rank);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < a.side_rank) zt[k] = __half2float(__ushort_as_half(zp[k]));
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = qv[g][0] * c[0] + qv[g][1] * c[1] + qv[g][2] * c[2] + qv[g][3] * c[3];
        s *= nu;
        if (KQJL) s += rk * (sq[g][0] * sg[0] + sq[g][1] * sg[1] + sq[g][2] * sg[2] + sq[g][3] * sg[3]);
#pragma unroll
        for (int k = 0; k < 8; ++k) s = fmaf(wz[g][k], zt[k], s);
        part[g][jj] = s;
      }
    }
    // ---- online softmax over the 8 tokens
    const bool valid = tile + my_tok < t_end;
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float s = reduce8(part[g], lane);
      s = valid ? s : -INFINITY;
      float tmax = fmaxf(s, __shfl_xor_sync(kFull, s, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
      const float mnew = fmaxf(m[g], tmax);  // finite: token `tile` is valid
      const float scale = __expf(m[g] - mnew);
      p[g] = valid ? __expf(s - mnew) : 0.f;
      float psum = p[g] + __shfl_xor_sync(kFull, p[g], 4);
      psum += __shfl_xor_sync(kFull, psum, 8);
      psum += __shfl_xor_sync(kFull, psum, 16);
      l[g] = l[g] * scale + psum;
      m[g] = mnew;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[g][j] *= scale;
        if (VQJL) sacc[g][j] *= scale;
      }
    }
    // ---- values, in the rotated unit domain
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      const int t = tile + jj;
      if (t >= t_end) break;
      const int src = lane_of_tile_token(jj);
      const long long sl = ps(t);
      uint32_t code[4];
      lane_codes_vt<VB>(a.v_codes, sl, a.bb, lane, code);  // pair-interleaved value codes
      float c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = s_cb[16 + code[j]];
      const float nu = recf(a.v_norm, sl);
      uint32_t sb[4] = {0u, 0u, 0u, 0u};
      float rv = 0.f;
      if (VQJL) {
        lane_signs(rec32(a.v_signs, sl, 16), lane, sb);
        rv = recf(a.v_rnorm, sl);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pj = __shfl_sync(kFull, p[g], src);
        const float w = pj * nu;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = fmaf(w, c[j], acc[g][j]);
        if (VQJL) {
          const float wr = pj * rv;
#pragma unroll
          for (int j = 0; j < 4; ++j) sacc[g][j] += sb[j] ? wr : -wr;
        }
      }
    }
  }

  // ---- merge the four warps of the CTA
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s_acc[warp][g][4 * lane + j] = acc[g][j];
      if (VQJL) s_sacc[warp][g][4 * lane + j] = sacc[g][j];
    }
  }
  __syncthreads();
  const int i = tid;  // coordinate
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, s_m[w][g]);
    float L = 0.f, A = 0.f, Sg = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float e = (s_m[w][g] == -INFINITY) ? 0.f : __expf(s_m[w][g] - M);
      L += s_l[w][g] * e;
      A += s_acc[w][g][i] * e;
      if (VQJL) Sg += s_sacc[w][g][i] * e;
    }
    float *rec = a.partials + (((size_t)b * a.heads_q + hk * G + g) * a.splits + split) * kPartialFloats;
    if (i == 0) {
      rec[0] = M;
      rec[1] = L;
    }
    rec[2 + i] = A;
    rec[2 + kD + i] = Sg;
  }
}

struct CombineArgs {
  int batch, heads_q, splits, rotate, sketch_v;
  const float *partials;
  const float *diag;
  const float *sketch;
  float *out;
  // persistent layout (tile_prefix != nullptr): records [(cta + unit) * groups + group],
  // one query head per KV head
  const int32_t *tile_prefix;
  int persist_ctas, heads_kv, persist_groups;
  int group = 1;  // query heads per KV head (persistent records hold `group` heads per slot)
  int *error = nullptr;
  const float *rot = nullptr;  // dense rotation M (o = M^T o_rot), or nullptr (Walsh-Hadamard)
  int num_sms = 0;             // the device's SMs (sizes the combine's grid)
};

// The partial records of one query row: split-K ones in a row, or the persistent kernel's
// (cta, group) records of every CTA whose slice touched the row's head. record(k) is the
// k-th of count() records, or nullptr for a CTA whose slice was empty (it wrote nothing).
struct RowRecords {
  const CombineArgs &a;
  const float *base = nullptr;
  // persistent slices: CTA c holds tiles [bnd(c), bnd(c + 1)), bnd(c) = min(T, 4 floor(T4 c / C))
  long long T = 0, T4 = 1, C = 1, c_lo = 0, c_hi = -1;
  int unit = 0, hh = 0, nrec = 0;
  bool narrow = true;  // every quotient below fits 32-bit division

  __device__ __forceinline__ long long qdiv(long long n, long long d) const {
    return narrow ? (long long)((uint32_t)n / (uint32_t)d) : n / d;
  }
  __device__ __forceinline__ long long bnd(long long c) const { return min(T, 4 * qdiv(T4 * c, C)); }

  __device__ __forceinline__ RowRecords(const CombineArgs &args, int row) : a(args) {
    base = a.partials + (size_t)row * a.splits * kPartialFloats;
    if (!a.tile_prefix) {
      nrec = a.splits;
      return;
    }
    const int b = row / a.heads_q, h = (row % a.heads_q) / a.group;
    hh = (row % a.heads_q) % a.group;
    const int p0 = __ldg(a.tile_prefix + b), nb = __ldg(a.tile_prefix + b + 1) - p0;
    T = (long long)a.heads_kv * __ldg(a.tile_prefix + a.batch);
    T4 = (T + 3) / 4;
    C = a.persist_ctas;
    narrow = (T4 + 1) * (C + 1) < (1LL << 32);
    unit = b * a.heads_kv + h;
    if (nb > 0) {
      const long long us = (long long)a.heads_kv * p0 + (long long)h * nb, ue = us + nb;
      // the CTA holding tile g: the largest c with bnd(c) <= g
      c_lo = qdiv((us / 4 + 1) * C - 1, T4);
      c_hi = qdiv(((ue - 1) / 4 + 1) * C - 1, T4);
    }
    nrec = (int)(a.persist_groups * (c_hi - c_lo + 1));
  }
  __device__ __forceinline__ const float *record(int k) const {
    if (!a.tile_prefix) return base + (size_t)k * kPartialFloats;
    const int ng = a.persist_groups;
    const long long c = c_lo + k / ng;
    if (bnd(c) == bnd(c + 1)) return nullptr;
    return a.partials + (((size_t)(c + unit) * ng + (k % ng)) * a.group + hh) * kPartialFloats;
  }
};

// Finish R query rows per CTA of 512 threads: a team of W = 16 / R warps per row merges the
// row's partial records in parallel -- the records' maximum M first, then warp w sums
// e^(m_k - M) (l_k, A_k, Sg_k) over records k = w (mod W), and the team adds the W partial
// sums -- then adds the sketch term (sqrt(pi/2)/m) S^T Sg with S staged in shared memory,
// divides by L and undoes the rotation (inverse WHT, then D; or M^T).
constexpr int kCombineThreads = 512;
constexpr int kPartStride = 2 * kD + 4;  // floats per warp's partial sums: A, Sg, L (16-byte rows)

template <int R>
__global__ void __launch_bounds__(kCombineThreads) combine_tq_kernel(CombineArgs a) {
  constexpr int W = 16 / R, TS = 32 * W, NS = TS / kD;  // warps, threads, S^T k-slices per row
  extern __shared__ __align__(16) float s_comb[];
  __shared__ uint64_t s_bar;
  __shared__ float s_red[16];
  float *s_sk = s_comb;                              // [128][128] S (sketch_v only)
  float *s_part = s_sk + (a.sketch_v ? kD * kD : 0);  // [16 warps][kPartStride] partial sums
  float *s_v = s_part + 16 * kPartStride;            // [R][NS][128] S^T slices, then [R][128] outputs
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rr = warp / W, w = warp % W, t = tid % TS;  // row of the CTA, warp and thread in its team
  const int nrows = a.batch * a.heads_q;
  const int row = blockIdx.x * R + rr;
  // S (a context constant) streams into shared memory while the records are merged
  if (a.sketch_v && tid == 0) {
    mbar_init(&s_bar, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(&s_bar, kD * kD * sizeof(float));
    tma_load_1d(s_sk, a.sketch, kD * kD * sizeof(float), &s_bar);
  }
  pdl_wait();     // the partial records come from the decode kernel before
  pdl_trigger();  // the next kernel of the stream (e.g. the next step's append) may be scheduled
  const bool live = row < nrows;
  const RowRecords rec(a, live ? row : 0);
  const int nrec = live ? rec.nrec : 0;

  // the records' maximum
  float m = -INFINITY;
  for (int k = t; k < nrec; k += TS) {
    const float *r = rec.record(k);
    if (r) m = fmaxf(m, __ldg(r));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < W; ++j) M = fmaxf(M, s_red[rr * W + j]);

  // this warp's share: lane L holds coordinates 2L, 2L + 1, 64 + 2L, 65 + 2L
  float L = 0.f, A[4] = {0.f, 0.f, 0.f, 0.f}, G[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int k = w; k < nrec; k += W) {
    const float *r = rec.record(k);
    if (!r) continue;
    const float ms = __ldg(r);
    if (ms == -INFINITY) continue;
    const float e = __expf(ms - M);
    L = fmaf(__ldg(r + 1), e, L);
    const float2 a0 = __ldg(reinterpret_cast<const float2 *>(r + 2) + lane);
    const float2 a1 = __ldg(reinterpret_cast<const float2 *>(r + 2 + 64) + lane);
    A[0] = fmaf(a0.x, e, A[0]);
    A[1] = fmaf(a0.y, e, A[1]);
    A[2] = fmaf(a1.x, e, A[2]);
    A[3] = fmaf(a1.y, e, A[3]);
    if (a.sketch_v) {
      const float2 g0 = __ldg(reinterpret_cast<const float2 *>(r + 2 + kD) + lane);
      const float2 g1 = __ldg(reinterpret_cast<const float2 *>(r + 2 + kD + 64) + lane);
      G[0] = fmaf(g0.x, e, G[0]);
      G[1] = fmaf(g0.y, e, G[1]);
      G[2] = fmaf(g1.x, e, G[2]);
      G[3] = fmaf(g1.y, e, G[3]);
    }
  }
  float *mine = s_part + warp * kPartStride;
  reinterpret_cast<float2 *>(mine)[lane] = make_float2(A[0], A[1]);
  reinterpret_cast<float2 *>(mine + 64)[lane] = make_float2(A[2], A[3]);
  reinterpret_cast<float2 *>(mine + kD)[lane] = make_float2(G[0], G[1]);
  reinterpret_cast<float2 *>(mine + kD + 64)[lane] = make_float2(G[2], G[3]);
  if (lane == 0) mine[2 * kD] = L;
  __syncthreads();
  // the team's sums: thread t < 128 of the team takes coordinate t (A, and Sg into slot W)
  const float *team = s_part + rr * W * kPartStride;
  float Lr = 0.f;
#pragma unroll
  for (int j = 0; j < W; ++j) Lr += team[j * kPartStride + 2 * kD];
  float Ar = 0.f, Gr = 0.f;
  if (t < kD) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      Ar += team[j * kPartStride + t];
      Gr += team[j * kPartStride + kD + t];
    }
  }
  __syncthreads();  // every team read its partial sums
  float *sg = s_part + rr * kD;  // the team's Sg, over its (now free) partial sums
  if (t < kD) sg[t] = Gr;
  __syncthreads();
  // sketch term: slice j = t / 128 of the team sums k in [j * 128 / NS, (j + 1) * 128 / NS)
  float *slices = s_v + rr * NS * kD;
  if (a.sketch_v) {
    const bool ok = mbar_wait_bounded(&s_bar, 0, a.error);
    const int i = t % kD, j = t / kD;
    float acc = 0.f;
    if (ok) {
#pragma unroll 8
      for (int k = j * (kD / NS); k < (j + 1) * (kD / NS); ++k) acc = fmaf(s_sk[k * kD + i], sg[k], acc);
    }
    slices[j * kD + i] = acc;
  }
  __syncthreads();
  float *s_o = s_v + R * NS * kD;  // [R][128]
  if (t < kD) {
    float o = Ar;
    if (a.sketch_v) {
      float x = 0.f;
#pragma unroll
      for (int j = 0; j < NS; ++j) x += slices[j * kD + t];
      o += (kSqrtHalfPi / kD) * x;
    }
    s_o[rr * kD + t] = (Lr > 0.f) ? o / Lr : 0.f;
  }
  __syncthreads();
  // rotate back: the team's first warp
  if (w == 0 && live) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = s_o[rr * kD + 4 * lane + j];
    if (a.rotate && a.rot) {
      matvec_t_warp(a.rot, v, lane);
    } else if (a.rotate) {
      wht128(v, lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= __ldg(a.diag + 4 * lane + j);
    }
    reinterpret_cast<float4 *>(a.out + (size_t)row * kD)[lane] = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// rows per CTA: four when the rows fill the GPU three times over, else fewer, so that the
// records of few rows spread over more warps
int combine_rows_per_cta(int rows, int num_sms) {
  if (num_sms <= 0) num_sms = 1;
  if (rows >= 3 * num_sms) return 4;
  if (rows >= (3 * num_sms) / 2) return 2;
  return 1;
}

size_t combine_smem(const CombineArgs &a, int R) {
  const int NS = (kCombineThreads / R) / kD;
  return sizeof(float) * ((a.sketch_v ? kD * kD : 0) + 16 * kPartStride + R * NS * kD + R * kD);
}

template <int R>
int launch_combine_r(const CombineArgs &a, cudaStream_t st) {
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(combine_tq_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(float) * kD * kD + combine_smem(CombineArgs{}, R))) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  const int rows = a.batch * a.heads_q;
  return launch_overlapped(true, combine_tq_kernel<R>, dim3((rows + R - 1) / R), dim3(kCombineThreads),
                           combine_smem(a, R), st, a) == cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

int launch_combine(const CombineArgs &a, cudaStream_t st) {
  const int R = combine_rows_per_cta(a.batch * a.heads_q, a.num_sms);
  if (R == 4) return launch_combine_r<4>(a, st);
  if (R == 2) return launch_combine_r<2>(a, st);
  return launch_combine_r<1>(a, st);
}

// ---------------------------------------------------------------- decode step

__global__ void step_lengths_kernel(const int32_t *seq_lens, int batch, int capacity, int32_t *out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) {
    const int len = __ldg(seq_lens + b);
    out[b] = (len < 0) ? 0 : min(len, capacity - 1) + 1;
  }
}

// ---------------------------------------------------------------- KIVI decode
// Scores and values from 2-bit grouped codes ("Your KV cache is not a bit
// problem but a geometry problem", "What quantisation error is made of":
// x_hat = zero + step * code) for tokens [0, nq) and from the bfloat16 window
// for [nq, len); same online softmax and split-K partials as above, with no
// rotation and no sketch.

struct KiviDecodeKernelArgs {
  const uint8_t *k_codes;
  const uint8_t *v_codes;
  const uint16_t *k_stats;
  const uint16_t *v_stats;
  const uint16_t *k_ring;
  const uint16_t *v_ring;
  int capacity, heads_kv, heads_q, chunk, splits, window;
  const int32_t *seq_lens;
  const float *qprep;
  float *partials;
};

__device__ __forceinline__ void half2_pair(uint32_t st, float &z, float &s) {
  z = __half2float(__ushort_as_half((unsigned short)(st & 0xffffu)));
  s = __half2float(__ushort_as_half((unsigned short)(st >> 16)));
}

// A code c (0..3) enters the arithmetic as the exact float 1 + c/4 (its two bits placed in the
// top of the mantissa of 1.0). A dequantised value
// z + s c is then 4 s (1 + c/4) + (z - 4 s), so the two stats fold into per-group (or per-token)
// constants and a code costs no int-to-float conversion. kivi_codes4 gives those floats for a
// lane's four channels, two per lookup: byte `sel` picks (this lane's byte of a record word,
// moved to bits 8..15 by one byte permute) indexes a lane-replicated table of the 16 nibble
// values, T[n][lane] = (1 + (n & 3)/4, 1 + (n >> 2)/4), at byte offset n * 256 + lane * 8 (a
// warp's 32 lookups of one nibble fill two wavefronts, no conflict).
__device__ __forceinline__ void kivi_codes4(const unsigned char *tab, uint32_t lane8, uint32_t word, uint32_t sel,
                                            float2 &c01, float2 &c23) {
  const uint32_t x = __byte_perm(word, 0u, sel);
  c01 = *reinterpret_cast<const float2 *>(tab + ((x & 0xF00u) | lane8));
  c23 = *reinterpret_cast<const float2 *>(tab + (((x >> 4) & 0xF00u) | lane8));
}

// four channels 4L..4L+3 of a window token's bfloat16 row staged in shared memory (64 words)
__device__ __forceinline__ void kivi_window_row(const uint32_t *row, int lane, float (&x)[4]) {
  const uint2 w = reinterpret_cast<const uint2 *>(row)[lane];
  x[0] = bf16_bits_to_float(w.x & 0xffffu);
  x[1] = bf16_bits_to_float(w.x >> 16);
  x[2] = bf16_bits_to_float(w.y & 0xffffu);
  x[3] = bf16_bits_to_float(w.y >> 16);
}

template <bool KPC, bool VPT, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_kivi_kernel(KiviDecodeKernelArgs a) {
  __shared__ float s_m[kDecodeWarps][G], s_l[kDecodeWarps][G];
  __shared__ float s_acc[kDecodeWarps][G][kD];
  __shared__ __align__(16) float2 s_nib[16][32];  // kivi_codes4's table
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = min(max(__ldg(a.seq_lens + b), 0), a.capacity);
  const int nq = (len < a.window + 32) ? 0 : 32 * ((len - a.window) / 32);
  const int t_begin = split * a.chunk;
  const int t_end = min(t_begin + a.chunk, len);
  const int R = a.window + 32;

  float qv[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float4 q4 = __ldg(reinterpret_cast<const float4 *>(a.qprep + ((size_t)b * a.heads_q + hk * G + g) * 2 * kD) + lane);
    qv[g][0] = q4.x; qv[g][1] = q4.y; qv[g][2] = q4.z; qv[g][3] = q4.w;
  }
  // accumulators of this lane's channels 4L..4L+3 as two pairs (packed fp32 FMAs)
  float m[G], l[G];
  float2 acc[G][2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) acc[g][j] = make_float2(0.f, 0.f);
  }
  for (int e = tid; e < 16 * 32; e += kDecodeWarps * 32) {
    const int n = e >> 5;
    s_nib[n][e & 31] = make_float2(1.f + 0.25f * (float)(n & 3), 1.f + 0.25f * (float)(n >> 2));
  }
  __syncthreads();
  const unsigned char *nib = reinterpret_cast<const unsigned char *>(&s_nib[0][0]);
  const uint32_t lane8 = (uint32_t)lane << 3, bsel = 0x4404u | ((uint32_t)(lane & 3) << 4);
  const size_t bh = (size_t)b * a.heads_kv + hk;
  const uint32_t *kc = reinterpret_cast<const uint32_t *>(a.k_codes) + bh * a.capacity * 8;
  const uint32_t *vc = reinterpret_cast<const uint32_t *>(a.v_codes) + bh * a.capacity * 8;
  // per-token stats: [slot][4 groups]; per-channel stats: [group][128 channels]
  const uint32_t *ks_tok = reinterpret_cast<const uint32_t *>(a.k_stats) + bh * a.capacity * 4;
  const uint32_t *vs_tok = reinterpret_cast<const uint32_t *>(a.v_stats) + bh * a.capacity * 4;
  const uint32_t *ks_ch = reinterpret_cast<const uint32_t *>(a.k_stats) + bh * (a.capacity / 32) * kD;
  const uint32_t *vs_ch = reinterpret_cast<const uint32_t *>(a.v_stats) + bh * (a.capacity / 32) * kD;
  const uint16_t *kring = a.k_ring + bh * R * kD;
  const uint16_t *vring = a.v_ring + bh * R * kD;
  const int my_tok = tile_token_of_lane(lane);

  // per lane: the sum of its query coordinates (per-token key stats)
  float qsum[G];
#pragma unroll
  for (int g = 0; g < G; ++g) qsum[g] = (qv[g][0] + qv[g][1]) + (qv[g][2] + qv[g][3]);

  // Quantised tokens stream through a per-warp double buffer in shared memory, one 32-token
  // group per stage (cp.async, 16 bytes per lane and copy): the K and V codes (1 KB each) and
  // the group's K and V statistics (512 B each: per-channel [128] or per-token [32][4]
  // (zero, step) pairs). A warp takes whole groups; window tokens are read directly.
  __shared__ __align__(16) uint32_t s_buf[kDecodeWarps][2][768];  // kc 256 | vc 256 | ks 128 | vs 128 words
  auto prefetch = [&](int tile0, int bi) {
    uint32_t *sb = s_buf[warp][bi];
    const uint32_t *k0 = kc + (size_t)tile0 * 8, *v0 = vc + (size_t)tile0 * 8;
    cp_async_16(sb + 8 * lane, k0 + 8 * lane);
    cp_async_16(sb + 8 * lane + 4, k0 + 8 * lane + 4);
    cp_async_16(sb + 256 + 8 * lane, v0 + 8 * lane);
    cp_async_16(sb + 256 + 8 * lane + 4, v0 + 8 * lane + 4);
    const uint32_t *ks0 = KPC ? ks_ch + (size_t)(tile0 / 32) * kD : ks_tok + (size_t)tile0 * 4;
    const uint32_t *vs0 = VPT ? vs_tok + (size_t)tile0 * 4 : vs_ch + (size_t)(tile0 / 32) * kD;
    cp_async_16(sb + 512 + 4 * lane, ks0 + 4 * lane);
    cp_async_16(sb + 640 + 4 * lane, vs0 + 4 * lane);
    cp_async_commit();
  };
  constexpr int kGroupTok = 32;
  const int qend = min(t_end, nq);  // this chunk's quantised tokens end here
  int it = 0;
  if (t_begin + warp * kGroupTok < qend) prefetch(t_begin + warp * kGroupTok, 0);
  for (int tile0 = t_begin + warp * kGroupTok; tile0 < t_end; tile0 += kDecodeWarps * kGroupTok, ++it) {
    const bool quant = tile0 < nq;  // groups lie wholly in the quantised part or the window
    const uint32_t *sb = s_buf[warp][it & 1];
    if (quant) {
      const int nxt = tile0 + kDecodeWarps * kGroupTok;
      if (nxt < qend) {
        prefetch(nxt, (it + 1) & 1);
        cp_async_wait_one();
      } else {
        cp_async_wait_all();
      }
      __syncwarp();
    }
    float kz[4] = {0.f, 0.f, 0.f, 0.f}, kscl[4] = {0.f, 0.f, 0.f, 0.f};
    float vz[4] = {0.f, 0.f, 0.f, 0.f}, vscl[4] = {0.f, 0.f, 0.f, 0.f};
    if (quant && KPC) {
      const uint4 s4 = reinterpret_cast<const uint4 *>(sb + 512)[lane];
      half2_pair(s4.x, kz[0], kscl[0]); half2_pair(s4.y, kz[1], kscl[1]);
      half2_pair(s4.z, kz[2], kscl[2]); half2_pair(s4.w, kz[3], kscl[3]);
    }
    if (quant && !VPT) {
      const uint4 s4 = reinterpret_cast<const uint4 *>(sb + 640)[lane];
      half2_pair(s4.x, vz[0], vscl[0]); half2_pair(s4.y, vz[1], vscl[1]);
      half2_pair(s4.z, vz[2], vscl[2]); half2_pair(s4.w, vz[3], vscl[3]);
    }
    // per-channel key stats: this lane's part of q . k_hat = cst + sum_j (4 q_j s_j) (1 + c_j / 4)
    float q4s[G][4], cst[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      cst[g] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        q4s[g][j] = 4.f * qv[g][j] * kscl[j];
        cst[g] = fmaf(qv[g][j], fmaf(-4.f, kscl[j], kz[j]), cst[g]);
      }
    }
    // one 8-token sub-tile; QUANT: of a quantised group (always whole: chunks and groups are
    // 32-token aligned), so no token is masked and every record offset is a constant
    auto sub8 = [&](const int tile, auto quant_c) {
      constexpr bool QUANT = decltype(quant_c)::value;
      // window tokens: the sub-tile's K and V rows (8 x 256 B each) staged in this warp's
      // buffer in one round of copies (no quantised group is in flight once the window starts)
      const uint32_t *wb = &s_buf[warp][0][0];
      if constexpr (!QUANT) {
#pragma unroll
        for (int c = lane; c < 256; c += 32) {
          const int tensor = c >> 7, jj = (c >> 4) & 7, part = c & 15;
          const int t = min(tile + jj, t_end - 1);
          cp_async_16(&s_buf[warp][0][0] + tensor * 512 + jj * 64 + 4 * part,
                      (tensor ? vring : kring) + (size_t)(t % R) * kD + 8 * part);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncwarp();
      }
      float part[G][kTile];
#pragma unroll
      for (int jj = 0; jj < kTile; ++jj) {
        const int t = QUANT ? tile + jj : min(tile + jj, t_end - 1);
        if constexpr (QUANT) {
          // keys: the code floats by bit placement (two logic ops each) -- the table lookups
          // that the values use would put the shared-memory path, already the busier one,
          // further ahead (measured 2 % slower for keys)
          float2 c01, c23;
          {
            const uint32_t f = sb[(t - tile0) * 8 + (lane >> 2)] >> (8 * (lane & 3));
            auto cf = [&](int j) { return __uint_as_float(0x3F800000u | ((f << (21 - 2 * j)) & 0x600000u)); };
            c01 = make_float2(cf(0), cf(1));
            c23 = make_float2(cf(2), cf(3));
          }
          if (KPC) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float2 d2 = __ffma2_rn(make_float2(q4s[g][0], q4s[g][1]), c01, make_float2(cst[g], 0.f));
              d2 = __ffma2_rn(make_float2(q4s[g][2], q4s[g][3]), c23, d2);
              part[g][jj] = d2.x + d2.y;
            }
          } else {
            // per-token key stats of this lane's channel group: z q_sum + 4 s (sum_j q_j f_j - q_sum)
            float z, sc;
            half2_pair(sb[512 + (t - tile0) * 4 + (lane >> 3)], z, sc);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float2 d2 = __fmul2_rn(make_float2(qv[g][0], qv[g][1]), c01);
              d2 = __ffma2_rn(make_float2(qv[g][2], qv[g][3]), c23, d2);
              const float d = d2.x + d2.y;
              part[g][jj] = fmaf(4.f * sc, d - qsum[g], z * qsum[g]);
            }
          }
        } else {
          float x[4];
          kivi_window_row(wb + jj * 64, lane, x);
#pragma unroll
          for (int g = 0; g < G; ++g) part[g][jj] = qv[g][0] * x[0] + qv[g][1] * x[1] + qv[g][2] * x[2] + qv[g][3] * x[3];
        }
      }
      const bool valid = QUANT || tile + my_tok < t_end;
      float p[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = reduce8(part[g], lane);
        s = valid ? s : -INFINITY;
        float tmax = fmaxf(s, __shfl_xor_sync(kFull, s, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
        const float mnew = fmaxf(m[g], tmax);
        const float scale = __expf(m[g] - mnew);
        p[g] = valid ? __expf(s - mnew) : 0.f;
        float psum = p[g] + __shfl_xor_sync(kFull, p[g], 4);
        psum += __shfl_xor_sync(kFull, psum, 8);
        psum += __shfl_xor_sync(kFull, psum, 16);
        l[g] = l[g] * scale + psum;
        m[g] = mnew;
#pragma unroll
        for (int j = 0; j < 2; ++j) acc[g][j] = __fmul2_rn(acc[g][j], make_float2(scale, scale));
      }
      // values: p (z + s c) = (4 p s) (1 + c/4) + p (z - 4 s); per-token stats fold into the
      // token's weight, per-channel ones into the tile's sums u_j = sum p (1 + c_j / 4), P = sum p
      float2 u[G][2];
      float pz[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pz[g] = 0.f;
        u[g][0] = u[g][1] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int jj = 0; jj < kTile; ++jj) {
        const int t = tile + jj;
        if (!QUANT && t >= t_end) break;
        float w[G];
#pragma unroll
        for (int g = 0; g < G; ++g) w[g] = __shfl_sync(kFull, p[g], lane_of_tile_token(jj));
        if constexpr (QUANT) {
          float2 c01, c23;
          kivi_codes4(nib, lane8, sb[256 + (t - tile0) * 8 + (lane >> 2)], bsel, c01, c23);
          if (VPT) {
            float z, sc;
            half2_pair(sb[640 + (t - tile0) * 4 + (lane >> 3)], z, sc);
            const float s4 = 4.f * sc, z4 = fmaf(-4.f, sc, z);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float2 w1 = make_float2(w[g] * s4, w[g] * s4);
              acc[g][0] = __ffma2_rn(w1, c01, acc[g][0]);
              acc[g][1] = __ffma2_rn(w1, c23, acc[g][1]);
              pz[g] = fmaf(w[g], z4, pz[g]);
            }
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              u[g][0] = __ffma2_rn(make_float2(w[g], w[g]), c01, u[g][0]);
              u[g][1] = __ffma2_rn(make_float2(w[g], w[g]), c23, u[g][1]);
              pz[g] += w[g];
            }
          }
        } else {
          float x[4];
          kivi_window_row(wb + 512 + jj * 64, lane, x);
#pragma unroll
          for (int g = 0; g < G; ++g)
          {
            acc[g][0] = __ffma2_rn(make_float2(w[g], w[g]), make_float2(x[0], x[1]), acc[g][0]);
            acc[g][1] = __ffma2_rn(make_float2(w[g], w[g]), make_float2(x[2], x[3]), acc[g][1]);
          }
        }
      }
      if constexpr (QUANT) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int j = 0; j < 4; ++j)
          {
            const float uj = (j & 1) ? u[g][j >> 1].y : u[g][j >> 1].x;
            const float add = VPT ? pz[g] : fmaf(4.f * vscl[j], uj, fmaf(-4.f, vscl[j], vz[j]) * pz[g]);
            if (j & 1) acc[g][j >> 1].y += add;
            else acc[g][j >> 1].x += add;
          }
      } else {
        __syncwarp();  // every lane is done with the staged rows before the next copies
      }
    };
    if (quant) {
#pragma unroll
      for (int sub = 0; sub < kGroupTok / kTile; ++sub) sub8(tile0 + kTile * sub, std::true_type{});
    } else {
      for (int tile = tile0; tile < tile0 + kGroupTok && tile < t_end; tile += kTile) sub8(tile, std::false_type{});
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s_acc[warp][g][4 * lane + j] = (j & 1) ? acc[g][j >> 1].y : acc[g][j >> 1].x;
  }
  __syncthreads();
  const int i = tid;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, s_m[w][g]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float e = (s_m[w][g] == -INFINITY) ? 0.f : __expf(s_m[w][g] - M);
      L += s_l[w][g] * e;
      A += s_acc[w][g][i] * e;
    }
    float *rec = a.partials + (((size_t)b * a.heads_q + hk * G + g) * a.splits + split) * kPartialFloats;
    if (i == 0) {
      rec[0] = M;
      rec[1] = L;
    }
    rec[2 + i] = A;
    rec[2 + kD + i] = 0.f;
  }
}

template <bool KPC, bool VPT>
int launch_kivi_g(const KiviDecodeKernelArgs &k, int G, dim3 grid, cudaStream_t st) {
  switch (G) {
    case 1: decode_kivi_kernel<KPC, VPT, 1><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 2: decode_kivi_kernel<KPC, VPT, 2><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 4: decode_kivi_kernel<KPC, VPT, 4><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 8: decode_kivi_kernel<KPC, VPT, 8><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return TQ_OK;
}

template <int KB, int VB, bool KQJL, bool VQJL>
int launch_decode_g(const DecodeKernelArgs &k, int G, dim3 grid, cudaStream_t st) {
  switch (G) {
    case 1: decode_tq_kernel<KB, VB, KQJL, VQJL, 1><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 2: decode_tq_kernel<KB, VB, KQJL, VQJL, 2><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 4: decode_tq_kernel<KB, VB, KQJL, VQJL, 4><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    case 8: decode_tq_kernel<KB, VB, KQJL, VQJL, 8><<<grid, kDecodeWarps * 32, 0, st>>>(k); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return TQ_OK;
}

}  // namespace

int launch_decode_tq(const DecodeArgs &a, void *stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const tq_ctx *ctx = a.ctx;
  const int G = a.heads_q / a.heads_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TQ_ERR_UNSUPPORTED;

  // the persistent kernels (one query head per KV head, or GQA groups of 2 / 4 without
  // key sketches) take the per-batch tile prefix the query prep computes
  const bool persist_ok = G == 1 || ((G == 2 || G == 4) && ctx->scheme != TQ_SCHEME_QKQV);
  PrepArgs p{a.q, a.q_dtype == TQ_BF16, a.batch, a.heads_q, ctx->k.rotate, ctx->k.qjl,
             ctx->dparams->diag, ctx->dparams->sketch, a.qprep,
             a.seq_lens, a.cache->capacity, persist_ok ? a.tile_prefix : nullptr};
  p.rot_t = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot_t : nullptr;
  p.sketch_tp = ctx->dparams->sketch_tp;
  p.side_ur = ctx->side_ur;
  p.side_rank = ctx->side_rank;
  p.group = G;
  const int rows = a.batch * a.heads_q;
  if (launch_overlapped(true, qprep_kernel, dim3((rows + 3) / 4), dim3(128), 0, st, p) != cudaSuccess)
    return TQ_ERR_CUDA;

  // the TMA / tensor-core kernels cover one query head per KV head
  if (ctx->prof_decode_start) cudaEventRecord((cudaEvent_t)ctx->prof_decode_start, st);
  int persist_ctas = 0;
  DecodeArgs a2 = a;
  if (!persist_ok) a2.tile_prefix = nullptr;
  // keys with side codes: the scalar kernel below adds their logit correction
  int r2 = ctx->side_rank ? TQ_ERR_UNSUPPORTED : launch_decode2_g1(a2, &persist_ctas, stream);
  if (r2 == TQ_OK) {
    if (ctx->prof_decode_stop) cudaEventRecord((cudaEvent_t)ctx->prof_decode_stop, st);
    CombineArgs cmb{a.batch, a.heads_q, a.splits, ctx->v.rotate, ctx->v.qjl, a.partials,
                    ctx->dparams->diag, ctx->dparams->sketch, a.out,
                    persist_ctas ? a.tile_prefix : nullptr, persist_ctas, a.heads_kv, G == 1 ? 1 : kPersistGroups};
    cmb.group = G;
    cmb.error = &ctx->dparams->error;
    cmb.num_sms = ctx->num_sms;
    cmb.rot = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot : nullptr;
    return launch_combine(cmb, st);
  }
  if (r2 != TQ_ERR_UNSUPPORTED) return r2;

  DecodeKernelArgs k{};
  const tq_cache *c = a.cache;
  const RecLayout &L = ctx->lay;
  auto plane = [&](int p) -> const uint8_t * { return L.tok[p] ? c->records + L.off[p] : nullptr; };
  k.k_codes = plane(TQ_PLANE_K_CODES); k.k_norm = reinterpret_cast<const float *>(plane(TQ_PLANE_K_NORM));
  k.k_signs = plane(TQ_PLANE_K_SIGNS); k.k_rnorm = reinterpret_cast<const float *>(plane(TQ_PLANE_K_RNORM));
  k.v_codes = plane(TQ_PLANE_V_CODES); k.v_norm = reinterpret_cast<const float *>(plane(TQ_PLANE_V_NORM));
  k.v_signs = plane(TQ_PLANE_V_SIGNS); k.v_rnorm = reinterpret_cast<const float *>(plane(TQ_PLANE_V_RNORM));
  k.bb = L.bb;
  k.cap16 = cap16_of(c->capacity);
  k.btab = c->block_table;
  k.pool_blocks = c->pool_blocks;
  k.error = &ctx->dparams->error;
  k.side_rank = ctx->side_rank;
  k.k_side = ctx->side_rank ? reinterpret_cast<const uint16_t *>(c->records + L.off[TQ_PLANE_K_SIDE]) : nullptr;
  k.capacity = c->capacity;
  k.heads_kv = a.heads_kv;
  k.heads_q = a.heads_q;
  k.chunk = a.chunk;
  k.splits = a.splits;
  k.seq_lens = a.seq_lens;
  k.qprep = a.qprep;
  k.partials = a.partials;
  k.k_centroids = ctx->dparams->k_centroids;
  k.v_centroids = ctx->dparams->v_centroids;
  dim3 grid(a.splits, a.heads_kv, a.batch);
  const int kb = ctx->k.bits, vb = ctx->v.bits;
  int r = TQ_ERR_UNSUPPORTED;
  if (ctx->prof_decode_start) cudaEventRecord((cudaEvent_t)ctx->prof_decode_start, st);
  switch (ctx->scheme) {
    case TQ_SCHEME_KV:
      if (kb == 2) r = launch_decode_g<2, 2, false, false>(k, G, grid, st);
      else if (kb == 3) r = launch_decode_g<3, 3, false, false>(k, G, grid, st);
      else if (kb == 4) r = launch_decode_g<4, 4, false, false>(k, G, grid, st);
      break;
    case TQ_SCHEME_KQV:
      if (kb == 2) r = launch_decode_g<2, 1, false, true>(k, G, grid, st);
      else if (kb == 3) r = launch_decode_g<3, 2, false, true>(k, G, grid, st);
      else if (kb == 4) r = launch_decode_g<4, 3, false, true>(k, G, grid, st);
      break;
    case TQ_SCHEME_QKQV:
      if (kb == 1) r = launch_decode_g<1, 1, true, true>(k, G, grid, st);
      else if (kb == 2) r = launch_decode_g<2, 2, true, true>(k, G, grid, st);
      else if (kb == 3) r = launch_decode_g<3, 3, true, true>(k, G, grid, st);
      break;
    default: break;
  }
  (void)vb;
  if (ctx->prof_decode_stop) cudaEventRecord((cudaEvent_t)ctx->prof_decode_stop, st);
  if (r != TQ_OK) return r;

  CombineArgs cmb{a.batch, a.heads_q, a.splits, ctx->v.rotate, ctx->v.qjl, a.partials,
                  ctx->dparams->diag, ctx->dparams->sketch, a.out, nullptr, 0, a.heads_kv, 1};
  cmb.error = &ctx->dparams->error;
  cmb.num_sms = ctx->num_sms;
  cmb.rot = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot : nullptr;
  return launch_combine(cmb, st);
}

int launch_step_lengths(const int32_t *seq_lens, int batch, int capacity, int32_t *lens_out, void *stream) {
  step_lengths_kernel<<<(batch + 127) / 128, 128, 0, (cudaStream_t)stream>>>(seq_lens, batch, capacity, lens_out);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

int launch_decode_step_tq(const DecodeArgs &a, const StepArgs &s, void *stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const tq_ctx *ctx = a.ctx;
  if (ctx->prof_decode_start) cudaEventRecord((cudaEvent_t)ctx->prof_decode_start, st);
  int persist_ctas = 0;
  const int r = launch_decode2_step(a, s, &persist_ctas, stream);
  if (r != TQ_OK) return r;
  if (ctx->prof_decode_stop) cudaEventRecord((cudaEvent_t)ctx->prof_decode_stop, st);
  CombineArgs cmb{a.batch, a.heads_q, a.splits, ctx->v.rotate, ctx->v.qjl, a.partials,
                  ctx->dparams->diag, ctx->dparams->sketch, a.out, a.tile_prefix, persist_ctas, a.heads_kv, 1};
  cmb.group = 1;
  cmb.error = &ctx->dparams->error;
  cmb.num_sms = ctx->num_sms;
  cmb.rot = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot : nullptr;
  return launch_combine(cmb, st);
}

int launch_decode_kivi(const DecodeArgs &a, void *stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const tq_ctx *ctx = a.ctx;
  const int G = a.heads_q / a.heads_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TQ_ERR_UNSUPPORTED;
  if (ctx->kivi_group != 32) return TQ_ERR_UNSUPPORTED;
  PrepArgs p{a.q, a.q_dtype == TQ_BF16, a.batch, a.heads_q, 0, 0, ctx->dparams->diag, ctx->dparams->sketch, a.qprep,
             a.seq_lens, a.cache->capacity, nullptr};
  const int rows = a.batch * a.heads_q;
  if (launch_overlapped(true, qprep_kernel, dim3((rows + 3) / 4), dim3(128), 0, st, p) != cudaSuccess)
    return TQ_ERR_CUDA;
  const tq_cache *c = a.cache;
  KiviDecodeKernelArgs k{};
  k.k_codes = c->k_codes; k.v_codes = c->v_codes;
  k.k_stats = c->k_stats; k.v_stats = c->v_stats;
  k.k_ring = c->k_window; k.v_ring = c->v_window;
  k.capacity = c->capacity;
  k.heads_kv = a.heads_kv;
  k.heads_q = a.heads_q;
  k.chunk = a.chunk;
  k.splits = a.splits;
  k.window = ctx->kivi_window;
  k.seq_lens = a.seq_lens;
  k.qprep = a.qprep;
  k.partials = a.partials;
  dim3 grid(a.splits, a.heads_kv, a.batch);
  const bool kpc = ctx->kivi_k_per_channel != 0, vpt = ctx->kivi_v_per_token != 0;
  int r;
  if (ctx->prof_decode_start) cudaEventRecord((cudaEvent_t)ctx->prof_decode_start, st);
  if (kpc && vpt) r = launch_kivi_g<true, true>(k, G, grid, st);
  else if (kpc) r = launch_kivi_g<true, false>(k, G, grid, st);
  else if (vpt) r = launch_kivi_g<false, true>(k, G, grid, st);
  else r = launch_kivi_g<false, false>(k, G, grid, st);
  if (ctx->prof_decode_stop) cudaEventRecord((cudaEvent_t)ctx->prof_decode_stop, st);
  if (r != TQ_OK) return r;
  CombineArgs cmb{a.batch, a.heads_q, a.splits, 0, 0, a.partials, ctx->dparams->diag, ctx->dparams->sketch, a.out,
                  nullptr, 0, a.heads_kv, 1};
  cmb.error = &ctx->dparams->error;
  cmb.num_sms = ctx->num_sms;
  return launch_combine(cmb, st);
}

}  // namespace tq
