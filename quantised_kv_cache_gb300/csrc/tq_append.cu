// Append-quantise: norm -> seeded +/-1 diagonal -> in-register Walsh-Hadamard
// -> branch-free bucketize against the float32 Lloyd-Max boundaries -> packed
// code record; for sketched vectors also sign(S r) and rho = ||x|| ||r||.
//
// "Statistical Inference and Quality Measures of KV Cache Quantisations
// Inspired by TurboQuant", technical summary, "Quantisation schemes" (WHT +
// scalar Lloyd-Max, with a 1-bit QJL sketch of the residual for the (n-1)-bit
// vectors) and "Main contribution 1" (the sketch keeps only sign(S r) and the
// residual's norm). "KVQuant++", "Fast codebook lookup": the code is found by
// counting boundaries (bucketize) rather than by an argmin over centroids.
//
// One warp quantises one vector (lane L holds coordinates 4L..4L+3). For
// sketched vectors a warp collects 8 vectors' unit-domain residuals in shared
// memory and forms S r for all 8 at once against a block-resident copy of S,
// so each S element read from shared memory feeds 8 FMAs.

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kWarps = 8;
constexpr int kVecPerWarp = 8;

struct AppendKernelArgs {
  const void *x;
  int batch, heads, n_new, capacity, cap16, bb;
  int vt;  // value role: codes in the pair-interleaved layout (merged atomically)
  const int32_t *seq_lens;
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  const float *centroids;
  const float *bounds;
  const float *diag;
  const float *sketch;
  int *error;
};

// shared layout (floats): [0,16) centroids | [16,32) bounds | QJL: S^T permuted
// [128][128] (entry (i, 4L+j) = S[L + 32j][i]) | per-warp residuals [8][128]
constexpr int kSmemTables = 32;
constexpr int kSmemSketch = kD * kD;
constexpr int kSmemResid = kWarps * kD * kVecPerWarp;

template <int BITS, bool ROT, bool QJL, bool BF16>
__global__ void __launch_bounds__(kWarps * 32, 2) append_tq_kernel(AppendKernelArgs a) {
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  float *s_cent = sm;
  float *s_bound = sm + 16;
  float *s_st = sm + kSmemTables;
  float *s_res = s_st + kSmemSketch;

  constexpr int L = 1 << BITS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < L) s_cent[tid] = a.centroids[tid];
  if (tid < L - 1) s_bound[tid] = a.bounds[tid];
  if (QJL) {
    // entry (i, 4L + m) = S[row][i] for the coordinate row = 8(L/2) + 2m + (L&1) whose sign
    // bit is bit L of sign word m, so one ballot per m yields the record's word m
    for (int e = tid; e < kD * kD; e += blockDim.x) {
      const int i = e >> 7, col = e & 127, l = col >> 2, m = col & 3;
      const int row = 8 * (l >> 1) + 2 * m + (l & 1);
      s_st[e] = __ldg(a.sketch + row * kD + i);
    }
  }
  float dg[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) dg[j] = ROT ? __ldg(a.diag + 4 * lane + j) : 1.f;
  __syncthreads();
  float bnd[L - 1];
#pragma unroll
  for (int k = 0; k < L - 1; ++k) bnd[k] = s_bound[k];

  const long long total = (long long)a.batch * a.heads * a.n_new;
  const long long groups = (total + kVecPerWarp - 1) / kVecPerWarp;
  float *my_res = s_res + warp * kD * kVecPerWarp;

  for (long long g = (long long)blockIdx.x * kWarps + warp; g < groups; g += (long long)gridDim.x * kWarps) {
    float nu_v[kVecPerWarp], rho_v[kVecPerWarp];
    long long slot_v[kVecPerWarp];
#pragma unroll
    for (int v = 0; v < kVecPerWarp; ++v) {
      const long long vec = g * kVecPerWarp + v;
      slot_v[v] = -1;
      nu_v[v] = 0.f;
      rho_v[v] = 0.f;
      if (vec >= total) {
        if (QJL) reinterpret_cast<float4 *>(my_res + v * kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int t = (int)(vec % a.n_new);
      const long long bh = vec / a.n_new;
      const int b = (int)(bh / a.heads);
      const int len = __ldg(a.seq_lens + b);
      const int pos = len + t;
      // a sequence whose new tokens would not all fit is skipped whole
      const bool ok = len >= 0 && len + a.n_new <= a.capacity;
      if (!ok && lane == 0) set_error(a.error, TQ_ERR_CAPACITY);
      const long long slot = bh * a.cap16 + pos;

      float x[4];
      load4(a.x, (size_t)vec * kD + 4 * lane, BF16, x);
      const float nu = sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]));
      float y[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) y[j] = (nu > 0.f) ? (x[j] / nu) * dg[j] : 0.f;
      if (ROT) wht128(y, lane);
      int idx[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int c = 0;
#pragma unroll
        for (int k = 0; k < L - 1; ++k) c += (y[j] >= bnd[k]) ? 1 : 0;
        idx[j] = c;
      }
      const uint32_t fa = (uint32_t)idx[0] | ((uint32_t)idx[1] << BITS);
      const uint32_t fb = (uint32_t)idx[2] | ((uint32_t)idx[3] << BITS);
      const uint32_t word = pack_slot_word<BITS>(fa, fb, lane);
      if (ok) {
        if (a.vt) {
          uint32_t *row = vt_row<BITS>(a.codes, slot, a.bb);
#pragma unroll
          for (int j = 0; j < 4; ++j) store_code_vt<BITS>(row, 4 * lane + j, (int)(slot & 1), (uint32_t)idx[j]);
        } else if (lane < 4 * BITS) {
          reinterpret_cast<uint32_t *>(rec_at(a.codes, slot, a.bb, BITS * kD / 8))[lane] = word;
        }
        if (!QJL && lane == 0) *rec_at(a.norms, slot, a.bb, 4) = nu;
      }
      if (QJL) {
        float r[4], rr = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          r[j] = y[j] - s_cent[idx[j]];
          rr += r[j] * r[j];
        }
        rr = warp_sum(rr);
        reinterpret_cast<float4 *>(my_res + v * kD)[lane] =
            (nu > 0.f) ? make_float4(r[0], r[1], r[2], r[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        nu_v[v] = nu;
        rho_v[v] = (nu > 0.f) ? nu * sqrtf(rr) : 0.f;
        slot_v[v] = ok ? slot : -1;
      }
    }
    if (QJL) {
      __syncwarp();
      float acc[kVecPerWarp][4];
#pragma unroll
      for (int v = 0; v < kVecPerWarp; ++v)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[v][j] = 0.f;
      const float4 *st4 = reinterpret_cast<const float4 *>(s_st);
      const float4 *rs4 = reinterpret_cast<const float4 *>(my_res);
#pragma unroll 1
      for (int i4 = 0; i4 < kD / 4; ++i4) {
        float4 r4[kVecPerWarp];
#pragma unroll
        for (int v = 0; v < kVecPerWarp; ++v) r4[v] = rs4[v * (kD / 4) + i4];  // broadcast
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const float4 s = st4[(4 * i4 + ii) * 32 + lane];
#pragma unroll
          for (int v = 0; v < kVecPerWarp; ++v) {
            const float rv = ii == 0 ? r4[v].x : ii == 1 ? r4[v].y : ii == 2 ? r4[v].z : r4[v].w;
            acc[v][0] = fmaf(s.x, rv, acc[v][0]);
            acc[v][1] = fmaf(s.y, rv, acc[v][1]);
            acc[v][2] = fmaf(s.z, rv, acc[v][2]);
            acc[v][3] = fmaf(s.w, rv, acc[v][3]);
          }
        }
      }
#pragma unroll
      for (int v = 0; v < kVecPerWarp; ++v) {
        uint32_t w0 = __ballot_sync(kFull, acc[v][0] >= 0.f);
        uint32_t w1 = __ballot_sync(kFull, acc[v][1] >= 0.f);
        uint32_t w2 = __ballot_sync(kFull, acc[v][2] >= 0.f);
        uint32_t w3 = __ballot_sync(kFull, acc[v][3] >= 0.f);
        const long long slot = slot_v[v];
        if (slot >= 0) {
          if (nu_v[v] == 0.f) w0 = w1 = w2 = w3 = 0xffffffffu;
          uint32_t *srec = reinterpret_cast<uint32_t *>(rec_at(a.signs, slot, a.bb, kD / 8));
          const uint32_t wsel = (lane == 0) ? w0 : (lane == 1) ? w1 : (lane == 2) ? w2 : w3;
          if (lane < 4) srec[lane] = wsel;
          if (lane == 0) {
            *rec_at(a.norms, slot, a.bb, 4) = nu_v[v];
            *rec_at(a.rnorms, slot, a.bb, 4) = rho_v[v];
          }
        }
      }
      __syncwarp();
    }
  }
}

int g_num_sms = 0;

int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 152;
  }
  return g_num_sms;
}

template <int BITS, bool ROT, bool QJL, bool BF16>
int launch_one(const AppendKernelArgs &k, long long total, cudaStream_t st) {
  const size_t smem = sizeof(float) * (kSmemTables + (QJL ? kSmemSketch + kSmemResid : 0));
  auto fn = append_tq_kernel<BITS, ROT, QJL, BF16>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  const long long groups = (total + kVecPerWarp - 1) / kVecPerWarp;
  long long blocks = (groups + kWarps - 1) / kWarps;
  const long long cap = 2LL * num_sms();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fn<<<(unsigned)blocks, kWarps * 32, smem, st>>>(k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <bool ROT, bool QJL, bool BF16>
int dispatch_bits(int bits, const AppendKernelArgs &k, long long total, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_one<1, ROT, QJL, BF16>(k, total, st);
    case 2: return launch_one<2, ROT, QJL, BF16>(k, total, st);
    case 3: return launch_one<3, ROT, QJL, BF16>(k, total, st);
    case 4: return launch_one<4, ROT, QJL, BF16>(k, total, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_append_tq(const AppendArgs &a, void *stream) {
  if (a.ctx) {
    int r = launch_append_bulk(a, a.ctx, stream);  // rotated roles, bf16 input
    if (r != TQ_ERR_UNSUPPORTED) return r;
    r = launch_append_tc(a, a.ctx, stream);  // rotated roles
    if (r != TQ_ERR_UNSUPPORTED) return r;
    r = launch_append2(a, a.ctx, stream);  // unrotated roles
    if (r != TQ_ERR_UNSUPPORTED) return r;
  }
  AppendKernelArgs k{};
  k.x = a.x;
  k.batch = a.batch;
  k.heads = a.heads;
  k.n_new = a.n_new;
  k.capacity = a.capacity;
  k.cap16 = a.cap16;
  k.bb = a.bb;
  k.vt = a.vt;
  k.seq_lens = a.seq_lens;
  k.codes = a.codes;
  k.norms = a.norms;
  k.signs = a.signs;
  k.rnorms = a.rnorms;
  k.centroids = a.centroids;
  k.bounds = a.bounds;
  k.diag = a.params->diag;
  k.sketch = a.params->sketch;
  k.error = a.error;
  const long long total = (long long)a.batch * a.heads * a.n_new;
  cudaStream_t st = (cudaStream_t)stream;
  const bool bf16 = a.dtype == TQ_BF16;
  const Role r = a.role;
  if (r.qjl && !r.rotate) return TQ_ERR_UNSUPPORTED;
  if (r.qjl) return bf16 ? dispatch_bits<true, true, true>(r.bits, k, total, st)
                         : dispatch_bits<true, true, false>(r.bits, k, total, st);
  if (r.rotate) return bf16 ? dispatch_bits<true, false, true>(r.bits, k, total, st)
                            : dispatch_bits<true, false, false>(r.bits, k, total, st);
  return bf16 ? dispatch_bits<false, false, true>(r.bits, k, total, st)
              : dispatch_bits<false, false, false>(r.bits, k, total, st);
}

}  // namespace tq
