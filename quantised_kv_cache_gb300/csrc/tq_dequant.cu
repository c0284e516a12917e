// Dequantise ("decompress", "KVQuant++" forum post, "Deployment and use"):
//   x_hat = nu D H c[idx]  (+ rho sqrt(pi/2)/m D H S^T sigma for sketched vectors)
// The sketch term is the QJL reconstruction of the residual ("Statistical
// Inference ... Inspired by TurboQuant", technical summary, "Main contribution
// 1"). One warp per vector, lane L owning coordinates 4L..4L+3. Used for
// reconstruction-quality measurements and tests, not on the decode path.

#include "tq_device.cuh"

namespace tq {
namespace {

struct DequantKernelArgs {
  const uint8_t *codes;
  const float *norms;
  const uint8_t *signs;
  const float *rnorms;
  int bb, cap16;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  int *error;
  int vt;  // value codes: pair-interleaved layout
  int batch, heads, capacity, t0, t1;
  const float *centroids;
  const float *diag;
  const float *sketch;
  float *out;
  const float *rot;  // dense rotation M (x = M^T y), or nullptr (Walsh-Hadamard)
  // key side codes (side_rank > 0): x_hat += U z_hat, U [heads][d][rank] as given
  const uint16_t *side;
  const float *side_u;
  int side_rank;
};

template <int BITS, bool ROT, bool QJL>
__global__ void __launch_bounds__(256) dequant_tq_kernel(DequantKernelArgs a) {
  __shared__ float s_c[16];
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < (1 << BITS)) s_c[threadIdx.x] = a.centroids[threadIdx.x];
  __syncthreads();
  const int n = a.t1 - a.t0;
  const long long total = (long long)a.batch * a.heads * n;
  const long long vec = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (vec >= total) return;
  const long long bh = vec / n;
  const int t = a.t0 + (int)(vec % n);
  const long long slot = phys_slot(a.btab, a.pool_blocks, (long long)bh * a.cap16 + t, a.error);
  if (slot < 0) {  // an unmapped block (the error word says so): zeros
    reinterpret_cast<float4 *>(a.out + (size_t)vec * kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  uint32_t code[4];
  if (a.vt) lane_codes_vt<BITS>(a.codes, slot, a.bb, lane, code);
  else lane_codes<BITS>(reinterpret_cast<const uint32_t *>(rec_at(a.codes, slot, a.bb, BITS * 16)), lane, code);
  const float nu = __ldg(rec_at(a.norms, slot, a.bb, 4));
  float y[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) y[j] = nu * s_c[code[j]];
  if (QJL) {
    const uint32_t *srec = reinterpret_cast<const uint32_t *>(rec_at(a.signs, slot, a.bb, 16));
    uint32_t sw[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) sw[w] = __ldg(srec + w);
    float r[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < kD; ++k) {
      // coordinate k = 8n + 2t + e sits at sign word t, bit 2n + e
      const int word = (k >> 1) & 3, bit = 2 * (k >> 3) + (k & 1);
      const float sg = ((sw[word] >> bit) & 1u) ? 1.f : -1.f;
      const float4 s = __ldg(reinterpret_cast<const float4 *>(a.sketch + k * kD) + lane);
      r[0] = fmaf(s.x, sg, r[0]);
      r[1] = fmaf(s.y, sg, r[1]);
      r[2] = fmaf(s.z, sg, r[2]);
      r[3] = fmaf(s.w, sg, r[3]);
    }
    const float rho = __ldg(rec_at(a.rnorms, slot, a.bb, 4)) * (kSqrtHalfPi / kD);
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = fmaf(rho, r[j], y[j]);
  }
  if (ROT && a.rot) {
    matvec_t_warp(a.rot, y, lane);
  } else if (ROT) {
    wht128(y, lane);
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] *= __ldg(a.diag + 4 * lane + j);
  }
  if (a.side_rank) {
    const uint16_t *zp = rec_at(a.side, slot, a.bb, 2 * a.side_rank);
    const float *U = a.side_u + (size_t)(bh % a.heads) * kD * a.side_rank;
    for (int k = 0; k < a.side_rank; ++k) {
      const float z = __half2float(__ushort_as_half(zp[k]));
#pragma unroll
      for (int j = 0; j < 4; ++j) y[j] = fmaf(__ldg(U + (4 * lane + j) * a.side_rank + k), z, y[j]);
    }
  }
  reinterpret_cast<float4 *>(a.out + (size_t)vec * kD)[lane] = make_float4(y[0], y[1], y[2], y[3]);
}

template <bool ROT, bool QJL>
int go(int bits, const DequantKernelArgs &k, unsigned blocks, cudaStream_t st) {
  switch (bits) {
    case 1: dequant_tq_kernel<1, ROT, QJL><<<blocks, 256, 0, st>>>(k); break;
    case 2: dequant_tq_kernel<2, ROT, QJL><<<blocks, 256, 0, st>>>(k); break;
    case 3: dequant_tq_kernel<3, ROT, QJL><<<blocks, 256, 0, st>>>(k); break;
    case 4: dequant_tq_kernel<4, ROT, QJL><<<blocks, 256, 0, st>>>(k); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

int launch_dequant_tq(const DequantArgs &a, void *stream) {
  DequantKernelArgs k{a.codes, a.norms, a.signs, a.rnorms, a.bb, a.cap16, a.btab, a.pool_blocks, a.error, a.vt,
                      a.batch, a.heads, a.capacity, a.t0, a.t1, a.centroids, a.params->diag, a.params->sketch,
                      a.out, a.rot, a.side, a.side_u, a.side_rank};
  const long long total = (long long)a.batch * a.heads * (a.t1 - a.t0);
  const unsigned blocks = (unsigned)((total + 7) / 8);
  cudaStream_t st = (cudaStream_t)stream;
  if (a.role.qjl) return a.role.rotate ? go<true, true>(a.role.bits, k, blocks, st) : TQ_ERR_UNSUPPORTED;
  return a.role.rotate ? go<true, false>(a.role.bits, k, blocks, st) : go<false, false>(a.role.bits, k, blocks, st);
}

}  // namespace tq
