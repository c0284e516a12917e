// Bulk append-quantise of bf16 vectors on the rotated roles (keys and values of
// KQV and QKQV): a warp-specialised persistent kernel, one CTA per SM.
//
// "Statistical Inference and Quality Measures of KV Cache Quantisations
// Inspired by TurboQuant", technical summary, "Quantisation schemes" (norm,
// randomised Walsh-Hadamard rotation, scalar Lloyd-Max codes; the (n-1)-bit
// vectors keep a 1-bit QJL sketch of their residual) and "Main contribution 1"
// (sign(S r) and rho = ||x|| ||r||). "KVQuant++", "Fast codebook lookup": a
// code is the count of boundaries at or below the coordinate.
//
// Per tile of 128 vectors:
// * one control thread (warp 0) loads the tile with one tensor-map copy of an
//   8 x 128 x 16 bf16 box (x viewed as [column block][row][8 columns]), which lands
//   exactly as the K-major core-matrix layout of the MMA's A operand (rows past
//   the end read as zeros), into a ring of
//   stages, and issues y = x (H D)^T on the tensor cores (bf16 inputs are
//   exact, the Hadamard-times-diagonal operand is +-1; fp32 accumulate in
//   tensor memory, accumulator column n = the coordinate stored at code offset
//   n); for sketched vectors, once the residuals are in tensor memory, it
//   issues z = S r in three fp16 passes (hi x hi, lo x hi, hi x lo) into the
//   columns y used;
// * two (sketched roles) or three groups of four epilogue warps take the tiles
//   in turn (one thread per vector = tensor-memory lane), so groups compute
//   while the others' MMAs run: ||y|| = sqrt(d) ||x|| gives the norm and the boundary scale, codes are
//   counted against the boundaries times ||y|| (no division), the residual
//   r = y / ||y|| - c[code], scaled by 2^10 and split into fp16 hi + lo, is
//   stored to tensor memory as the sketch MMA's A operand, and signs come out
//   of z 32 at a time. Signs within a bound on the dropped terms and the
//   accumulation error are recomputed in fp32 from the residual rebuilt from
//   its hi + lo parts, so a sign can differ from exact arithmetic only where
//   |z| is about 1e-6 or less.

#include <cuda.h>
#include <cuda_fp16.h>

#include "tq_ptx.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

constexpr int kTV = 128;                      // vectors per tile = MMA M
constexpr int kTileBytes = kTV * kD * 2;      // one bf16 tile (32 KB)
constexpr int kOpB = kD * kD * 2;             // one 16-bit 128 x 128 operand
constexpr float kRScaleB = 1024.f;            // residual scale for the fp16 split (|r| < 2)

// Epilogue groups of four warps (one tensor-memory slot each): sketched roles need 256
// columns a slot (y / z, residual hi, residual lo), so two fit in the 512 columns; the
// others need 128, so three groups share the SM -- three warps per scheduler to hide the
// tensor-memory and shared-memory latencies of the code search.
template <bool QJL>
constexpr int bulk_groups() { return QJL ? 2 : 3; }
template <bool QJL>
constexpr int bulk_threads() { return 32 * (1 + 4 * bulk_groups<QJL>()); }

template <bool QJL>
struct BulkGeo {
  static constexpr int NG = bulk_groups<QJL>();
  static constexpr int NS = QJL ? 3 : 4;                      // x stages
  static constexpr int x0 = 0;
  static constexpr int hd = NS * kTileBytes;                  // H D, bf16
  static constexpr int sk = hd + kOpB;                        // S hi, S lo (fp16)
  static constexpr int ent = QJL ? 16 : 8;                    // bytes of one cell-table entry
  static constexpr int ct = sk + (QJL ? 2 * kOpB : 0);        // cell table, [kCells][32 lanes] entries
  static constexpr int bar = ct + kCells * 32 * ent;          // barriers
  static constexpr int nbar = 2 * NS + 4 * NG + 2;
  static constexpr int total = bar + nbar * 8 + 16;
  static constexpr uint32_t tcols = 512u;                     // NG slots (a power of two >= NG slots)
  static constexpr uint32_t slot_cols = QJL ? 256u : 128u;    // Y / Z | R hi | R lo
};

struct BulkArgs {
  int batch, heads, n_new, capacity, cap16, bb;
  const int32_t *btab;  // paged caches (NULL: contiguous)
  int pool_blocks;
  long long total;
  const int32_t *seq_lens;
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  const float *sketch_perm;  // S in storage order, fp32 (rare-path exact signs)
  const uint16_t *hd_bf;   // DevParams::hadamard_bf
  const uint16_t *s_hl;    // DevParams::sketch_hl
  float sketch_rowmax;
  int *error;
  CellTable cells;  // the role's code-search table
  FastDiv div_new, div_heads;  // by n_new and by heads (vector indices are below 2^31)
};

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// D (TMEM) (+)= A (shared, descriptor) x B (shared, descriptor); one thread.
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// tcgen05.st of 16 columns without its wait, and the wait, which names the stored
// registers so that none of them is overwritten before the stores have read them
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::st.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}

// tcgen05.ld without its wait, and the wait, which names the loaded registers so
// that no use of them can be scheduled before it
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                 "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

__device__ __forceinline__ void split_pair_b(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Rare path, run by whole warps until no lane has a flagged sign left: each
// round every flagged lane recomputes one sign in fp32 from its residual,
// rebuilt from the hi + lo parts at r_hi / r_hi + 64 (storage order), against
// S in storage order (sperm[n][k] = S[coordinate of n][coordinate of k]).
// flag / sw hold the four sign words.
__device__ __forceinline__ void certify_rounds(uint32_t r_hi, const float *sperm, uint32_t (&flag)[4],
                                               uint32_t (&sw)[4]) {
  while (__any_sync(kFull, (flag[0] | flag[1] | flag[2] | flag[3]) != 0u)) {
    const bool has = (flag[0] | flag[1] | flag[2] | flag[3]) != 0u;
    const int c = flag[0] ? 0 : flag[1] ? 1 : flag[2] ? 2 : 3;
    const uint32_t fw = c == 0 ? flag[0] : c == 1 ? flag[1] : c == 2 ? flag[2] : flag[3];
    const int bit = has ? __ffs(fw) - 1 : 0;
    const float4 *row = reinterpret_cast<const float4 *>(sperm + (size_t)(32 * c + bit) * kD);
    // four partial sums: a short dependency chain (the rounding order is immaterial
    // at this precision)
    float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int chunk = 0; chunk < 4; ++chunk) {
      uint32_t hi[16], lo[16];
      tmem_ld16(r_hi + 16 * chunk, hi);  // warp-collective: every lane takes part
      tmem_ld16(r_hi + 64 + 16 * chunk, lo);
      if (has) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 sv = __ldg(row + 8 * chunk + q);
          const uint32_t h0 = hi[2 * q], l0 = lo[2 * q], h1 = hi[2 * q + 1], l1 = lo[2 * q + 1];
          z4[0] = fmaf(sv.x, (half_lo(h0) + half_lo(l0)) * (1.f / kRScaleB), z4[0]);
          z4[1] = fmaf(sv.y, (half_hi(h0) + half_hi(l0)) * (1.f / kRScaleB), z4[1]);
          z4[2] = fmaf(sv.z, (half_lo(h1) + half_lo(l1)) * (1.f / kRScaleB), z4[2]);
          z4[3] = fmaf(sv.w, (half_hi(h1) + half_hi(l1)) * (1.f / kRScaleB), z4[3]);
        }
      }
    }
    const float zz = (z4[0] + z4[1]) + (z4[2] + z4[3]);
    if (has) {
      const uint32_t m = 1u << bit;
      const uint32_t v = (zz >= 0.f) ? m : 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q == c) {
          flag[q] &= ~m;
          sw[q] = (sw[q] & ~m) | v;
        }
      }
    }
  }
}

template <int BITS, bool QJL, bool VT>
__global__ void __launch_bounds__(bulk_threads<QJL>(), 1)
    append_bulk_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ BulkArgs a) {
  using G = BulkGeo<QJL>;
  constexpr int NS = G::NS;
  constexpr int L = 1 << BITS, H = L / 2 - 1;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + G::bar);
  uint64_t *x_full = bars, *x_empty = bars + NS;
  constexpr int NG = G::NG;
  uint64_t *y_full = bars + 2 * NS, *r_full = y_full + NG, *z_full = r_full + NG, *s_empty = z_full + NG;
  uint64_t *op_bar = s_empty + NG, *drain = op_bar + 1;
  uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bars + G::nbar);
  volatile int *s_abort = reinterpret_cast<volatile int *>(s_taddr + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long ntiles = (a.total + kTV - 1) / kTV;
  // this CTA's tiles: blockIdx.x + k gridDim.x, k = 0 .. nloc - 1
  const long long nloc = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 1);
    }
    for (int g = 0; g < NG; ++g) {
      mbar_init(&y_full[g], 1);
      mbar_init(&r_full[g], 4);
      mbar_init(&z_full[g], 1);
      mbar_init(&s_empty[g], 4);
    }
    mbar_init(op_bar, 1);
    mbar_init(drain, 1);
    *s_abort = 0;
    mbar_fence_init();
    mbar_arrive_expect_tx(op_bar, (QJL ? 3 : 1) * kOpB);
    tma_load_1d(smem + G::hd, a.hd_bf, kOpB, op_bar);
    if (QJL) {
      tma_load_1d(smem + G::sk, a.s_hl, kOpB, op_bar);
      tma_load_1d(smem + G::sk + kOpB, a.s_hl + kD * kD, kOpB, op_bar);
    }
  }
  {  // the role's cell table, replicated per lane ([cell][lane]): a warp's lookups of one
     // coordinate hit 32 consecutive entries, whatever the cells
    unsigned char *tab = smem + G::ct;
    for (int i = tid; i < kCells * 32; i += bulk_threads<QJL>()) {
      const CellEntry &e = a.cells.e[i >> 5];
      if constexpr (QJL)
        *reinterpret_cast<float4 *>(tab + i * 16) = make_float4(__int_as_float(e.below), e.thr, e.c_lo, e.c_hi);
      else
        *reinterpret_cast<float2 *>(tab + i * 8) = make_float2(__int_as_float(e.below), e.thr);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_taddr), G::tcols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *s_taddr;

  if (warp == 0) {
    // ---------------- control thread: tile loads (tensor-map TMA) and MMA issue
    if (lane == 0) {
      auto load = [&](long long j) {  // local tile j into stage j % NS (the stage is free)
        const int s = (int)(j % NS);
        mbar_arrive_expect_tx(&x_full[s], kTileBytes);
        const int row0 = (int)((blockIdx.x + j * gridDim.x) * kTV);
        tma_load_3d(smem + G::x0 + s * kTileBytes, &xmap, 0, row0, 0, &x_full[s]);
      };
      long long loaded = 0;
      for (; loaded < NS && loaded < nloc; ++loaded) load(loaded);
      bool ok = mbar_wait_bounded(op_bar, 0, a.error);
      tc_fence_after_sync();
      constexpr uint32_t id_rot = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) |
                                  ((uint32_t)(128 >> 4) << 24);  // bf16 x bf16 -> f32, M = N = 128
      constexpr uint32_t id_sk = tc_idesc_f16_f32(128, 128);     // fp16 x fp16 -> f32
      const uint32_t sa_x = smem_u32(smem + G::x0), sa_h = smem_u32(smem + G::hd), sa_s = smem_u32(smem + G::sk);
      auto sketch = [&](long long k) -> bool {
        const int g = (int)(k % NG);
        if (!mbar_wait_bounded(&r_full[g], (uint32_t)((k / NG) & 1), a.error)) return false;  // (already complete)
        tc_fence_after_sync();
        const uint32_t d = tbase + G::slot_cols * g;
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t dh = tc_sdesc_kmajor(sa_s + 256 * ks, 128, 2048);
          const uint64_t dl = tc_sdesc_kmajor(sa_s + kOpB + 256 * ks, 128, 2048);
          tc_mma_f16_ts(d, d + 128 + 8 * ks, dh, id_sk, ks > 0);
          tc_mma_f16_ts(d, d + 192 + 8 * ks, dh, id_sk, true);
          tc_mma_f16_ts(d, d + 128 + 8 * ks, dl, id_sk, true);
        }
        tc_commit(smem_u32(&z_full[g]));
        return true;
      };
      // the rotation of tile k into slot k % NG (once the slot is free and the tile has landed),
      // then the refill of the stage tile k - 1 used (its rotation was issued one round ago)
      auto rotate = [&](long long k) -> bool {
        const int g = (int)(k % NG), s = (int)(k % NS);
        const uint32_t d = tbase + G::slot_cols * g;
#pragma unroll 1
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t da = tc_sdesc_kmajor(sa_x + s * kTileBytes + 4096 * ks, 2048, 128);
          const uint64_t db = tc_sdesc_kmajor(sa_h + 256 * ks, 128, 2048);
          tc_mma_ss(d, da, db, id_rot, ks > 0);
        }
        tc_commit(smem_u32(&x_empty[s]));
        tc_commit(smem_u32(&y_full[g]));
        if (k >= 1 && loaded < nloc) {
          const int sp = (int)((k - 1) % NS);
          if (!mbar_wait_bounded(&x_empty[sp], (uint32_t)(((k - 1) / NS) & 1), a.error)) return false;
          load(loaded++);
        }
        return true;
      };
      long long k = 0;
      if constexpr (QJL) {
        // two streams of work, issued in whichever order they become ready: the sketch of
        // the oldest rotated tile (once its group has stored the residuals) and the rotation
        // of the next tile (once its slot is free). Issuing a sketch only after the next
        // rotation's slot came free would make each group wait for the other's signs.
        long long kz = 0;  // next tile to sketch (kz < k)
        uint64_t t_idle = global_ns();
        while (ok && (k < nloc || kz < k) && !*s_abort) {
          bool moved = false;
          if (kz < k && mbar_test_wait(&r_full[kz % NG], (uint32_t)((kz / NG) & 1))) {
            ok = sketch(kz++);
            moved = true;
          }
          if (ok && k < nloc) {
            const int g = (int)(k % NG), s = (int)(k % NS);
            if ((k < NG || mbar_test_wait(&s_empty[g], (uint32_t)(((k / NG) - 1) & 1))) &&
                mbar_test_wait(&x_full[s], (uint32_t)((k / NS) & 1))) {
              tc_fence_after_sync();
              ok = rotate(k++);
              moved = true;
            }
          }
          if (moved) {
            t_idle = global_ns();
          } else if (global_ns() - t_idle > kWaitBudgetNs) {
            set_error(a.error, TQ_ERR_TIMEOUT);
            ok = false;
          } else {
            __nanosleep(32);
          }
        }
      } else {
        for (; ok && k < nloc && !*s_abort; ++k) {
          const int g = (int)(k % NG), s = (int)(k % NS);
          if (k >= NG && !mbar_wait_bounded(&s_empty[g], (uint32_t)(((k / NG) - 1) & 1), a.error)) ok = false;
          if (ok && !mbar_wait_bounded(&x_full[s], (uint32_t)((k / NS) & 1), a.error)) ok = false;
          if (!ok) break;
          tc_fence_after_sync();
          ok = rotate(k);
        }
      }
      if (!ok) *s_abort = 1;
      // copies that landed for nobody (an abort) must not outlive the CTA
      for (long long j = k; j < loaded; ++j) mbar_wait_bounded(&x_full[j % NS], (uint32_t)((j / NS) & 1), a.error);
    }
  } else {
    // ---------------- epilogue: group g (four warps, one thread per vector) takes local tiles k = g (mod NG)
    const int g = (warp - 1) >> 2, qd = warp & 3;
    const int row = 32 * qd + lane;  // vector within the tile = TMEM lane
    const uint32_t tslot = tbase + G::slot_cols * g + ((uint32_t)(32 * qd) << 16);
    const unsigned char *tab = smem + G::ct + lane * G::ent;  // this lane's copy of the cell table
    const float smax = a.sketch_rowmax;
    // sequence lengths are loaded a tile ahead: the L2 round trip of the current tile's length
    // would otherwise stall the warp at the top of every tile
    auto len_of = [&](long long kk) -> int {
      const long long v = (blockIdx.x + kk * gridDim.x) * kTV + row;
      return v < a.total ? __ldg(a.seq_lens + fast_div(fast_div((uint32_t)v, a.div_new), a.div_heads)) : 0;
    };
    int len_next = (g < nloc) ? len_of(g) : 0;
    for (long long k = g; k < nloc; k += NG) {
      const int par = (int)((k / NG) & 1);
      const long long tile = blockIdx.x + k * gridDim.x;
      const long long vec = tile * kTV + row;
      const int len = len_next;
      if (k + NG < nloc) len_next = len_of(k + NG);
      long long slot = -1;
      if (vec < a.total) {
        const uint32_t bh32 = fast_div((uint32_t)vec, a.div_new);
        const int t = (int)((uint32_t)vec - bh32 * (uint32_t)a.n_new);
        const long long bh = bh32;
        if (len >= 0 && len + a.n_new <= a.capacity) slot = phys_slot(a.btab, a.pool_blocks, bh * a.cap16 + len + t, a.error);
        else if (t == 0) set_error(a.error, TQ_ERR_CAPACITY);  // the sequence is skipped whole
      }
      // value codes: is the other token of this token's pair (slot ^ 1) the neighbouring lane's?
      bool paired = false;
      if (VT) {
        const long long ps = ((long long)__shfl_xor_sync(kFull, (int)(slot >> 32), 1) << 32) |
                             (uint32_t)__shfl_xor_sync(kFull, (int)(uint32_t)slot, 1);
        paired = slot >= 0 && ps >= 0 && ps == (slot ^ 1);
      }
      if (*s_abort || !__all_sync(kFull, mbar_wait_bounded(&y_full[g], (uint32_t)par, a.error))) {
        *s_abort = 1;
        break;
      }
      tc_fence_after_sync();
      // pass 1: ||y||^2 = d ||x||^2 (each chunk's load overlaps the previous chunk's sums)
      float ss = 0.f;
      {
        uint32_t ya[32], yb[32];
        __syncwarp();
        tmem_ld32_async(tslot, ya);
        tmem_ld_wait(ya);
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          tmem_ld32_async(tslot + 32 * (c + 1), yb);
#pragma unroll
          for (int j = 0; j < 32; ++j) ss = fmaf(__uint_as_float(ya[j]), __uint_as_float(ya[j]), ss);
          tmem_ld_wait(yb);
          if (c + 2 < 4) tmem_ld32_async(tslot + 32 * (c + 2), ya);
#pragma unroll
          for (int j = 0; j < 32; ++j) ss = fmaf(__uint_as_float(yb[j]), __uint_as_float(yb[j]), ss);
          if (c + 2 < 4) tmem_ld_wait(ya);
        }
      }
      const float sv = ss > 0.f ? sqrtf(ss) : 1.f;  // sqrt(d) ||x||, the boundary scale
      const float inv = ss > 0.f ? kRScaleB / sv : 0.f;
      const float A = a.cells.inv2u / sv;  // t = sat(y A + 1/2) places y on the cell grid
      // pass 2: codes and residuals of chunk c (32 storage offsets)
      float rr = 0.f;
      uint32_t *crec = reinterpret_cast<uint32_t *>(rec_at(a.codes, slot >= 0 ? slot : 0, a.bb, BITS * kD / 8));
      auto chunk_codes = [&](uint32_t (&yz)[32], int c) {
        // key records: BITS words per chunk in code-offset order; value codes: the chunk's
        // 32 fields of the pair row (2 BITS words), this token's half only
        constexpr int NW = VT ? 2 * BITS : BITS;
        uint32_t word[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) word[w] = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          // the code: the cell of y (one fused multiply-add, saturated; the cell index lands
          // in the low mantissa bits of t 63 stride + 1.5 2^23, already times the entry
          // stride), then the one boundary the cell may hold
          const float yv = __uint_as_float(yz[j]);
          const float t = __saturatef(fmaf(yv, A, 0.5f));
          constexpr float kMul = 63.f * (QJL ? 512.f : 256.f);
          constexpr uint32_t kMask = QJL ? 0x7E00u : 0x3F00u;
          const uint32_t key = __float_as_uint(fmaf(t, kMul, 12582912.f)) & kMask;
          uint32_t code;
          float cneg = 0.f;
          if constexpr (QJL) {
            const float4 e = *reinterpret_cast<const float4 *>(tab + key);
            const bool up = yv >= e.y * sv;
            code = (uint32_t)__float_as_int(e.x) + (up ? 1u : 0u);
            cneg = -(up ? e.w : e.z);
          } else {
            const float2 e = *reinterpret_cast<const float2 *>(tab + key);
            code = (uint32_t)__float_as_int(e.x) + (yv >= e.y * sv ? 1u : 0u);
          }
          const int off = VT ? 2 * BITS * (16 * (j & 1) + (j >> 1)) : BITS * j;
          word[off >> 5] |= code << (off & 31);
          if ((off & 31) + BITS > 32) word[(off >> 5) + 1] |= code >> (32 - (off & 31));
          if (QJL) {
            const float r = fmaf(__uint_as_float(yz[j]), inv, cneg);  // r 2^10
            rr = fmaf(r, r, rr);
            yz[j] = __float_as_uint(r);
          }
        }
        if constexpr (VT) {
          const int half = (int)(slot & 1);
          if (half) {  // this token's codes go to the high half of each field
#pragma unroll
            for (int i = NW - 1; i > 0; --i) word[i] = (word[i] << BITS) | (word[i - 1] >> (32 - BITS));
            word[0] <<= BITS;
          }
          vt_store_chunk<BITS>(vt_row<BITS>(a.codes, slot >= 0 ? slot : 0, a.bb), c, word, half, paired,
                               slot >= 0);
        } else if (slot >= 0) {
#pragma unroll
          for (int w = 0; w < BITS; ++w) crec[BITS * c + w] = word[w];
        }
        if (QJL) {
          uint32_t rh[16], rl[16];
#pragma unroll
          for (int p = 0; p < 16; ++p)
            split_pair_b(__uint_as_float(yz[2 * p]), __uint_as_float(yz[2 * p + 1]), rh[p], rl[p]);
          __syncwarp();
          tmem_st16_async(tslot + 128 + 16 * c, rh);
          tmem_st16_async(tslot + 192 + 16 * c, rl);
          tmem_st_wait(rh, rl);
        }
      };
      {
        uint32_t ya[32], yb[32];
        __syncwarp();
        tmem_ld32_async(tslot, ya);
        tmem_ld_wait(ya);
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          tmem_ld32_async(tslot + 32 * (c + 1), yb);
          chunk_codes(ya, c);
          tmem_ld_wait(yb);
          if (c + 2 < 4) tmem_ld32_async(tslot + 32 * (c + 2), ya);
          chunk_codes(yb, c + 1);
          if (c + 2 < 4) tmem_ld_wait(ya);
        }
      }
      const float nu = (ss > 0.f) ? sv * 0.08838834764831845f : 0.f;  // ||y|| / sqrt(d)
      if (slot >= 0) *rec_at(a.norms, slot, a.bb, 4) = nu;
      if constexpr (QJL) {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&r_full[g]);
        if (!__all_sync(kFull, mbar_wait_bounded(&z_full[g], (uint32_t)par, a.error))) {
          *s_abort = 1;
          break;
        }
        tc_fence_after_sync();
        // dropped terms + accumulation error of z' = 2^10 S r
        const float E = 0x1p-16f * smax * sqrtf(rr) + 0x1p-20f * smax;
        uint32_t sw[4], flag[4];
        // sign bits by funnel shifts (bit j of a word <- the sign bit of z[j]; inverted at
        // the end, so z = -0 reads as negative, but |z| = 0 is flagged and recomputed)
        auto chunk_signs = [&](const uint32_t (&z)[32], uint32_t &wv, uint32_t &fv) {
          uint32_t ns = 0u, nf = 0u;
#pragma unroll
          for (int bit = 31; bit >= 0; --bit) {
            ns = __funnelshift_l(z[bit], ns, 1);
            nf = __funnelshift_l(__float_as_uint(E - fabsf(__uint_as_float(z[bit]))), nf, 1);
          }
          wv = ~ns;  // z >= 0
          fv = ~nf;  // |z| <= E
        };
        {
          uint32_t za[32], zb[32];
          __syncwarp();
          tmem_ld32_async(tslot, za);
          tmem_ld_wait(za);
          tmem_ld32_async(tslot + 32, zb);
          chunk_signs(za, sw[0], flag[0]);
          tmem_ld_wait(zb);
          tmem_ld32_async(tslot + 64, za);
          chunk_signs(zb, sw[1], flag[1]);
          tmem_ld_wait(za);
          tmem_ld32_async(tslot + 96, zb);
          chunk_signs(za, sw[2], flag[2]);
          tmem_ld_wait(zb);
          chunk_signs(zb, sw[3], flag[3]);
        }
        certify_rounds(tslot + 128, a.sketch_perm, flag, sw);
        if (slot >= 0) {
          if (ss == 0.f) sw[0] = sw[1] = sw[2] = sw[3] = 0xffffffffu;  // a zero vector: every sign set, rho = 0
          *reinterpret_cast<uint4 *>(rec_at(a.signs, slot, a.bb, kD / 8)) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
          *rec_at(a.rnorms, slot, a.bb, 4) = (ss > 0.f) ? nu * sqrtf(rr) * (1.f / kRScaleB) : 0.f;
        }
      }
      // this warp is done with the slot's tensor memory
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[g]);
    }
  }

  // ---------------- teardown: no tensor-core work in flight, then free TMEM
  __syncthreads();
  if (warp == 0) {
    if (*s_abort && lane == 0) {  // a last, bounded chance for MMAs still running
      tc_commit(smem_u32(drain));
      mbar_wait_bounded(drain, 0, a.error);
    }
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tbase, G::tcols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int g_sms_bulk = 0;

template <int BITS, bool QJL, bool VT>
int go_bulk(const CUtensorMap &map, const BulkArgs &k, long long ntiles, cudaStream_t st) {
  if (g_sms_bulk == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_bulk, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms_bulk <= 0) g_sms_bulk = 152;
  }
  using G = BulkGeo<QJL>;
  auto fn = append_bulk_kernel<BITS, QJL, VT>;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, G::total) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_done = true;
  }
  long long blocks = ntiles < g_sms_bulk ? ntiles : g_sms_bulk;
  if (blocks < 1) blocks = 1;
  fn<<<(unsigned)blocks, bulk_threads<QJL>(), G::total, st>>>(map, k);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

// Bulk append of bf16 vectors on rotated roles; TQ_ERR_UNSUPPORTED when it does not apply.
int launch_append_bulk(const AppendArgs &a, const tq_ctx *ctx, void *stream) {
  if (!a.role.rotate || a.dtype != TQ_BF16 || a.role.bits < 1 || a.role.bits > 4 || (a.role.qjl && a.role.bits > 3))
    return TQ_ERR_UNSUPPORTED;
  // the rotation operand here is the exact +-1 Walsh-Hadamard one; a dense rotation takes the
  // fp16 hi / lo passes of the tensor-core kernel for fp32 inputs
  if (ctx->rotation != TQ_ROTATION_WHT) return TQ_ERR_UNSUPPORTED;
  if (a.side_rank) return TQ_ERR_UNSUPPORTED;  // keys with side codes: the tensor-core kernel below
  const long long total = (long long)a.batch * a.heads * a.n_new;
  if (total < 2LL * kTV || total > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return TQ_ERR_UNSUPPORTED;
  // x, a [total][128] bf16 matrix, seen as [16 column blocks][total rows][8 columns] (strides 16 B
  // and 256 B): one box of 8 x 128 x 16 lands a whole 128-vector tile as the MMA's K-major A
  // operand, 16 column blocks of 16 core matrices each, in a single copy
  CUtensorMap map;
  const cuuint64_t dims[3] = {8, (cuuint64_t)total, (cuuint64_t)kD / 8};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 16};
  const cuuint32_t box[3] = {8, (cuuint32_t)kTV, (cuuint32_t)kD / 8};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TQ_ERR_UNSUPPORTED;
  BulkArgs k{};
  k.batch = a.batch;
  k.heads = a.heads;
  k.n_new = a.n_new;
  k.capacity = a.capacity;
  k.cap16 = a.cap16;
  k.bb = a.bb;
  k.btab = a.btab;
  k.pool_blocks = a.pool_blocks;
  k.total = total;
  k.seq_lens = a.seq_lens;
  k.codes = a.codes;
  k.norms = a.norms;
  k.signs = a.signs;
  k.rnorms = a.rnorms;
  k.sketch_perm = ctx->dparams->sketch_perm;
  k.hd_bf = ctx->dparams->hadamard_bf;
  k.s_hl = ctx->dparams->sketch_hl;
  k.sketch_rowmax = ctx->sketch_rowmax;
  k.error = a.error;
  const bool is_k = a.centroids == ctx->dparams->k_centroids;
  k.cells = ctx->cells[is_k ? 0 : 1];
  k.div_new = make_fastdiv((uint32_t)a.n_new);
  k.div_heads = make_fastdiv((uint32_t)a.heads);
  if (k.cells.stride != (a.role.qjl ? 512 : 256)) return TQ_ERR_UNSUPPORTED;
  const long long ntiles = (total + kTV - 1) / kTV;
  cudaStream_t st = (cudaStream_t)stream;
  if (a.role.qjl && a.vt) {
    switch (a.role.bits) {
      case 1: return go_bulk<1, true, true>(map, k, ntiles, st);
      case 2: return go_bulk<2, true, true>(map, k, ntiles, st);
      case 3: return go_bulk<3, true, true>(map, k, ntiles, st);
      default: return TQ_ERR_UNSUPPORTED;
    }
  }
  if (a.role.qjl) {
    switch (a.role.bits) {
      case 1: return go_bulk<1, true, false>(map, k, ntiles, st);
      case 2: return go_bulk<2, true, false>(map, k, ntiles, st);
      case 3: return go_bulk<3, true, false>(map, k, ntiles, st);
      default: return TQ_ERR_UNSUPPORTED;
    }
  }
  if (a.vt) {
    switch (a.role.bits) {
      case 1: return go_bulk<1, false, true>(map, k, ntiles, st);
      case 2: return go_bulk<2, false, true>(map, k, ntiles, st);
      case 3: return go_bulk<3, false, true>(map, k, ntiles, st);
      case 4: return go_bulk<4, false, true>(map, k, ntiles, st);
      default: return TQ_ERR_UNSUPPORTED;
    }
  }
  switch (a.role.bits) {
    case 1: return go_bulk<1, false, false>(map, k, ntiles, st);
    case 2: return go_bulk<2, false, false>(map, k, ntiles, st);
    case 3: return go_bulk<3, false, false>(map, k, ntiles, st);
    case 4: return go_bulk<4, false, false>(map, k, ntiles, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

}  // namespace tq
