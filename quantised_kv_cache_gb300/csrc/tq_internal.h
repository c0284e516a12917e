// Internal declarations shared by the host code and the CUDA translation units
// of libtq. Not part of the ABI (include/tq.h is).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kD = 128;          // the head dimension this build implements
constexpr int kMaxLevels = 16;   // 4-bit codebooks at most
constexpr int kMaxGroup = 8;     // query heads per KV head handled by one CTA
constexpr int kPartialFloats = 260;  // m, l, acc[128], sign_acc[128], 2 pad
constexpr int kDecodeTile = 64;      // tokens per tile of the TMA decode kernels
constexpr int kPersistGroups = 4;    // partial records per (CTA, head) of the persistent decode (one CTA per SM)

// Device-resident parameter block of a context (one cudaMalloc).
struct DevParams {
  float k_centroids[kMaxLevels];
  float k_bounds[kMaxLevels];  // 2^b - 1 used
  float v_centroids[kMaxLevels];
  float v_bounds[kMaxLevels];
  float diag[kD];              // D as +/-1.0f
  float sketch[kD * kD];       // S, row-major [row][col]
  int error;                   // sticky device error word (a tq_status)
  int pad[3];
  // tensor-core B operands in the K-major core-matrix layout, set on the device at
  // context creation (16-byte aligned): the unnormalised Hadamard matrix times the
  // seeded diagonal, H D, with its rows in code-storage order, and S as fp16 hi + lo parts (hi = fp16(S),
  // lo = fp16(S - hi)) with rows and columns in storage order
  uint16_t hadamard_b[kD * kD];
  uint16_t sketch_hl[2 * kD * kD];
  // H D again, as bf16 (+-1 is exact in both formats), for bf16 inputs
  uint16_t hadamard_bf[kD * kD];
  // S with rows and columns in storage order, fp32: sketch_perm[n][k] = S[coord(n)][coord(k)]
  float sketch_perm[kD * kD];
  // S transposed for the warp-per-vector append: entry (i, 4L + m) = S[8(L/2) + 2m + (L&1)][i]
  float sketch_tp[kD * kD];
  // the dense rotation (contexts set to TQ_ROTATION_DENSE; y = M u): M and M^T row-major, and
  // sqrt(d) M as fp16 hi + lo tensor-core B operands (rows in code-storage order, K-major core
  // matrices), like hadamard_b
  float rot[kD * kD];
  float rot_t[kD * kD];
  uint16_t rot_hl[2 * kD * kD];
};
// fills DevParams::hadamard_b and DevParams::sketch_hl (stream order)
int launch_operand_prep(DevParams *dp, void *stream);
// fills DevParams::sketch_tp (stream order)
int launch_sketch_transpose(DevParams *dp, void *stream);
// fills DevParams::rot_hl from DevParams::rot (stream order)
int launch_rotation_prep(DevParams *dp, void *stream);
// the dense rotation drawn for `seed` (row-major d x d, y = M u), in double
bool draw_dense_rotation(uint64_t seed, int d, double *M);

// Unsigned 32-bit division by a divisor fixed for a launch, as one multiply-high, one
// subtraction, one add and two shifts (Granlund and Montgomery, "Division by Invariant Integers
// using Multiplication", 1994, section 4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0),
// t = umulhi(m, n), for every 32-bit n.
struct FastDiv {
  uint32_t d = 1, m = 1, s1 = 0, s2 = 0;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  if (d == 0) d = 1;
  int l = 0;
  while (l < 32 && (1ull << l) < d) ++l;
  f.d = d;
  f.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  f.s1 = l < 1 ? (uint32_t)l : 1u;
  f.s2 = l > 1 ? (uint32_t)(l - 1) : 0u;
  return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}
#endif

struct Role {
  int bits = 0;
  bool rotate = false;
  bool qjl = false;
};

// Blocked record layout of the TQ schemes: 16-token blocks of `bb` bytes; plane p holds
// tok[p] bytes per token at byte offset off[p] of its block (tq_plane order).
constexpr int kBlockTokens = 16;
struct RecLayout {
  int bb = 0;
  int off[TQ_NUM_PLANES] = {};
  int tok[TQ_NUM_PLANES] = {};
};

// Byte offset of token slot `slot` = sequence-head * cap16 + t (cap16 = the capacity rounded up
// to whole blocks) in a plane of the blocked layout, from that plane's offset in block 0.
__host__ __device__ __forceinline__ long long rec_off(long long slot, int bb, int tok) {
  return (slot >> 4) * (long long)bb + (long long)(slot & 15) * tok;
}
template <typename T>
__host__ __device__ __forceinline__ T *rec_at(T *plane, long long slot, int bb, int tok) {
  return reinterpret_cast<T *>(reinterpret_cast<uintptr_t>(plane) + rec_off(slot, bb, tok));
}
__host__ __device__ __forceinline__ int cap16_of(int capacity) { return (capacity + 15) & ~15; }

// Code search by cells (the bulk append). A coordinate y of a vector whose boundary scale is
// s (= ||y||) maps to t = sat(y * inv2u / s + 1/2) in [0, 1] and to cell
// k = floor(round(t * 63 * stride) / stride) (stride 256 for 8-byte table entries, 512 for
// 16-byte ones), i.e. t * 63 in [k - 1/(2 stride), k + 1 - 1/(2 stride)). The grid is chosen on
// the host so that no cell holds two boundaries and every boundary lies at least
// kCellMargin cells from a cell edge; the code is then below[k] + [y >= fl(thr[k] * s)]
// -- the count of boundaries b_j with y >= fl(b_j * s), found with one lookup and one compare.
constexpr int kCells = 64;
constexpr double kCellMargin = 0.05;
struct CellEntry {
  int below;   // boundaries entirely below the cell
  float thr;   // the boundary inside the cell (unit domain), or +inf
  float c_lo;  // 2^10 c[below], 2^10 c[below + 1]: the centroids of the two possible codes
  float c_hi;  //   (sketched roles: the residual y / s - c[code])
};
struct CellTable {
  CellEntry e[kCells];
  float inv2u;  // 1 / (2U): the cells cover the unit-domain line [-U, U]
  int stride;   // 256 or 512 (see above)
};
// Build the table for sorted float32 boundaries (2^bits - 1 of them); false if no grid of
// the searched widths satisfies the margin (it always does for the Lloyd-Max boundaries).
bool build_cell_table(const float *bounds, const float *centroids, int bits, int stride, CellTable *out);

}  // namespace tq

struct tq_ctx {
  int d = 0;
  int bits = 0;
  int scheme = 0;
  uint64_t seed = 0;
  int device = 0;
  int num_sms = 0;  // of `device`
  tq::Role k, v;
  tq::RecLayout lay;  // TQ schemes
  // KIVI options
  int kivi_group = 32;
  int kivi_window = 128;
  int kivi_k_per_channel = 1;
  int kivi_v_per_token = 1;
  // host copies of the float32 parameters
  float k_centroids[tq::kMaxLevels] = {};
  float k_bounds[tq::kMaxLevels] = {};
  float v_centroids[tq::kMaxLevels] = {};
  float v_bounds[tq::kMaxLevels] = {};
  int8_t diag[tq::kD] = {};
  float *sketch = nullptr;  // host, d*d
  float sketch_rowmax = 0.f;  // an upper bound of max_j ||S_j||
  tq::CellTable cells[2];     // bulk append code search (keys, values)
  int rotation = TQ_ROTATION_WHT;  // tq_rotation of the rotated roles
  // key side codes (tq_set_side_basis): rank, KV heads, device bases [heads][d][rank] as
  // given (natural coordinates), rotated (natural coordinate order of the rotated domain)
  // and rotated in code-storage order (row n = the coordinate stored at code offset n)
  int side_rank = 0, side_heads = 0;
  float *side_u = nullptr, *side_ur = nullptr, *side_urs = nullptr;
  tq::DevParams *dparams = nullptr;
  // a library-owned stream and two events: the key and value appends of one call
  // run concurrently (fork / join on the caller's stream)
  void *side_stream = nullptr, *ev_fork = nullptr, *ev_join = nullptr;
  // optional CUDA events recorded around the decode / append kernels
  void *prof_decode_start = nullptr, *prof_decode_stop = nullptr;
  void *prof_append_start = nullptr, *prof_append_stop = nullptr;
};

namespace tq {

// Launchers implemented in the .cu translation units. All return a tq_status.
struct AppendArgs {
  const void *x;         // [batch][heads][n_new][d]
  int dtype;             // TQ_F32 / TQ_BF16
  int batch, heads, n_new, capacity;
  const int32_t *seq_lens;
  // plane bases (block 0) of this role in the blocked records; slot = sequence-head * cap16 + t
  uint8_t *codes;
  float *norms;
  uint8_t *signs;
  float *rnorms;
  int bb, cap16;
  const int32_t *btab;  // paged caches: the block table (NULL: contiguous)
  int pool_blocks;
  int vt;  // 1: the value role (codes in the pair-interleaved layout)
  // key side codes (keys of a context with tq_set_side_basis; 0 / nullptr otherwise): the
  // side plane base, the bases in the code coordinates, natural and code-storage order
  int side_rank;
  uint16_t *side;
  const float *side_ur, *side_urs;
  Role role;
  const float *centroids;  // device pointers into DevParams
  const float *bounds;
  const DevParams *params;
  int *error;
  const tq_ctx *ctx;
};
int launch_append_tq(const AppendArgs &a, void *stream);

// Launch `fn` so that it may overlap the tail of the previous kernel in the stream
// (programmatic stream serialization); `fn` must call pdl_wait() before it reads
// anything earlier work writes. Plain stream order when `overlap` is false.
template <typename... P, typename... A>
inline cudaError_t launch_overlapped(bool overlap, void (*fn)(P...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, A &&...args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, static_cast<A &&>(args)...);
}
// thread-per-vector append for vectors without a sketch; TQ_ERR_UNSUPPORTED otherwise
int launch_append2(const AppendArgs &a, const tq_ctx *ctx, void *stream);
// thread-per-vector append of rotated vectors with the rotation and the QJL sketch on
// tcgen05 tensor cores; TQ_ERR_UNSUPPORTED otherwise
int launch_append_tc(const AppendArgs &a, const tq_ctx *ctx, void *stream);
// warp-specialised persistent append of bf16 vectors on rotated roles (tensor-map loads,
// bf16 MMA rotation); TQ_ERR_UNSUPPORTED otherwise
int launch_append_bulk(const AppendArgs &a, const tq_ctx *ctx, void *stream);
// warp-per-vector append of the keys and values of one call in a single launch, for calls
// of at most kSmallAppendMax vectors per tensor (TQ schemes)
constexpr long long kSmallAppendMax = 8192;
bool append_small_fits(const tq_ctx *ctx, long long vectors);
int launch_append_small(const AppendArgs &k, const AppendArgs &v, const tq_ctx *ctx, void *stream);

struct DecodeArgs {
  const tq_ctx *ctx;
  const tq_cache *cache;
  const void *q;
  int q_dtype;
  int batch, heads_q, heads_kv, max_len, splits, chunk;
  const int32_t *seq_lens;
  float *qprep;     // [batch][heads_q][2][d]
  int32_t *tile_prefix;  // [batch + 1] decode tiles before each batch (computed by the query prep)
  float *partials;  // split-K: [batch][heads_q][splits][kPartialFloats]; persistent: [ctas + units][kPersistGroups][...]
  float *out;
};
int launch_decode_tq(const DecodeArgs &a, void *stream);
// TMA-staged, tensor-core decode for one query head per KV head; returns
// TQ_ERR_UNSUPPORTED when the request falls outside what it covers.
// *persist_ctas receives the persistent grid size, or 0 when the split-K kernel ran.
int launch_decode2_g1(const DecodeArgs &a, int *persist_ctas, void *stream);
int launch_decode_kivi(const DecodeArgs &a, void *stream);

// A decode step: one new token per sequence appended at slot seq_lens[b], then decode
// attention over seq_lens[b] + 1 tokens (DecodeArgs::seq_lens are the lengths before it).
struct StepArgs {
  const void *k_new, *v_new;  // [batch][heads_kv][d]
  int kv_dtype;               // TQ_F32 / TQ_BF16
};
// the step on the persistent decode kernel with the append and the query preparation
// fused in (TQ_ERR_UNSUPPORTED, with nothing launched, outside what it covers)
int launch_decode2_step(const DecodeArgs &a, const StepArgs &s, int *persist_ctas, void *stream);
// that kernel followed by the combine
int launch_decode_step_tq(const DecodeArgs &a, const StepArgs &s, void *stream);
// lens_out[b] = seq_lens[b] + 1 clamped to [0, capacity]
int launch_step_lengths(const int32_t *seq_lens, int batch, int capacity, int32_t *lens_out, void *stream);

struct DequantArgs {
  const uint8_t *codes;  // plane bases in the blocked records (see AppendArgs)
  const float *norms;
  const uint8_t *signs;
  const float *rnorms;
  int bb, cap16;
  const int32_t *btab;  // paged caches: the block table (NULL: contiguous)
  int pool_blocks;
  int *error;
  int vt;  // 1: value codes (pair-interleaved layout)
  int batch, heads, capacity, t0, t1;
  Role role;
  const float *centroids;
  const DevParams *params;
  float *out;
  const float *rot;  // dense rotation M, or nullptr (Walsh-Hadamard)
  const uint16_t *side = nullptr;  // key side codes: plane base, bases as given, rank
  const float *side_u = nullptr;
  int side_rank = 0;
};
int launch_dequant_tq(const DequantArgs &a, void *stream);

struct KiviAppendArgs {
  const tq_ctx *ctx;
  const tq_cache *cache;
  const void *k, *v;
  int dtype, batch, heads, n_new;
  const int32_t *seq_lens;
  int *error;
};
int launch_append_kivi(const KiviAppendArgs &a, void *stream);

struct KiviDequantArgs {
  const tq_ctx *ctx;
  const tq_cache *cache;
  int batch, heads, t0, t1;
  const int32_t *seq_lens;
  float *k_out, *v_out;
};
int launch_dequant_kivi(const KiviDequantArgs &a, void *stream);

// split count / chunk policy shared by sizing and launch
void choose_splits(int batch, int heads_kv, int max_len, int requested, int *splits, int *chunk);

}  // namespace tq
