/*
 * tq.h -- C ABI of libtq: TurboQuant-style KV-cache compression and decode
 * attention read directly from the compressed cache, for one NVIDIA GB300
 * (sm_103a). Plain pointers and sizes only; no framework types.
 *
 * Sources, cited by page title and section:
 *   [TQ-stats]  "Statistical Inference and Quality Measures of KV Cache
 *               Quantisations Inspired by TurboQuant" (technical summary:
 *               "Theoretical framework", "Quantisation schemes",
 *               "Main contribution 1").
 *   [HeadQ]     "HeadQ: Model-Visible Distortion and Score-Space Correction
 *               for KV-Cache Quantization", sections 2.1-2.2 and 3 (keys are
 *               read through logits, values through the p-weighted sum; the
 *               cache-write / cache-read split).
 *   [KIVI-geom] "Your KV cache is not a bit problem but a geometry problem"
 *               ("What quantisation error is made of", "Keys", "Values",
 *               "The systems tax").
 *   [KVQuant++] "KVQuant++" forum post ("Codebook design", "Fast codebook
 *               lookup", "Deployment and use": a quantiser built from
 *               head_dim and num_bits with compress / decompress calls).
 *
 * ---------------------------------------------------------------------------
 * Conventions for every call
 * ---------------------------------------------------------------------------
 *  - Every function returns tq_status; nothing throws across the ABI.
 *  - "d_" pointers are device pointers on the device that was current when
 *    the context was created; "h_" pointers are host pointers.
 *  - The caller owns every buffer it passes (cache planes, inputs, outputs,
 *    workspace). The library allocates only the context's parameter block
 *    (codebooks, D, S, the device error word, S and H D prepared as
 *    tensor-core operands; about 320 KB), one non-blocking stream and two
 *    events in tq_init, and frees them in tq_destroy. The library never
 *    frees caller memory.
 *  - Launches are asynchronous on the given stream (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream). No call synchronises except
 *    tq_get_device_error.
 *  - Argument errors are found on the host before any launch (TQ_ERR_ARG,
 *    TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN). Conditions only the device can see
 *    (a write past a cache's capacity) set a sticky device error word and
 *    skip the offending writes; read it with tq_get_device_error.
 *  - A failed CUDA launch returns TQ_ERR_CUDA.
 *
 * ---------------------------------------------------------------------------
 * Storage format (both the library and the independent CPU checker implement
 * this text)
 * ---------------------------------------------------------------------------
 *  Cache geometry (TQ schemes): one records array of 16-token blocks,
 *  [batch][heads_kv][ceil(capacity / 16)] blocks (row-major). A block holds
 *  the records of its 16 token slots plane by plane, in tq_plane order: the
 *  K code records [16][d*b_K/8], the K norms [16] (float32), for sketched
 *  keys the K sign records [16][d/8] and the K residual norms [16], then the
 *  same four planes for V; unused planes take no bytes. Every plane starts at
 *  a multiple of 16 bytes, so token slot t of sequence-head (b, h) is at
 *  block (b * heads_kv + h) * ceil(capacity / 16) + t / 16, entry t % 16 of
 *  each plane, and the 16 tokens of a block are one contiguous copy
 *  (tq_cache_sizes gives the block size and the plane offsets).
 *  Exception: the V code plane of a block is not [16][record] but eight pair
 *  rows of d*b_V/4 bytes: row j holds tokens 2j and 2j+1, coordinate i in
 *  field 16 (i mod 8) + i / 8 (d = 128) of 2*b_V bits at bit 2*b_V*field of
 *  the row's little-endian bit string, token 2j's index in the low b_V bits and
 *  token 2j+1's in the high ones (two tokens' codes of one coordinate side by
 *  side, the operand order of the decode's tensor-core value sums).
 *
 *  Code records: a vector's d coordinates each get a b-bit index into the
 *  Lloyd-Max codebook (index 0 = the most negative centroid). The d/2
 *  coordinate pairs (2p, 2p+1), p = 4n + t (t = p mod 4), are stored in slot
 *  order: pair p occupies slot (d/8) t + n, so coordinate i = 8n + 2t + e
 *  (e = i mod 2) has its index at bit offset b ((d/4) t + 2n + e) of the
 *  record's d*b-bit little-endian string (string bit k = bit k % 8 of byte
 *  k / 8); the record is d*b/8 bytes. (With d = 128 the 16 pairs a tensor-core
 *  thread consumes -- fixed t, n = 0..15 -- are contiguous.)
 *  Sign records (QJL): the same offsets with b = 1; the bit is 1 when
 *  (S r)_i >= 0. Norm records: float32.
 *
 *  Per scheme, for a budget of n bits per coordinate ([TQ-stats]
 *  "Quantisation schemes"):
 *    TQ_SCHEME_KV   K: n-bit codes of the unrotated unit vector + norm.
 *                   V: the same.
 *    TQ_SCHEME_KQV  K: n-bit codes of the rotated unit vector + norm.
 *                   V: (n-1)-bit codes of the rotated unit vector + norm
 *                      + d sign bits + residual norm.
 *    TQ_SCHEME_QKQV K and V: (n-1)-bit codes + norm + signs + residual norm.
 *  Unused planes have 0 bytes per token.
 *
 *  Quantisation of one vector x (fp32 arithmetic on the device; the CPU
 *  checker repeats it in fp64 and codes must agree except where the exact
 *  value lies within 1e-6 of a decision boundary):
 *    nu = ||x||_2;   u = x / nu   (nu == 0: stored nu = 0, codes of u = 0,
 *                                  all sign bits 1, rho = 0)
 *    y  = H_d D u  for rotated schemes (D = seeded +/-1 diagonal, H_d the
 *                  orthonormal Sylvester Hadamard in natural order); y = u
 *                  for TQ_SCHEME_KV
 *    idx_i = number of codebook boundaries b_j with y_i >= b_j
 *    QJL:  r = y - c[idx] (unit domain), sign_i = [(S r)_i >= 0],
 *          rho = nu * ||r||   (stored float32)
 *  Codebook: the Lloyd-Max quantiser of the density (1 - t^2)^((d-3)/2) on
 *  [-1, 1] ([KVQuant++] "Codebook design"; [TQ-stats] "Theoretical
 *  framework"), fitted in fp64 and stored as float32 (centroids and midpoint
 *  boundaries, each rounded to nearest).
 *  Method randomness: SplitMix64 (Steele, Lea & Flood 2014) evaluated at
 *  counter c: w(seed, c) = mix64(seed + c * 0x9E3779B97F4A7C15 mod 2^64),
 *  c = stream * 2^32 + i + 1.  D_i = (w(seed, 1<<32 | i) >> 63) ? -1 : +1.
 *  S (d x d, row-major entry k = row*d + col) uses stream 2:
 *  u1 = ((w_{2k} >> 11) + 1) 2^-53, u2 = (w_{2k+1} >> 11) 2^-53,
 *  S_k = (float)(sqrt(-2 log u1) * cos(2 pi u2)) in double precision.
 *
 *  Reconstruction ("dequantise"): x_hat = nu D H c[idx]
 *    (+ rho sqrt(pi/2)/d D H S^T sigma, sigma_i = +/-1, for sketched vectors;
 *     D and H dropped for TQ_SCHEME_KV).
 *
 *  KIVI records (TQ_SCHEME_KIVI, [KIVI-geom]): separate planes, each an array
 *  over [batch][heads_kv][capacity] token slots. 2-bit codes per element in
 *  plain channel order, channel i at bits [2i, 2i+2) (d/4 bytes per token),
 *  for both K and V; float16
 *  (zero, step) pairs per group, zero = fp16(group min), step =
 *  fp16((max - min) / 3) with the quotient in fp64, code =
 *  clamp(round_half_even((x - zero) / step), 0, 3) (0 when step == 0).
 *  A per-channel tensor groups `group` consecutive quantised tokens of one
 *  channel: stats plane [batch][heads_kv][capacity/group][d][2] halves.
 *  A per-token tensor groups `group` consecutive channels of one token:
 *  stats plane [batch][heads_kv][capacity][d/group][2] halves.
 *  The most recent tokens stay in a bfloat16 window: ring buffer
 *  [batch][heads_kv][window + group][d], token t in slot t % (window+group).
 *  After a sequence holds N tokens, its first nq = group*floor((N-window)/
 *  group) tokens (0 while N < window + group) are quantised and tokens
 *  [nq, N) are in the window.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_ABI_VERSION 3

typedef struct tq_ctx tq_ctx; /* opaque, host-owned */

typedef enum {
  TQ_OK = 0,
  TQ_ERR_ARG = 1,         /* a null pointer, a negative size, a bad enum value */
  TQ_ERR_UNSUPPORTED = 2, /* a valid request this build does not implement   */
  TQ_ERR_CAPACITY = 3,    /* (device) an append ran past a cache's capacity  */
  TQ_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed            */
  TQ_ERR_TIMEOUT = 5,     /* (device) a bounded wait gave up                 */
  TQ_ERR_STATE = 6,       /* the call does not fit the context's scheme      */
  TQ_ERR_ALIGN = 7,       /* a pointer is not 16-byte aligned                */
  TQ_ERR_WORKSPACE = 8    /* the workspace is smaller than tq_workspace_size */
} tq_status;

typedef enum {
  TQ_SCHEME_KV = 0,
  TQ_SCHEME_KQV = 1,
  TQ_SCHEME_QKQV = 2,
  TQ_SCHEME_KIVI = 3
} tq_scheme;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1 } tq_dtype;

/* The rotation of the rotated roles (KQV and QKQV keys and values). */
typedef enum {
  TQ_ROTATION_WHT = 0,   /* y = H_d D u: the randomised Walsh-Hadamard transform (default) */
  TQ_ROTATION_DENSE = 1  /* y = M u, M a seeded random rotation in SO(d) (see tq_set_rotation) */
} tq_rotation;

/* The planes of a block of the records array (TQ schemes), in storage order. */
typedef enum {
  TQ_PLANE_K_CODES = 0, TQ_PLANE_K_NORM = 1, TQ_PLANE_K_SIGNS = 2, TQ_PLANE_K_RNORM = 3,
  TQ_PLANE_V_CODES = 4, TQ_PLANE_V_NORM = 5, TQ_PLANE_V_SIGNS = 6, TQ_PLANE_V_RNORM = 7,
  TQ_PLANE_K_SIDE = 8, /* keys' rank-r side codes (tq_set_side_basis): r float16 per token */
  TQ_NUM_PLANES = 9
} tq_plane;

/* Device pointers of one cache. Sizes come from tq_cache_sizes; a pointer
 * whose size is 0 is unused and may be NULL. Every non-NULL pointer must be
 * 16-byte aligned.
 *
 * Paged layout (TQ schemes only; [KIVI-geom] "The systems tax": decoding appends
 * one token at a time, so a serving cache grows block by block). With
 * block_table == NULL the records array is the contiguous
 * [batch][heads_kv][ceil(capacity / 16)] block grid described above. With a
 * block table, `records` is a pool of `pool_blocks` 16-token blocks (each
 * tq_cache_sizes.block_bytes, same plane layout) and
 *   block_table : int32 [batch][heads_kv][ceil(capacity / 16)], device memory,
 * maps block j of sequence-head (b, h) -- its token slots 16 j .. 16 j + 15 --
 * to pool block block_table[(b * heads_kv + h) * ceil(capacity / 16) + j].
 * Entries a call reaches (the blocks holding the slots it writes or reads) must
 * lie in [0, pool_blocks) and distinct sequence-heads must not share a block;
 * entries no call reaches are ignored (-1 is a conventional "unmapped"). A
 * reached entry outside [0, pool_blocks) is skipped (no access through it) and
 * sets the device error word to TQ_ERR_ARG. The table is read, never written,
 * by the library; the caller owns it and may change entries between calls (in
 * stream order). Results are the contiguous layout's, bit for bit, whatever the
 * mapping. */
typedef struct tq_cache {
  int batch, heads_kv, capacity;
  uint8_t *records;                          /* TQ schemes: the blocked records (or the pool) */
  uint8_t *k_codes;  uint8_t *v_codes;       /* KIVI: 2-bit codes */
  uint16_t *k_stats; uint16_t *v_stats;      /* KIVI: fp16 (zero, step) */
  uint16_t *k_window; uint16_t *v_window;    /* KIVI: bf16 ring buffers */
  const int32_t *block_table;                /* TQ schemes: NULL (contiguous) or the block table */
  int pool_blocks;                           /* blocks in the pool when block_table != NULL */
} tq_cache;

typedef struct tq_cache_sizes {
  size_t records;                    /* TQ schemes: bytes of the records array */
  size_t block_bytes;                /* TQ schemes: bytes of one 16-token block */
  size_t plane_offset[TQ_NUM_PLANES]; /* TQ schemes: byte offset of each plane in a block */
  size_t plane_bytes[TQ_NUM_PLANES];  /* TQ schemes: bytes per token of each plane (0: unused) */
  size_t k_codes, v_codes, k_stats, v_stats, k_window, v_window; /* KIVI plane bytes */
  size_t record_bytes; /* algorithmic bytes of one token-head (K + V records) */
} tq_cache_sizes;

/* ABI version of the loaded library (TQ_ABI_VERSION it was built with). */
int tq_abi_version(void);

/* Human-readable name of a status code (static string; never NULL). */
const char *tq_status_str(int status);

/* Create a context ([KVQuant++] "Deployment and use": a quantiser from
 * head_dim and num_bits; [TQ-stats] "Quantisation schemes": the scheme and
 * its budget). d: head dimension (this build: 128). bits: the budget n in
 * bits per coordinate, 2..4 (TQ_SCHEME_KIVI: must be 2). scheme: a
 * tq_scheme. seed: selects D and S. Fits the needed codebooks on the host
 * (fp64), draws D and S, copies them to the current device.
 * *out receives the handle (NULL on failure). */
tq_status tq_init(int d, int bits, int scheme, uint64_t seed, tq_ctx **out);

/* Free the context's device parameter block and the handle. NULL is a no-op. */
void tq_destroy(tq_ctx *ctx);

/* KIVI options ([KIVI-geom]): group size (32), full-precision window length
 * (128, a multiple of group), and the grouping axes: k_per_channel = 1 groups
 * keys along tokens per channel, 0 along channels per token; v_per_token = 1
 * groups values along channels per token, 0 along tokens per channel. Call
 * before sizing or using a cache; TQ_ERR_STATE for other schemes. */
tq_status tq_set_kivi(tq_ctx *ctx, int group, int window, int k_per_channel, int v_per_token);

/* Choose the rotation of the rotated roles ([KVQuant++] "Rotation-invariance
 * guarantee" and "Rate-distortion performance": a random QR rotation or a
 * Hadamard transform, the rotation kept in SO(d), determinant +1).
 * TQ_ROTATION_DENSE: G is the d x d Gaussian matrix of the method's counter
 * generator in stream 3 (entry k = row * d + col; the Box-Muller recipe of S,
 * kept in double), G = Q R with diag(R) > 0, the last column of Q negated when
 * det Q = -1, and M = Q^T (rounded to float32); y = M u on the cache write and
 * the query, x_hat = M^T y_hat on reconstruction and on the attention output.
 * Call before any cache is written with the context (the codes of the two
 * rotations differ). With the dense rotation the bulk append of bf16 vectors
 * runs on the tensor-core kernel of fp32 inputs and the decode step runs its
 * append and query preparation as separate kernels. TQ_ERR_STATE for KIVI, and
 * after tq_set_side_basis (choose the rotation first). */
tq_status tq_set_rotation(tq_ctx *ctx, int rotation);

/* Host utility: the dense rotation M (d*d floats, row-major, y = M u) a context
 * created with `seed` uses under TQ_ROTATION_DENSE. */
tq_status tq_draw_rotation(uint64_t seed, int d, float *h_rotation);

/* Rank-r key side codes ([HeadQ] section 3: a score-space correction in a basis
 * learned from calibration queries; [KVQuant++] "Core innovation 4": a low-rank
 * correction of the key quantisation residual). Each key j of KV head h stores,
 * besides its base code, z_j = fp16(U_h^T (k_j - k_hat_j)) (plane TQ_PLANE_K_SIDE,
 * rank float16 values), k_hat_j being the base reconstruction; decoding uses the
 * corrected key k_hat_j + U_h z_j, i.e. adds q^T U_h z_j / sqrt(d) to each logit,
 * and tq_dequantize returns the corrected keys.
 *   rank    : 1..8, or 0 to switch side codes off
 *   heads_kv: the KV heads every cache used with this context has
 *   h_basis : float [heads_kv][d][rank] (host), head h's basis U_h with orthonormal
 *             columns (TQ_ERR_ARG when U_h^T U_h is not the identity to 1e-3)
 * Applies to the unsketched key roles (TQ_SCHEME_KV, TQ_SCHEME_KQV); TQ_ERR_STATE
 * otherwise. Call before any cache is sized or written: the record layout gains
 * the side plane. The context copies the bases to the device (heads_kv * d *
 * rank floats, twice: as given and in the rotated coordinates) and frees them in
 * tq_destroy. Appends and decodes of a context with side codes take the general
 * tensor-core / warp append kernels and the split-K decode kernel. */
tq_status tq_set_side_basis(tq_ctx *ctx, int rank, int heads_kv, const float *h_basis);

/* Host utility for calibrating side-code bases: the `rank` leading principal
 * directions (about the origin) of the n rows of h_x (float [n][d]): the
 * eigenvectors of sum_j x_j x_j^T for its largest eigenvalues, in decreasing
 * order, each signed so that its largest-magnitude component is positive,
 * written to h_basis (float [d][rank]). Rows of calibration queries give HeadQ's
 * basis; rows of key residuals k - k_hat (tq_dequantize) give the low-rank
 * correction's basis (their top right singular vectors). */
tq_status tq_principal_basis(const float *h_x, int n, int d, int rank, float *h_basis);

/* Byte sizes of a cache of `capacity` token slots for [batch][heads_kv]
 * sequences-heads: TQ schemes the records array (whole 16-token blocks per
 * sequence-head), its block size and plane offsets; KIVI the sizes of its
 * planes (capacity must be a multiple of the group). */
tq_status tq_cache_sizes_get(const tq_ctx *ctx, int batch, int heads_kv, int capacity,
                             tq_cache_sizes *out);

/* The same call under the name the cache-sizing step was first specified with
 * (tq_cache_bytes): identical arguments, results and errors. */
tq_status tq_cache_bytes(const tq_ctx *ctx, int batch, int heads_kv, int capacity, tq_cache_sizes *out);

/* Quantise and write n_new tokens per sequence ([HeadQ] 3, "cache write";
 * [KIVI-geom] "The systems tax": per-token append).
 *   d_k, d_v : [batch][heads_kv][n_new][d] contiguous, dtype TQ_F32 or TQ_BF16
 *   d_seq_lens : int32 [batch], the current length of each sequence; token t
 *                of sequence b goes to slot d_seq_lens[b] + t. The library
 *                does not advance it: the caller adds n_new afterwards, in
 *                stream order.
 * A sequence whose slots would exceed the capacity is skipped and the
 * device error word is set to TQ_ERR_CAPACITY. KIVI: keeps the window rule
 * stated above (groups leave the window when it reaches window + group).
 * Calls of at most 8192 vectors per tensor quantise keys and values in one
 * launch; larger ones run the key kernel on the context's own stream,
 * forked from and joined back into `stream` with events, so all of the
 * call's work is still ordered before anything later enqueued on `stream`.
 * (The context's stream and events are shared state: do not call this on one
 * context from two host threads at once.) */
tq_status tq_append_quantize(const tq_ctx *ctx, const tq_cache *cache, const void *d_k,
                             const void *d_v, int dtype, int batch, int heads_kv, int n_new,
                             const int32_t *d_seq_lens, void *stream);

/* Workspace bytes tq_decode_attention and tq_decode_step need for these
 * sizes: the prepared queries, a per-batch tile prefix, per-batch step
 * lengths, and the partial softmax records (per split for the split-K
 * kernels, or four per (CTA + head) slot for the persistent kernel, whichever
 * is larger). splits = 0 asks for the library's choice for max_len. */
tq_status tq_workspace_size(const tq_ctx *ctx, int batch, int heads_q, int heads_kv, int max_len,
                            int splits, size_t *out);

/* The same call as tq_workspace_size under the name the workspace-sizing step was
 * first specified with (tq_workspace_bytes): identical arguments, results, errors. */
tq_status tq_workspace_bytes(const tq_ctx *ctx, int batch, int heads_q, int heads_kv, int max_len, int splits,
                             size_t *out);

/* Decode attention read straight from the compressed cache ([HeadQ] 2.1-2.2;
 * [TQ-stats] "Theoretical framework": keys through the logits, values
 * linearly):  out[b][h] = softmax(q[b][h] . K_hat^T / sqrt(d)) V_hat over the
 * first d_seq_lens[b] tokens of KV head h / (heads_q / heads_kv).
 *   d_q   : [batch][heads_q][d], dtype TQ_F32 or TQ_BF16
 *   d_seq_lens : int32 [batch], each in [0, max_len], max_len <= capacity;
 *                a sequence of length 0 yields zeros
 *   splits: token chunks per (batch, kv head) for the split-K kernels; 0 =
 *           library's choice. With one query head per KV head, batch <= 256
 *           and a capacity that is a multiple of 4, a persistent kernel
 *           divides the (batch, head, 64-token tile) space evenly over the
 *           SMs instead and splits does not change the work division.
 *   d_workspace : >= tq_workspace_size(...) bytes, 16-byte aligned, no
 *                 initial contents required
 *   d_out : float32 [batch][heads_q][d]
 * heads_q must be a multiple of heads_kv with heads_q / heads_kv <= 8. */
tq_status tq_decode_attention(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype,
                              int batch, int heads_q, int heads_kv, const int32_t *d_seq_lens,
                              int max_len, int splits, void *d_workspace, size_t workspace_bytes,
                              float *d_out, void *stream);

/* One decode step: append one new token per sequence, then attend over the
 * sequence including it. The same results as tq_append_quantize(n_new = 1,
 * d_seq_lens) followed by tq_decode_attention over d_seq_lens[b] + 1 tokens
 * (bit for bit when batch * heads_kv <= 8192, where that append runs the
 * same warp-per-vector arithmetic), in fewer launches: the new
 * token is quantised where its keys and values are consumed ([HeadQ] 3,
 * "cache write" then "decode"; [KIVI-geom] "The systems tax": decoding
 * appends one token at a time and then reads the whole cache).
 *   d_q : [batch][heads_q][d], dtype q_dtype (TQ_F32 or TQ_BF16)
 *   d_k_new, d_v_new : [batch][heads_kv][d], dtype kv_dtype (TQ_F32 or TQ_BF16)
 *   d_seq_lens : int32 [batch], lengths BEFORE the step; the new token of
 *                sequence b goes to slot d_seq_lens[b]. Not modified: the
 *                caller adds 1 afterwards, in stream order.
 *   max_len : >= every d_seq_lens[b] + 1, <= capacity
 *   d_workspace : >= tq_workspace_size(ctx, batch, heads_q, heads_kv,
 *                 max_len, 0) bytes, 16-byte aligned
 *   d_out : float32 [batch][heads_q][d]
 * A sequence whose new token would not fit (d_seq_lens[b] < 0 or >=
 * capacity) is not appended, the device error word is set to
 * TQ_ERR_CAPACITY, and it is attended over min(d_seq_lens[b] + 1, capacity)
 * tokens (none when negative). With one query head per KV head, the KV or
 * KQV scheme and batch <= 256, the step is one persistent decode kernel
 * (the CTA that reads a head's last tile quantises the new token before
 * copying that tile, and rotates the queries itself) plus the combine;
 * every other configuration runs a small length kernel, the append and the
 * decode in stream order. The context's stream and events are used as by
 * tq_append_quantize. */
tq_status tq_decode_step(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype,
                         const void *d_k_new, const void *d_v_new, int kv_dtype, int batch,
                         int heads_q, int heads_kv, const int32_t *d_seq_lens, int max_len,
                         void *d_workspace, size_t workspace_bytes, float *d_out, void *stream);

/* Reconstruct tokens [t0, t1) of every (batch, kv head) into fp32
 * ([KVQuant++] "Deployment and use": decompress). d_k_hat / d_v_hat:
 * [batch][heads_kv][t1 - t0][d] (either may be NULL to skip). For KIVI the
 * window tokens are returned as stored (bf16 values). d_seq_lens (KIVI only,
 * may be NULL otherwise) gives each sequence's length so the quantised/window
 * split is known. */
tq_status tq_dequantize(const tq_ctx *ctx, const tq_cache *cache, int batch, int heads_kv, int t0,
                        int t1, const int32_t *d_seq_lens, float *d_k_hat, float *d_v_hat,
                        void *stream);

/* Copy the context's float32 parameters to host buffers (any may be NULL):
 * the codebook used for K and for V (centroids: 2^bits floats, boundaries:
 * 2^bits - 1 floats, for the widths *h_k_bits / *h_v_bits), D (d int8) and
 * S (d*d floats, row-major). */
tq_status tq_export_params(const tq_ctx *ctx, int *h_k_bits, float *h_k_centroids, float *h_k_bounds,
                           int *h_v_bits, float *h_v_centroids, float *h_v_bounds, int8_t *h_diag,
                           float *h_sketch);

/* Host utility: the fp64 Lloyd-Max codebook for dimension d and width bits
 * (1..4): 2^bits centroids ascending and 2^bits - 1 midpoint boundaries. */
tq_status tq_codebook_f64(int d, int bits, double *h_centroids, double *h_bounds);

/* Host utility: the method randomness a context created with `seed` uses,
 * drawn by the SplitMix64 / Box-Muller recipe above: D (d int8, +/-1) and S
 * (d*d floats, row-major). Either output may be NULL. */
tq_status tq_draw_params(uint64_t seed, int d, int8_t *h_diag, float *h_sketch);

/* Instrumentation: when set (non-NULL cudaEvent_t handles passed as void*),
 * every later tq_decode_attention records `start` just before its split-K
 * decode kernel and `stop` just after it, on the call's stream, and every
 * tq_append_quantize records `append_start` / `append_stop` around its
 * quantise kernels. Pass NULLs to stop. The caller owns the events. */
tq_status tq_set_profile_events(tq_ctx *ctx, void *start, void *stop, void *append_start, void *append_stop);

/* Decode attention without a caller-provided workspace. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory themselves (an application that owns the whole device-memory budget
 * and hands this library only cache and output buffers, a latency-critical
 * decode loop that must never enter the CUDA allocator, a runtime with no
 * access to cudaMalloc). Arguments and results are those of
 * tq_decode_attention without d_workspace / workspace_bytes; the workspace
 * is a fixed array of tq_static_scratch_bytes() bytes (8 MiB) compiled into
 * the library, which every GPU that loads the library holds until the
 * process exits.
 *  - The call allocates nothing: no cudaMalloc, cudaFree or allocating
 *    library routine.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins. The current device must be the context's device
 *    (TQ_ERR_ARG otherwise). After cudaDeviceReset on a device the cached
 *    address is stale: do not call this entry point on that device again.
 *  - Requests whose workspace (tq_workspace_size) exceeds the array return
 *    TQ_ERR_WORKSPACE before any launch.
 *  - Every call shares the one array and the array keeps the last call's
 *    contents; nothing in it needs to start at zero. Calls that overlap on
 *    the GPU (different streams, or devices sharing a context) race on the
 *    array: serialise them. */
tq_status tq_decode_attention_static(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype,
                                     int batch, int heads_q, int heads_kv, const int32_t *d_seq_lens,
                                     int max_len, int splits, float *d_out, void *stream);

/* Size in bytes of the array tq_decode_attention_static uses. */
size_t tq_static_scratch_bytes(void);

/* Synchronise `stream`, then read and clear the context's sticky device
 * error word into *code (TQ_OK when nothing was recorded). */
tq_status tq_get_device_error(const tq_ctx *ctx, void *stream, int *code);

/* Self-test of the failure path every kernel's waits share: enqueues on `stream`
 * one warp that waits on an mbarrier nothing completes, with a budget of
 * `budget_ns` nanoseconds of %globaltimer time (at most 2e9, the kernels' own
 * budget). The wait gives up, records TQ_ERR_TIMEOUT in the context's device
 * error word (read it with tq_get_device_error) and the kernel returns; no copy
 * or tensor-core operation is in flight, so the context stays usable. The
 * context's GPU must be current. Errors: TQ_ERR_ARG (null context, budget
 * above 2e9, another device current), TQ_ERR_CUDA (launch). */
tq_status tq_selftest_bounded_wait(const tq_ctx *ctx, unsigned long long budget_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
