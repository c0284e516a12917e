// Append-quantise dispatch: picks the kernel family for one role of a call.
//
// "Statistical Inference and Quality Measures of KV Cache Quantisations
// Inspired by TurboQuant", technical summary, "Quantisation schemes": rotated
// roles (WHT + scalar Lloyd-Max, with a 1-bit QJL sketch of the residual for the
// (n-1)-bit vectors) and the unrotated KV role. Every supported role is served
// by one of three families:
//   * launch_append_bulk -- bf16 input, rotated roles, enough vectors for the
//     persistent tensor-map / tcgen05 kernel;
//   * launch_append_tc   -- rotated roles otherwise (fp32 input, or few bf16
//     vectors), thread-per-vector on tcgen05;
//   * launch_append2     -- unrotated roles (the KV scheme, 2..4 bits).
// Calls of at most 8192 vectors per tensor never come here: they take the
// warp-per-vector launch for keys and values together (launch_append_small).

#include "tq_internal.h"

namespace tq {

int launch_append_tq(const AppendArgs &a, void *stream) {
  if (!a.ctx) return TQ_ERR_ARG;
  int r = launch_append_bulk(a, a.ctx, stream);  // rotated roles, bf16 input
  if (r != TQ_ERR_UNSUPPORTED) return r;
  r = launch_append_tc(a, a.ctx, stream);  // rotated roles
  if (r != TQ_ERR_UNSUPPORTED) return r;
  return launch_append2(a, a.ctx, stream);  // unrotated roles
}

}  // namespace tq
