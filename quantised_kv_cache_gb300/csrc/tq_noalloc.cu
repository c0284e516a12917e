// Decode attention for callers that cannot allocate device memory.
//
// tq_decode_attention needs a caller-provided workspace (the prepared queries
// and the split-K partial results). Some callers have no way to provide one:
// a host application that owns the whole device-memory budget and hands this
// library nothing but the cache and output buffers, a latency-critical decode
// loop that must never enter the CUDA allocator, or an embedding runtime with
// no access to cudaMalloc at all. This entry point gives them the same
// computation with its workspace in a fixed array compiled into the library.
//
// The array is a file-scope static __device__ object of kStaticScratchBytes.
// Every GPU that loads this library holds it until the process exits. Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; every later call reuses the cached address. A
// cudaDeviceReset unloads the library's device code and frees the array, so the
// cached address is then stale: this entry point must not be called on a device
// after that device has been reset.

#include <cuda_runtime.h>

#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char tq_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
tq_status scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, tq_static_scratch) != cudaSuccess || p == nullptr) return TQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" {

size_t tq_static_scratch_bytes(void) { return kStaticScratchBytes; }

tq_status tq_decode_attention_static(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype,
                                     int batch, int heads_q, int heads_kv, const int32_t *d_seq_lens, int max_len,
                                     int splits, float *d_out, void *stream) {
  if (!ctx) return TQ_ERR_ARG;
  // the array is looked up on the current device, which must be the one holding the
  // context's parameters and the caller's buffers
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return TQ_ERR_CUDA;
  if (cur != ctx->device) return TQ_ERR_ARG;
  size_t need = 0;
  tq_status s = tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, splits, &need);
  if (s != TQ_OK) return s;
  if (need > kStaticScratchBytes) return TQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != TQ_OK) return s;
  return tq_decode_attention(ctx, cache, d_q, q_dtype, batch, heads_q, heads_kv, d_seq_lens, max_len, splits,
                             scratch, kStaticScratchBytes, d_out, stream);
}

}  // extern "C"
