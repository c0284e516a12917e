// Self-test of the bounded waits that every kernel of the library uses (mbar_wait_bounded): a
// one-warp kernel initialises an mbarrier that nothing will ever complete, waits on it with a
// caller-chosen budget, and must come back with TQ_ERR_TIMEOUT recorded in the context's device
// error word -- the path a kernel takes when an expected copy or tensor-core commit never lands.
// No copy, tensor-core operation or other CTA is involved, so the wait running out leaves
// nothing in flight: the kernel returns and the context stays usable.

#include <cuda_runtime.h>

#include "tq_ptx.cuh"

namespace tq {
namespace {

__global__ void bounded_wait_selftest_kernel(int *error, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  // phase 0 never completes: no thread arrives and no copy is tied to the barrier
  const bool done = mbar_wait_bounded(&bar, 0, threadIdx.x == 0 ? error : nullptr, budget_ns);
  if (threadIdx.x == 0 && done) set_error(error, TQ_ERR_STATE);  // a wait that claimed success
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_selftest_bounded_wait(const tq_ctx *ctx, unsigned long long budget_ns, void *stream) {
  if (!ctx || budget_ns > 2000000000ull) return TQ_ERR_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return TQ_ERR_CUDA;
  if (cur != ctx->device) return TQ_ERR_ARG;
  tq::bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(&ctx->dparams->error, budget_ns);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
