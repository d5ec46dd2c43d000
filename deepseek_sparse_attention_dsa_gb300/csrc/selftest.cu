// selftest.cu -- dsa_selftest_wait_timeout: the pipeline's bounded wait, made
// to run out on purpose.
//
// Every kernel of the library waits on mbarriers with mbar_wait (ptx.cuh),
// which gives up after a time limit, sets kErrTimeout in the context's error
// word and raises the CTA's abort flag so that every later wait of the CTA
// returns at once; the kernel then frees its tensor memory and exits, and the
// host reads DSA_ERR_TIMEOUT from dsa_get_error.  Nothing in a correct run
// reaches that path, so this entry point drives it directly: one CTA holds
// tensor memory, waits with a short limit on an mbarrier that nothing
// arrives on, waits on it a second time (which the raised abort flag must end
// at once), frees the tensor memory and exits.  No fault, trap or unbounded
// wait is involved.
#include <cuda_runtime.h>

#include <cstdio>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(int *err, uint64_t limit_ns, int64_t *result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);   // one arrival completes the phase; none comes
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  if (threadIdx.x == 32) {
    volatile int *flag = &abort_flag;
    const uint64_t t0 = globaltimer();
    const bool first = mbar_wait(smem_u32(&bar), 0, flag, err, limit_ns);
    const uint64_t t1 = globaltimer();
    const bool second = mbar_wait(smem_u32(&bar), 0, flag, err, limit_ns);
    const uint64_t t2 = globaltimer();
    result[0] = first ? 1 : 0;
    result[1] = static_cast<int64_t>(t1 - t0);
    result[2] = second ? 1 : 0;
    result[3] = static_cast<int64_t>(t2 - t1);
    result[4] = *flag;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, 32);
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_selftest_wait_timeout(dsa_ctx_t *ctx, uint64_t limit_ns, int64_t *result,
                                                dsa_stream_t stream) {
  if (!ctx || ctx->device < 0 || !result || limit_ns == 0 || limit_ns > dsa::kWaitLimitNs) return DSA_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  dsa::wait_timeout_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ctx->err, limit_ns, result);
  ctx->last_launches = 1;
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(ctx->last_cuda_error, sizeof(ctx->last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
