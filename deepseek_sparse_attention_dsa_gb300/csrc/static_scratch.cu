// static_scratch.cu -- dsa_index_topk_static: score + select without any
// device allocation.
//
// Who needs it: a caller whose process reserves device memory up front in
// its own pool and allows no driver allocation once serving starts (a
// cudaMalloc there can fail when the pool holds nearly all of HBM, and
// cudaMalloc / cudaFree can synchronise the device in the middle of a step).
// dsa_index_topk keeps its fp32 scores in the context's scratch, which
// dsa_plan grows with cudaMalloc; this entry point keeps them instead in the
// file-scope array below, which the CUDA runtime places in device memory when
// it loads this file's module on a GPU (dsa_create makes that happen), and
// which stays there until the process exits.
//
// The array holds DSA_STATIC_SCORES_MAX fp32 scores (16 MiB per GPU).  Every
// call shares it and the last call's contents stay in it; every score a call
// reads back was written by that same call (each row's positions 0..pos are all
// scored before the selection reads them), so nothing needs clearing.  Calls
// whose kernels overlap on the GPU (two streams, or two host threads) race on
// the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdio>

#include "dsa_internal.h"

namespace {

static __device__ __align__(256) float g_static_scores[DSA_STATIC_SCORES_MAX];

}  // namespace

namespace dsa {

// Device address of g_static_scores on `device` (which must be current).  In
// host code the array's name is only a stand-in for the symbol; the device
// address comes from cudaGetSymbolAddress.  Under lazy module loading that
// call is also what loads this file's module onto the device, i.e. what takes
// the array's 16 MiB, so dsa_create makes it: a context holds the address
// from creation on and the entry point below only reads it.
cudaError_t static_scores_address(int device, float **out) {
  *out = nullptr;
  if (device < 0) return cudaErrorInvalidDevice;
  float *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scores);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace dsa

extern "C" dsa_status dsa_index_topk_static(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                            const void *index_cache, int32_t *selection, dsa_stream_t stream) {
  if (!ctx || !plan || plan->ctx != ctx || ctx->device < 0) return DSA_ERR_INVALID_ARG;
  if (plan->num_scores > static_cast<int64_t>(DSA_STATIC_SCORES_MAX)) return DSA_ERR_SCRATCH_LIMIT;
  if (!ctx->static_scores) return DSA_ERR_INVALID_ARG;   // dsa_create records the address for every device context
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!q || !w || !index_cache || !selection) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t n = 0;
  cudaError_t e = dsa::launch_index_scores(ctx, plan, q, w, index_cache, ctx->static_scores, s, &n);
  if (e == cudaSuccess) e = dsa::launch_topk(ctx, plan, ctx->static_scores, selection, s, &n);
  ctx->last_launches = n;
  if (e != cudaSuccess) {
    snprintf(ctx->last_cuda_error, sizeof(ctx->last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
