// store_keys.cu -- scatter the step's index keys into the page-resident index
// cache (mstar DSAManager.store_keys: "each request's at its positions";
// IndexKeyStore.append: keys are stored before the step's selection).
//
// One warp per row.  bf16 rows are copied as 16-byte vectors; fp8 rows
// (128 e4m3 codes + fp32 scale, LLMServingSim "What the KV cache actually
// holds") go to the page-blocked layout: codes at slot * 128 of the page's
// code block, the scale at slot * 4 of its scale block.
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

__global__ void __launch_bounds__(256) store_keys_bf16_kernel(const uint4 *__restrict__ keys, uint4 *__restrict__ cache,
                                                              const int32_t *__restrict__ row_pos,
                                                              const int32_t *__restrict__ row_page_off,
                                                              const int32_t *__restrict__ row_npages,
                                                              const int32_t *__restrict__ row_page_start,
                                                              const int32_t *__restrict__ pages, int T, int P,
                                                              int vec_per_row, int num_pages, int *err) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= T || row_pos[row] < 0) return;   // past the rows, or a padding row of a capturable plan
  const int64_t slot = static_cast<int64_t>(row_page_start[row]) + row_pos[row];
  const int64_t pi = slot / P;
  if (pi >= row_npages[row]) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return;
  }
  const int page = pages[row_page_off[row] + pi];
  if (page < 0 || page >= num_pages) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return;
  }
  const int64_t dst_row = static_cast<int64_t>(page) * P + slot % P;
  for (int v = lane_id(); v < vec_per_row; v += 32)
    cache[dst_row * vec_per_row + v] = keys[static_cast<int64_t>(row) * vec_per_row + v];
}

__global__ void __launch_bounds__(256) store_keys_fp8_kernel(const uint8_t *__restrict__ keys, uint8_t *__restrict__ cache,
                                                             const int32_t *__restrict__ row_pos,
                                                             const int32_t *__restrict__ row_page_off,
                                                             const int32_t *__restrict__ row_npages,
                                                             const int32_t *__restrict__ row_page_start,
                                                             const int32_t *__restrict__ pages, int T, int P, int D,
                                                             int num_pages, int *err) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= T || row_pos[row] < 0) return;   // past the rows, or a padding row of a capturable plan
  const int64_t slot = static_cast<int64_t>(row_page_start[row]) + row_pos[row];
  const int64_t pi = slot / P;
  if (pi >= row_npages[row]) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return;
  }
  const int page = pages[row_page_off[row] + pi];
  if (page < 0 || page >= num_pages) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return;
  }
  const int64_t s = slot % P;
  uint8_t *base = cache + static_cast<int64_t>(page) * P * (D + 4);
  const uint8_t *src = keys + static_cast<int64_t>(row) * (D + 4);
  // codes: D bytes as 4-byte words (the row stride D + 4 keeps 4-byte alignment)
  for (int v = lane_id(); v < D / 4; v += 32)
    reinterpret_cast<uint32_t *>(base + s * D)[v] = reinterpret_cast<const uint32_t *>(src)[v];
  if (lane_id() == 0)
    *reinterpret_cast<uint32_t *>(base + static_cast<int64_t>(P) * D + s * 4) =
        *reinterpret_cast<const uint32_t *>(src + D);
}

}  // namespace

cudaError_t launch_store_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *keys, void *cache,
                              cudaStream_t s, int32_t *launches) {
  const dsa_config_t &c = ctx->cfg;
  const int rows_per_block = 8;
  const int grid = (plan->T + rows_per_block - 1) / rows_per_block;
  if (c.index_fmt == DSA_INDEX_BF16) {
    store_keys_bf16_kernel<<<grid, 256, 0, s>>>(
        static_cast<const uint4 *>(keys), static_cast<uint4 *>(cache), plan->row_pos, plan->row_page_off,
        plan->row_npages, plan->row_page_start, plan->pages, plan->T, c.page_size, c.index_dim * 2 / 16,
        plan->cache_pages, ctx->err);
  } else {
    store_keys_fp8_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(keys), static_cast<uint8_t *>(cache),
                                               plan->row_pos, plan->row_page_off, plan->row_npages,
                                               plan->row_page_start, plan->pages, plan->T, c.page_size, c.index_dim,
                                               plan->cache_pages, ctx->err);
  }
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace dsa
