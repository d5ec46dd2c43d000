// quantize.cu -- quantize-on-store: bf16 rows of the step into the fp8 cache
// formats at the slot of each row's own position.
//
// The pages store rows that are already in cache format (mstar
// DSAManager.store_keys); the fp8 layouts are LLMServingSim's "What the KV
// cache actually holds" (132-byte index rows: 128 e4m3 + one fp32 scale;
// 656-byte latent rows: 512 e4m3 + four fp32 scales, one per 128 columns, +
// 64 bf16 rope) and ttnn sparse_sdpa's packed kv row.  Quantisation: per group
// scale = amax / 448 in fp32 (1 for an all-zero group), code = E4M3 of the fp32
// quotient x / scale, rounded to nearest with ties to even and saturating at
// 448, the largest finite E4M3 value.
//
// One warp per row.
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

// fp32 -> E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits).  For a
// magnitude in the fp32 binade 2^e the E4M3 spacing is 2^(e-3) (2^-9 below
// 2^-6, the E4M3 subnormals): multiply by the exact power of two 2^(3-e),
// round to an integer with ties to even, and build the code from (e, integer).
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  const uint32_t sign = (__float_as_uint(x) >> 24) & 0x80u;
  const float a = fabsf(x);
  if (!(a < 448.f)) return sign | 0x7Eu;   // saturate (inputs are finite)
  int e = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu) - 127;
  if (e < -6) e = -6;
  const float scaled = a * __uint_as_float(static_cast<uint32_t>(127 + 3 - e) << 23);
  int k = __float2int_rn(scaled);
  if (e == -6 && k < 8) return sign | static_cast<uint32_t>(k);
  if (k == 16) {
    ++e;
    k = 8;
  }
  return sign | (static_cast<uint32_t>(e + 7) << 3) | static_cast<uint32_t>(k - 8);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// physical cache row of row r's own position, or -1 (bounds error flagged)
__device__ __forceinline__ int64_t own_row(int r, const int32_t *row_pos, const int32_t *row_page_off,
                                           const int32_t *row_npages, const int32_t *row_page_start,
                                           const int32_t *pages, int P, int num_pages, int *err) {
  const int64_t slot = static_cast<int64_t>(row_page_start[r]) + row_pos[r];
  const int64_t pi = slot / P;
  if (pi >= row_npages[r]) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return -1;
  }
  const int page = pages[row_page_off[r] + pi];
  if (page < 0 || page >= num_pages) {
    if (lane_id() == 0) atomicOr(err, kErrBounds);
    return -1;
  }
  return static_cast<int64_t>(page) * P + slot % P;
}

// 128 bf16 index values -> [codes at slot * 128 of the page's code block,
// scale at slot * 4 of its scale block]; lane l handles values 4l .. 4l+3.
__global__ void __launch_bounds__(256) quantize_keys_kernel(const uint2 *__restrict__ keys, uint8_t *__restrict__ cache,
                                                            const int32_t *__restrict__ row_pos,
                                                            const int32_t *__restrict__ row_page_off,
                                                            const int32_t *__restrict__ row_npages,
                                                            const int32_t *__restrict__ row_page_start,
                                                            const int32_t *__restrict__ pages, int T, int P,
                                                            int num_pages, int *err) {
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= T || row_pos[r] < 0) return;   // past the rows, or a padding row of a capturable plan
  const int lane = lane_id();
  const int64_t prow = own_row(r, row_pos, row_page_off, row_npages, row_page_start, pages, P, num_pages, err);
  if (prow < 0) return;
  const uint2 raw = keys[static_cast<int64_t>(r) * 32 + lane];
  const float v[4] = {bf16_bits_to_float(raw.x & 0xFFFFu), bf16_bits_to_float(raw.x >> 16),
                      bf16_bits_to_float(raw.y & 0xFFFFu), bf16_bits_to_float(raw.y >> 16)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) word |= e4m3_code(v[i] / scale) << (8 * i);
  const int64_t page = prow / P, s = prow % P;
  uint8_t *base = cache + page * static_cast<int64_t>(P) * 132;
  reinterpret_cast<uint32_t *>(base + s * 128)[lane] = word;
  if (lane == 0) *reinterpret_cast<float *>(base + static_cast<int64_t>(P) * 128 + s * 4) = scale;
}

// 512 + 64 bf16 latent values -> one 656-byte row.  Lane l quantises columns
// 16l .. 16l+15 (group l / 8 of 128 columns); lanes 0-7 copy the rope.
__global__ void __launch_bounds__(256) quantize_latents_kernel(const uint8_t *__restrict__ lat,
                                                               uint8_t *__restrict__ cache,
                                                               const int32_t *__restrict__ row_pos,
                                                               const int32_t *__restrict__ row_page_off,
                                                               const int32_t *__restrict__ row_npages,
                                                               const int32_t *__restrict__ row_page_start,
                                                               const int32_t *__restrict__ pages, int T, int P,
                                                               int num_pages, int *err) {
  constexpr int L = 512, R = 64, SRC = (L + R) * 2, ROW = L + 4 * (L / 128) + 2 * R;
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= T || row_pos[r] < 0) return;   // past the rows, or a padding row of a capturable plan
  const int lane = lane_id();
  const int64_t prow = own_row(r, row_pos, row_page_off, row_npages, row_page_start, pages, P, num_pages, err);
  if (prow < 0) return;
  const uint8_t *src = lat + static_cast<int64_t>(r) * SRC;
  const uint4 a = reinterpret_cast<const uint4 *>(src)[2 * lane];
  const uint4 b = reinterpret_cast<const uint4 *>(src)[2 * lane + 1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 4; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));   // 8-lane groups
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t c[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) c[i / 4] |= e4m3_code(v[i] / scale) << (8 * (i % 4));
  uint8_t *dst = cache + prow * ROW;
  reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
  if ((lane & 7) == 0) reinterpret_cast<float *>(dst + L)[lane / 8] = scale;
  if (lane < 8) reinterpret_cast<uint4 *>(dst + L + 4 * (L / 128))[lane] = reinterpret_cast<const uint4 *>(src + 2 * L)[lane];
}

// 128 bf16 values of one (row, head) of the indexer query -> 128 codes and one
// scale (dsa_quantize_q); lane l handles values 4l .. 4l+3.  Rows at position
// -1 (padding of a capturable plan) are skipped.
__global__ void __launch_bounds__(256) quantize_q_kernel(const uint2 *__restrict__ q, uint32_t *__restrict__ codes,
                                                         float *__restrict__ scales,
                                                         const int32_t *__restrict__ row_pos, int T, int Hi) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (g >= static_cast<int64_t>(T) * Hi || row_pos[g / Hi] < 0) return;
  const int lane = lane_id();
  const uint2 raw = q[g * 32 + lane];
  const float v[4] = {bf16_bits_to_float(raw.x & 0xFFFFu), bf16_bits_to_float(raw.x >> 16),
                      bf16_bits_to_float(raw.y & 0xFFFFu), bf16_bits_to_float(raw.y >> 16)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) word |= e4m3_code(v[i] / scale) << (8 * i);
  codes[g * 32 + lane] = word;
  if (lane == 0) scales[g] = scale;
}

}  // namespace

cudaError_t launch_quantize_q(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, void *codes, float *scales,
                              cudaStream_t s, int32_t *launches) {
  const int64_t groups = static_cast<int64_t>(plan->T) * ctx->cfg.index_heads;
  quantize_q_kernel<<<static_cast<unsigned>((groups + 7) / 8), 256, 0, s>>>(
      static_cast<const uint2 *>(q), static_cast<uint32_t *>(codes), scales, plan->row_pos, plan->T,
      ctx->cfg.index_heads);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_quantize_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *keys, void *cache,
                                 cudaStream_t s, int32_t *launches) {
  const int grid = (plan->T + 7) / 8;
  quantize_keys_kernel<<<grid, 256, 0, s>>>(static_cast<const uint2 *>(keys), static_cast<uint8_t *>(cache),
                                            plan->row_pos, plan->row_page_off, plan->row_npages, plan->row_page_start,
                                            plan->pages, plan->T, ctx->cfg.page_size, plan->cache_pages, ctx->err);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_quantize_latents(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *latents, void *cache,
                                    cudaStream_t s, int32_t *launches) {
  const int grid = (plan->T + 7) / 8;
  quantize_latents_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(latents), static_cast<uint8_t *>(cache),
                                               plan->row_pos, plan->row_page_off, plan->row_npages,
                                               plan->row_page_start, plan->pages, plan->T, ctx->cfg.page_size,
                                               plan->cache_pages, ctx->err);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace dsa
