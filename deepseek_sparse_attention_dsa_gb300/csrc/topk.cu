// topk.cu -- per-row causal top-k with ties to the earlier position
// (mstar select_topk_causal / index_topk: (T, topk) int32, -1 padded; a row's
// selection must not depend on the batch packing or the device, so equal
// scores are broken toward the lower position).
//
// One CTA per row.  Scores are mapped to order-preserving 32-bit keys (-0.0
// ranks as +0.0).  Three histogram passes (11 + 11 + 10 bits, shared-memory
// atomics; the first pass aggregates equal bins within a warp) pin down the
// exact key tau of the k-th largest score and how many scores equal to tau
// must be taken.  Then each warp owns a contiguous segment of the row: a
// counting pass gives every warp its output offset and its rank among the
// tau-ties, and a writing pass emits, in ascending position order, every
// position above tau plus the earliest tau-ties.  A row that sees at most
// topk keys takes them all and pads with -1.
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kBatch = 8;   // independent loads in flight per thread

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 and +0.0 are the same score
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *ws, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    ws[lane] = s;
  }
  __syncthreads();
  const int before = warp ? ws[warp - 1] : 0;
  *total = ws[kTopkWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Bin (counted from the top) that holds the need-th largest key; *above gets
// the number of keys in higher bins.
__device__ __forceinline__ int find_bin(const int *hist, int nbins, int need, int *ws, int *res, int *above) {
  const int b0 = nbins - 1 - 2 * static_cast<int>(threadIdx.x), b1 = b0 - 1;
  const int c0 = b0 >= 0 ? hist[b0] : 0, c1 = b1 >= 0 ? hist[b1] : 0;
  int total;
  const int ex = block_exclusive_scan(c0 + c1, ws, &total);
  if (ex < need && need <= ex + c0) {
    res[0] = b0;
    res[1] = ex;
  } else if (ex + c0 < need && need <= ex + c0 + c1) {
    res[0] = b1;
    res[1] = ex + c0;
  }
  __syncthreads();
  *above = res[1];
  const int b = res[0];
  __syncthreads();
  return b;
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const float *__restrict__ scores,
                                                               const int64_t *__restrict__ row_score_off,
                                                               const int32_t *__restrict__ row_pos, int K,
                                                               int32_t *__restrict__ sel) {
  __shared__ int hist[2048];
  __shared__ int ws[kTopkWarps];
  __shared__ int res[2];
  __shared__ int wgt[kTopkWarps], weq[kTopkWarps];

  const int row = blockIdx.x;
  const int n = row_pos[row] + 1;
  int32_t *out = sel + static_cast<int64_t>(row) * K;
  if (n <= K) {
    for (int i = threadIdx.x; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float *s = scores + row_score_off[row];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // ---- radix select of the k-th largest key.  Every loop below issues
  // kBatch independent loads per thread before using any of them, so each
  // pass is bound by L2 bandwidth rather than by one load's latency.
  uint32_t prefix = 0, pmask = 0;
  int need = K;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 2 ? 1024 : 2048;
    for (int i = threadIdx.x; i < 2048; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kTopkThreads * kBatch) {
      uint32_t k[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kTopkThreads + static_cast<int>(threadIdx.x);
        k[j] = i < n ? order_key(__ldg(s + i)) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const bool in = base + j * kTopkThreads + static_cast<int>(threadIdx.x) < n;
        if (pass == 0) {
          // equal bins of a warp are counted by one atomic
          const int bin = in ? static_cast<int>(k[j] >> 21) : -1;
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (in && (__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], __popc(peers));
        } else if (in && (k[j] & pmask) == prefix) {
          atomicAdd(&hist[(k[j] >> shift) & (nbins - 1)], 1);
        }
      }
    }
    __syncthreads();
    int above;
    const int b = find_bin(hist, nbins, need, ws, res, &above);
    prefix |= static_cast<uint32_t>(b) << shift;
    pmask |= static_cast<uint32_t>(nbins - 1) << shift;
    need -= above;
  }
  const uint32_t tau = prefix;  // exact key of the k-th largest score
  // `need` = how many scores equal to tau are taken (the earliest ones)

  // ---- ordered compaction, one contiguous segment per warp
  const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 32 * kBatch - 1) / (32 * kBatch) * (32 * kBatch);
  const int lo = warp * seg, hi = min(n, lo + seg);
  int cgt = 0, ceq = 0;
  for (int base = lo; base < hi; base += 32 * kBatch) {
    uint32_t k[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + 32 * j + lane;
      k[j] = i < hi ? order_key(__ldg(s + i)) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool in = base + 32 * j + lane < hi;
      cgt += __popc(__ballot_sync(0xffffffffu, in && k[j] > tau));
      ceq += __popc(__ballot_sync(0xffffffffu, in && k[j] == tau));
    }
  }
  if (lane == 0) {
    wgt[warp] = cgt;
    weq[warp] = ceq;
  }
  __syncthreads();
  int out_base = 0, eq_base = 0;
  for (int w = 0; w < warp; ++w) {
    const int take_eq = max(0, min(weq[w], need - eq_base));
    out_base += wgt[w] + take_eq;
    eq_base += weq[w];
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32 * kBatch) {
    uint32_t k[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + 32 * j + lane;
      k[j] = i < hi ? order_key(__ldg(s + i)) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + 32 * j + lane;
      const bool gt = i < hi && k[j] > tau;
      const bool eq = i < hi && k[j] == tau;
      const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
      const bool take = gt || (eq && eq_base + __popc(eqm & lt_mask) < need);
      const uint32_t tm = __ballot_sync(0xffffffffu, take);
      const int slot = out_base + __popc(tm & lt_mask);
      if (take && slot < K) out[slot] = i;
      out_base += __popc(tm);
      eq_base += __popc(eqm);
    }
  }
}

}  // namespace

cudaError_t launch_topk(const dsa_ctx *ctx, const dsa_plan_t *plan, const float *scores, int32_t *sel,
                        cudaStream_t s, int32_t *launches) {
  topk_kernel<<<plan->T, kTopkThreads, 0, s>>>(scores, plan->row_score_off, plan->row_pos, ctx->cfg.topk, sel);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace dsa
