// topk.cu -- per-row causal top-k with ties to the earlier position
// (mstar select_topk_causal / index_topk: (T, topk) int32, -1 padded; a row's
// selection must not depend on the batch packing or the device, so equal
// scores are broken toward the lower position).
//
// CTAs select one row at a time: 1024 threads with a row each when a step
// has at most one row per SM, else 512-thread CTAs, two per SM, taking rows
// in turn, or, for many rows of at most kShortRow keys, 256-thread CTAs, four
// per SM, with a quarter of the shared memory (candidate, sample and bitmap
// capacities halved or quartered): a row's phases are latency-bound, so more
// rows in flight per SM is what shortens the step.  Scores are mapped to order-preserving 32-bit keys (-0.0
// ranks as +0.0).  The selection is exact; only the amount of work depends on
// the data:
//   1. candidates: a row with at most kCandCap keys takes all of them.  A
//      longer row takes an evenly strided sample (kSampleMin..2 kSampleMin-1
//      keys: 4096 for 512 threads and up, 1024 for 256) into shared
//      memory, finds (to within a 2^10-key bin, below it) the sample key
//      whose rank, scaled by the stride, lies a safe margin above topk, and
//      keeps every key of the row at or above that bound (one pass over the
//      row, float4 loads compared as floats).  When that leaves fewer than topk keys or more
//      than kCandCap, the threshold is found by radix passes over the row in
//      global memory instead.
//   2. the k-th largest key tau and the number of tau ties to take (the
//      earliest ones) come from radix passes (11 + 11 + 10 bits, shared-memory
//      histograms) over the candidates;
//   3. output in ascending position order: the chosen positions are set in a
//      bitmap of the row (shared memory, up to kBitmapBits positions), whose
//      word counts are prefix-summed; every set bit is written at its rank.
//      Rows longer than the bitmap, or with more than kTieCap tau ties among
//      which some are dropped, use an ordered compaction over the row instead:
//      each warp owns a contiguous segment, a counting pass gives every warp
//      its output offset and its rank among the tau ties, and a writing pass
//      emits every position above tau plus the earliest ties.
// A row that sees at most topk keys takes them all and pads with -1.
#include <cuda_runtime.h>

#include <algorithm>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

// CTA sizes: 1024 threads, one CTA per SM, when every row has its own CTA;
// 512 threads, two per SM, when persistent CTAs take several rows each; 256
// threads, four per SM, for many rows of at most kShortRow keys
constexpr int kMaxWarps = 32;
constexpr int kBatch = 16;            // independent loads in flight per thread
constexpr int kScanBatch4 = 8;        // float4 loads in flight per thread in the candidate pass
constexpr int kTieCap = 2048;         // tau ties ranked by position in shared memory
constexpr int kShortRow = 32768;      // longest row the 256-thread CTAs take
// Shared-memory capacities by CTA size: candidate keys held, the strided
// sample's minimum (it holds kSampleMin .. 2*kSampleMin-1 keys) and the
// position bitmap's words.  At 256 threads a row of up to kShortRow keys
// leaves ~1.15 topk + 3 sigma candidates (<= 3.4K at topk 2048) under the cap.
template <int NT>
struct TopkCaps {
  static constexpr int kCandCap = NT >= 512 ? 8192 : 4096;
  static constexpr int kSampleMin = NT >= 512 ? 4096 : 1024;
  static constexpr int kBitmapWords = NT >= 512 ? 8192 : 2048;   // 262,144 or 65,536 positions
};

template <int NT>
struct TopkSmem {
  static constexpr int kWarps = NT / 32;
  union {
    uint32_t sample[2 * TopkCaps<NT>::kSampleMin];
    uint32_t bits[TopkCaps<NT>::kBitmapWords];
  };
  uint32_t ckey[TopkCaps<NT>::kCandCap];
  int32_t cpos[TopkCaps<NT>::kCandCap];
  int hist[2048];                     // radix histograms; tie positions during output
  int ws[kWarps];
  int res[2];
  int n_cand, n_tie;
  int wgt[kWarps], weq[kWarps];
};

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 and +0.0 are the same score
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The score of an order key (+0.0 for the key of both zeros).
__device__ __forceinline__ float key_to_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Exclusive prefix sum over the block of one int per thread; *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *ws, int *total) {
  constexpr int kTopkWarps = NT / 32;
  static_assert(kTopkWarps <= kMaxWarps, "one warp scans the per-warp sums");
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
    int s = lane < kTopkWarps ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kTopkWarps) ws[lane] = s;
  }
  __syncthreads();
  const int before = warp ? ws[warp - 1] : 0;
  *total = ws[kTopkWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Bin (counted from the top) that holds the need-th largest key of a
// histogram of NB <= 2048 bins; *above gets the number of keys in higher bins.
template <int NB, int NT>
__device__ __forceinline__ int find_bin(const int *hist, int need, int *ws, int *res, int *above) {
  constexpr int PER = NB >= NT ? NB / NT : 1;
  int c[PER];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int idx = static_cast<int>(threadIdx.x) * PER + j;   // rank of the bin from the top
    c[j] = idx < NB ? hist[NB - 1 - idx] : 0;
    sum += c[j];
  }
  int total;
  int run = block_exclusive_scan<NT>(sum, ws, &total);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (run < need && need <= run + c[j]) {
      res[0] = NB - 1 - (static_cast<int>(threadIdx.x) * PER + j);
      res[1] = run;
    }
    run += c[j];
  }
  __syncthreads();
  *above = res[1];
  const int b = res[0];
  __syncthreads();
  return b;
}

// The rank-th largest key (rank >= 1) of the keys produced by `for_each`
// (called as for_each(visit) with visit(key) for every key, by every thread
// over its share), by three radix passes of 11, 11 and 10 bits.  *ties gets
// how many keys equal to the result lie within the top `rank`.  With
// PASSES = 2 the result is the lower edge of the 2^10-key bin that holds it
// (a bound at or below the rank-th key; *ties is then meaningless).
template <int NT, int PASSES = 3, typename ForEach>
__device__ __forceinline__ uint32_t radix_select(ForEach for_each, int rank, TopkSmem<NT> &sm, int *ties) {
  uint32_t prefix = 0, pmask = 0;
  int need = rank;
#pragma unroll 1
  for (int pass = 0; pass < PASSES; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 2 ? 1024 : 2048;
    for (int i = threadIdx.x; i < 2048; i += NT) sm.hist[i] = 0;
    __syncthreads();
    for_each([&](uint32_t key) {
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & (nbins - 1)], 1);
    });
    __syncthreads();
    int above;
    const int b = pass == 2 ? find_bin<1024, NT>(sm.hist, need, sm.ws, sm.res, &above)
                            : find_bin<2048, NT>(sm.hist, need, sm.ws, sm.res, &above);
    prefix |= static_cast<uint32_t>(b) << shift;
    pmask |= static_cast<uint32_t>(nbins - 1) << shift;
    need -= above;
  }
  *ties = need;
  return prefix;
}

// Warp-aggregated append: lanes with `take` get consecutive slots after *counter.
__device__ __forceinline__ int warp_append(bool take, int *counter) {
  const uint32_t m = __ballot_sync(0xffffffffu, take);
  if (m == 0) return -1;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  return take ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

template <int NT>
__device__ __forceinline__ void select_row(const float *__restrict__ scores, const int64_t *__restrict__ row_score_off,
                                           const int32_t *__restrict__ row_pos, int K, int32_t *__restrict__ sel,
                                           int row, TopkSmem<NT> &sm) {
  constexpr int kTopkThreads = NT;
  constexpr int kTopkWarps = NT / 32;
  constexpr int kCandCap = TopkCaps<NT>::kCandCap;
  constexpr int kSampleMin = TopkCaps<NT>::kSampleMin;
  constexpr int kBitmapWords = TopkCaps<NT>::kBitmapWords;
  const int n = row_pos[row] + 1;
  int32_t *out = sel + static_cast<int64_t>(row) * K;
  if (n <= K) {
    for (int i = threadIdx.x; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float *s = scores + row_score_off[row];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tid = static_cast<int>(threadIdx.x);

  // ---- 1. candidates
  if (tid == 0) sm.n_cand = 0;
  __syncthreads();
  bool cand_ok;
  if (n <= kCandCap) {
    for (int i = tid; i < n; i += kTopkThreads) {
      sm.ckey[i] = order_key(__ldg(s + i));
      sm.cpos[i] = i;
    }
    if (tid == 0) sm.n_cand = n;
    cand_ok = true;
  } else {
    const int stride = n / kSampleMin;                 // >= 2
    const int m = (n + stride - 1) / stride;           // kSampleMin .. 2*kSampleMin-1
    for (int j = tid; j < m; j += kTopkThreads) sm.sample[j] = order_key(__ldg(s + static_cast<int64_t>(j) * stride));
    __syncthreads();
    // sample rank whose scaled count is about 1.15 topk plus three standard deviations
    const float ks = static_cast<float>(K) / static_cast<float>(stride);
    int rank = static_cast<int>(1.15f * ks + 3.f * sqrtf(ks)) + 8;
    rank = min(rank, m);
    // (a threshold at or below that key is all the pass needs: the lower
    // edge of its 2^10-key bin, two radix passes instead of three)
    int unused;
    const uint32_t l0 = radix_select<NT, 2>(
        [&](auto visit) {
          for (int j = tid; j < m; j += kTopkThreads) visit(sm.sample[j]);
        },
        rank, sm, &unused);
    // every key of the row at or above l0: the 16-byte-aligned body as
    // float4 loads (kScanBatch4 per thread in flight), compared as floats
    // against f0, the score whose key is l0 (order_key is monotone and maps
    // -0.0 and +0.0 to one key, as >= does), each batch's candidates placed
    // by one warp scan and one shared-memory atomic per warp; the unaligned
    // head and the tail (< 4 keys each) by warp 0
    const float f0 = key_to_score(l0);
    const int a0 = min(n, static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(s) >> 2) & 3u)) & 3u));
    const int nb4 = (n - a0) >> 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(s + a0);
    constexpr int kB4 = kScanBatch4;
    for (int base = 0; base < nb4; base += kTopkThreads * kB4) {
      float4 v[kB4];
#pragma unroll
      for (int j = 0; j < kB4; ++j) {
        const int i4 = base + j * kTopkThreads + tid;
        v[j] = i4 < nb4 ? __ldg(s4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // (past the row's end nothing counts, whatever f0 is)
      const int nvalid4 = min(kB4, max(0, (nb4 - base - tid + kTopkThreads - 1) / kTopkThreads));
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < kB4; ++j)
        if (j < nvalid4) cnt += (v[j].x >= f0) + (v[j].y >= f0) + (v[j].z >= f0) + (v[j].w >= f0);
      if (__any_sync(0xffffffffu, cnt > 0)) {
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int wbase = 0;
        if (lane == 31) wbase = atomicAdd(&sm.n_cand, incl);
        int c = __shfl_sync(0xffffffffu, wbase, 31) + incl - cnt;
        if (cnt > 0) {
#pragma unroll
          for (int j = 0; j < kB4; ++j) {
            if (j >= nvalid4) break;
            const float e4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (e4[e] >= f0) {
                if (c < kCandCap) {
                  sm.ckey[c] = order_key(e4[e]);
                  sm.cpos[c] = a0 + 4 * (base + j * kTopkThreads + tid) + e;
                }
                ++c;
              }
            }
          }
        }
      }
    }
    if (warp == 0) {
      // head keys [0, a0) and tail keys [a0 + 4 nb4, n)
      const int t0 = a0 + 4 * nb4;
      const int i = lane < 4 ? lane : t0 + (lane - 4);
      const bool in = lane < 4 ? lane < a0 : i < n;
      const uint32_t key = in ? order_key(__ldg(s + i)) : 0u;
      const int c = warp_append(in && key >= l0, &sm.n_cand);
      if (c >= 0 && c < kCandCap) {
        sm.ckey[c] = key;
        sm.cpos[c] = i;
      }
    }
    __syncthreads();
    cand_ok = sm.n_cand >= K && sm.n_cand <= kCandCap;
  }
  __syncthreads();
  const int n_cand = sm.n_cand;

  // ---- 2. tau and the number of tau ties taken
  int need;
  uint32_t tau;
  if (cand_ok) {
    tau = radix_select<NT>(
        [&](auto visit) {
          for (int i = tid; i < n_cand; i += kTopkThreads) visit(sm.ckey[i]);
        },
        K, sm, &need);
  } else {
    tau = radix_select<NT>(
        [&](auto visit) {
          for (int base = 0; base < n; base += kTopkThreads * kBatch) {
            uint32_t k[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              const int i = base + j * kTopkThreads + tid;
              k[j] = i < n ? order_key(__ldg(s + i)) : 0u;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              if (base + j * kTopkThreads + tid < n) visit(k[j]);
          }
        },
        K, sm, &need);
  }

  // ---- 3. output through a bitmap of the row
  if (cand_ok && n <= 32 * kBitmapWords) {
    const int nw = (n + 31) >> 5;
    for (int w = tid; w < nw; w += kTopkThreads) sm.bits[w] = 0u;
    if (tid == 0) sm.n_tie = 0;
    __syncthreads();
    for (int i = tid; i < n_cand; i += kTopkThreads) {
      const uint32_t key = sm.ckey[i];
      if (key > tau) {
        const int pos = sm.cpos[i];
        atomicOr(&sm.bits[pos >> 5], 1u << (pos & 31));
      } else if (key == tau) {
        const int t = atomicAdd(&sm.n_tie, 1);
        if (t < kTieCap) sm.hist[t] = sm.cpos[i];
      }
    }
    __syncthreads();
    const int n_tie = sm.n_tie;
    if (n_tie == need || n_tie <= kTieCap) {
      // the earliest `need` ties: a tie's rank is the number of ties before it
      for (int t = tid; t < min(n_tie, kTieCap); t += kTopkThreads) {
        const int pos = sm.hist[t];
        int r = 0;
        if (n_tie != need)
          for (int u = 0; u < n_tie; ++u) r += sm.hist[u] < pos ? 1 : 0;
        if (r < need) atomicOr(&sm.bits[pos >> 5], 1u << (pos & 31));
      }
      if (n_tie == need && n_tie > kTieCap) {
        for (int i = tid; i < n_cand; i += kTopkThreads)
          if (sm.ckey[i] == tau) atomicOr(&sm.bits[sm.cpos[i] >> 5], 1u << (sm.cpos[i] & 31));
      }
      __syncthreads();
      // each thread owns a contiguous run of words
      const int per = (nw + kTopkThreads - 1) / kTopkThreads;
      const int w0 = tid * per;
      int cnt = 0;
      for (int q = 0; q < per; ++q)
        if (w0 + q < nw) cnt += __popc(sm.bits[w0 + q]);
      int tot;
      int slot = block_exclusive_scan<NT>(cnt, sm.ws, &tot);
      for (int q = 0; q < per; ++q) {
        if (w0 + q >= nw) break;
        uint32_t b = sm.bits[w0 + q];
        while (b) {
          const int bit = __ffs(b) - 1;
          b &= b - 1u;
          if (slot < K) out[slot] = ((w0 + q) << 5) + bit;
          ++slot;
        }
      }
      return;
    }
  }

  // ---- ordered compaction over the row, one contiguous segment per warp
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
    sm.wgt[warp] = cgt;
    sm.weq[warp] = ceq;
  }
  __syncthreads();
  int out_base = 0, eq_base = 0;
  for (int w = 0; w < warp; ++w) {
    const int take_eq = max(0, min(sm.weq[w], need - eq_base));
    out_base += sm.wgt[w] + take_eq;
    eq_base += sm.weq[w];
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


template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) topk_kernel(const float *__restrict__ scores,
                                                           const int64_t *__restrict__ row_score_off,
                                                           const int32_t *__restrict__ row_pos, int T, int K,
                                                           int32_t *__restrict__ sel) {
  extern __shared__ uint8_t topk_smem_raw[];
  TopkSmem<NT> &sm = *reinterpret_cast<TopkSmem<NT> *>(topk_smem_raw);
  // CTA b takes rows b, b + gridDim.x, ...
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    if (row_pos[row] < 0) continue;   // padding row of a capturable plan (uniform over the CTA)
    __syncthreads();   // shared memory of the previous row is no longer read
    select_row<NT>(scores, row_score_off, row_pos, K, sel, row, sm);
  }
}

template <int NT>
cudaError_t run_topk(int device, const float *scores, const int64_t *row_score_off, const int32_t *row_pos, int T,
                     int K, int32_t *sel, int grid, cudaStream_t s) {
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(topk_kernel<NT>, static_cast<int>(sizeof(TopkSmem<NT>)), device, smem_limit_set);
      e != cudaSuccess)
    return e;
  topk_kernel<NT><<<grid, NT, sizeof(TopkSmem<NT>), s>>>(scores, row_score_off, row_pos, T, K, sel);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const dsa_ctx *ctx, const dsa_plan_t *plan, const float *scores, int32_t *sel,
                        cudaStream_t s, int32_t *launches) {
  // up to one row per SM: 1024-thread CTAs, one row each; more rows: 512-thread
  // CTAs, two per SM, each taking rows in turn; many rows (more than two per
  // SM) of at most kShortRow keys: 256-thread CTAs, four per SM
  cudaError_t e;
  if (plan->T <= ctx->num_sms)
    e = run_topk<1024>(ctx->device, scores, plan->row_score_off, plan->row_pos, plan->T, ctx->cfg.topk, sel, std::max(1, plan->T), s);
  else if (plan->T > 2 * ctx->num_sms && static_cast<int64_t>(plan->max_pos) + 1 <= kShortRow)
    e = run_topk<256>(ctx->device, scores, plan->row_score_off, plan->row_pos, plan->T, ctx->cfg.topk, sel,
                      std::min(plan->T, 4 * ctx->num_sms), s);
  else
    e = run_topk<512>(ctx->device, scores, plan->row_score_off, plan->row_pos, plan->T, ctx->cfg.topk, sel,
                      std::min(plan->T, 2 * ctx->num_sms), s);
  *launches += 1;
  return e;
}

}  // namespace dsa
