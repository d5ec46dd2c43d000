// indexer.cu -- DSA indexer score on sm_103a tensor cores.
//
//   s[r, j] = sum_h w[r,h] * relu(q[r,h] . k[j])      (fp32; j = 0 .. pos(r))
//
// (mstar "mstar.engine.resources.dsa.manager", module summary and index_topk.)
//
// The head dots of a tile of 128 keys are one UMMA (tcgen05.mma, kind::f16,
// bf16 inputs, fp32 accumulation in TMEM):
//     D[key, n] = sum_d K[key, d] * Q[n, d],   M = 128 keys, N = G rows x Hi heads, K = Di
// Keys come from the page-resident index cache through TMA (one box per
// page-contiguous run, 128-byte swizzle); the query block of a group of G rows
// of one request is the B operand and stays in shared memory while the group's
// key tiles stream through a ring of stages.  Four epilogue warps read the
// accumulator back (thread = key = TMEM lane) and reduce over the heads with
// the relu and the head weights in registers, so the reduction needs no
// cross-lane traffic.  The accumulator is double-buffered in TMEM so the
// epilogue of tile t overlaps the MMAs of tile t+1.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread) and TMEM owner, warps 2-5 epilogue.  The grid is persistent: each
// CTA walks a tile-balanced contiguous range of the plan's work items; single-
// row groups (decode) run two CTAs per SM.
//
// The MSA block selection of decode steps runs the bf16 kernel with a
// block-maximum epilogue instead of the score store: each epilogue warp
// reduces its 32 keys' scores per block they touch (a shuffle butterfly, the
// rows of a group interleaved) and raises the row's block word with one
// atomicMax of the order key, so no token score is written or read back.
//
// The fp8 index format (132-byte keys) runs index_fp8_tc_kernel, the same
// contraction behind a code -> bf16 conversion stage.  Shapes outside the
// tensor-core instances run index_simt_kernel, one CUDA-core thread per key.
#include <cuda_runtime.h>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kEpiWarps = 4;
constexpr int kIdxThreads = 64 + 32 * kEpiWarps;

template <int HI, int DI, int G>
struct IdxTraits {
  static constexpr int CH = DI >= 64 ? 64 : DI;     // bf16 elements per swizzled row
  static constexpr int NCH = DI / CH;               // chunks along the contraction
  static constexpr int ROWB = CH * 2;               // bytes per swizzled row: 128 or 64
  static constexpr uint32_t SWZ = ROWB == 128 ? kSwizzle128 : kSwizzle64;
  static constexpr uint32_t SBO = 8 * ROWB;         // 8-row swizzle atom
  static constexpr int N = ((G * HI + 15) / 16) * 16;
  static constexpr int KSTEPS = CH / 16;            // UMMA K = 16 for bf16
  static constexpr int KT_BYTES = 128 * DI * 2;
  static constexpr int Q_BYTES = N * DI * 2;
  static constexpr int QBUF = (G == 1) ? 2 : 1;
  // single-row groups run two CTAs per SM with two stages each: two
  // independent pipelines keep more of HBM busy than one CTA with six stages
  static constexpr int STAGES_MAX = (G == 1) ? 2 : 4;
  static constexpr int STAGES = (STAGES_MAX * KT_BYTES + QBUF * Q_BYTES <= 200 * 1024) ? STAGES_MAX : 3;
  static constexpr int TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64) ? 64 : (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  static constexpr uint32_t IDESC = mma_idesc(128, N, 1u, false, false);
  // shared memory layout (bytes from a 1024-aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = OFF_K + STAGES * KT_BYTES;
  static constexpr int OFF_W = OFF_Q + QBUF * Q_BYTES;
  static constexpr int OFF_BAR = OFF_W + ((G * HI * 4 + 15) / 16) * 16;
  static constexpr int NBAR = 2 * STAGES + 2 * QBUF + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(N <= 256 && N >= 16, "UMMA N");
  static_assert((kIndexTile / 8) * NCH <= 32, "one producer lane per (box, chunk) of a tile");
  static_assert(DI % CH == 0 && CH % 16 == 0, "index dim");
  static_assert(HI % 4 == 0, "heads");
};

struct IdxParams {
  CUtensorMap tm_keys;      // index cache as [pages*P, Di] bf16, box {CH, BH}
  CUtensorMap tm_q;         // q as [T*Hi, Di] bf16, box {CH, N}
  const float *w;           // [T, Hi]
  const IdxGroup *groups;
  const IdxItem *items;
  const int32_t *cta_begin;
  const int32_t *pages;
  const int64_t *row_score_off;
  float *scores;
  uint32_t *block_keys;     // block maxima (the BMAX instances) instead of scores
  int *err;
  int P, BH, num_pages;
  int block;                // positions per block of block_keys
};

// sum_h w[h] * relu(sign * v[h]) with the weights read four at a time from
// shared memory (one broadcast load per four heads) and four independent
// accumulators (the FMA latency is not a chain over all heads), held as two
// pairs for the packed fp32 FMA (fma.rn.f32x2: each lane is the same IEEE
// fma as fmaf, so the sum is unchanged, in half the instructions).
template <int HI>
__device__ __forceinline__ float weighted_relu_sum(const float *w, const float (&v)[HI], float sign) {
  static_assert(HI % 4 == 0, "heads");
  const float4 *w4 = reinterpret_cast<const float4 *>(w);
  uint64_t a01 = 0, a23 = 0;   // (+0, +0) pairs
#pragma unroll
  for (int h = 0; h < HI; h += 4) {
    const float4 ww = w4[h / 4];
    a01 = f2_fma(f2_pack(ww.x, ww.y), f2_pack(fmaxf(sign * v[h], 0.f), fmaxf(sign * v[h + 1], 0.f)), a01);
    a23 = f2_fma(f2_pack(ww.z, ww.w), f2_pack(fmaxf(sign * v[h + 2], 0.f), fmaxf(sign * v[h + 3], 0.f)), a23);
  }
  float a0, a1, a2, a3;
  f2_unpack(a01, a0, a1);
  f2_unpack(a23, a2, a3);
  return (a0 + a1) + (a2 + a3);
}

// BMAX: the block-maximum epilogue (p.block_keys, p.block) in place of the
// score store.
template <int HI, int DI, int G, bool BMAX>
__global__ void __launch_bounds__(kIdxThreads, 2) index_tc_kernel(const __grid_constant__ IdxParams p) {
  using C = IdxTraits<HI, DI, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto kfull = [&](int s) { return bar0 + 8u * s; };
  auto kempty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto qfull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto qempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + C::QBUF + b); };
  auto afull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * C::QBUF + b); };
  auto aempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * C::QBUF + 2 + b); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *wsm = reinterpret_cast<float *>(smem + C::OFF_W);

  const int warp = threadIdx.x / 32;
  const int lane = lane_id();
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kfull(s), 1);
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < C::QBUF; ++b) {
      mbar_init(qfull(b), 1);
      mbar_init(qempty(b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), 32 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_keys);
    tma_prefetch_desc(&p.tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t kphase = 0;
    int qb = -1, qcount = 0, cur_group = -1;
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      const IdxGroup g = p.groups[item.group];
      if (item.group != cur_group) {
        cur_group = item.group;
        qb = qcount % C::QBUF;
        const uint32_t use = qcount / C::QBUF;
        ++qcount;
        bool qok = true;
        if (lane == 0) {
          qok = mbar_wait(qempty(qb), (use & 1) ^ 1, abort_flag, p.err);
          if (qok) {
            mbar_arrive_expect_tx(qfull(qb), C::Q_BYTES);
            for (int c = 0; c < C::NCH; ++c)
              tma_load_2d(sbase + C::OFF_Q + qb * C::Q_BYTES + c * C::N * C::ROWB, &p.tm_q, c * C::CH,
                          g.row0 * HI, qfull(qb));
          }
        }
        if (__shfl_sync(0xffffffffu, qok ? 1 : 0, 0) == 0) break;
      }
      const int nrows_total = g.lead + g.pos0 + g.nrows;  // tile rows: lead rows, then keys 0 .. pos0+nrows-1
      // raw page id of this lane's box of tile t (kNoBox: the tile has no box
      // for this lane; -1: past the request's pages), looked up four tiles
      // ahead of its issue (a shift queue in registers); the check and the
      // cache row come when the tile is issued
      auto box_page = [&](int t) -> int {
        const int nb = t < item.tile1 ? (min(128, nrows_total - t * 128) + p.BH - 1) / p.BH : 0;
        if (lane >= nb) return kNoBox;
        // (32-bit: a slot is the tile's first slot, page_start - lead >= 0, plus a row)
        const uint32_t pi = (static_cast<uint32_t>(g.page_start - g.lead) + static_cast<uint32_t>(t * 128 + lane * p.BH)) /
                            static_cast<uint32_t>(p.P);
        return pi < static_cast<uint32_t>(g.npages) ? __ldg(p.pages + g.page_off + pi) : -1;
      };
      // physical cache row of this lane's box of tile t, or -1
      auto box_row = [&](int t, int page) -> int {
        if (page == kNoBox) return -1;
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.err, kErrBounds);
          return -1;
        }
        const uint32_t slot = static_cast<uint32_t>(g.page_start - g.lead) + static_cast<uint32_t>(t * 128 + lane * p.BH);
        return page * p.P + static_cast<int>(slot % static_cast<uint32_t>(p.P));
      };
      int la0 = box_page(item.tile0), la1 = box_page(item.tile0 + 1), la2 = box_page(item.tile0 + 2),
          la3 = box_page(item.tile0 + 3);
      // single-row (decode) score launches stream each key once: the keys go
      // into L2 evict-first, so the scores (stored evict-last) are still there
      // when the top-k reads them back; row groups re-read their keys
      constexpr bool kHint = G == 1 && !BMAX;
      const uint64_t kpol = kHint ? l2_policy_evict_first() : 0;
      for (int t = item.tile0; t < item.tile1; ++t) {
        const int nkeys = min(128, nrows_total - t * 128);
        const int nbox = (nkeys + p.BH - 1) / p.BH;
        const int myrow = box_row(t, la0);
        la0 = la1;
        la1 = la2;
        la2 = la3;
        la3 = box_page(t + 4);
        const uint32_t valid = __ballot_sync(0xffffffffu, myrow >= 0);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(kempty(stage), kphase ^ 1, abort_flag, p.err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t bytes = __popc(valid) * p.BH * C::ROWB * C::NCH;
        if (lane == 0) {
          if (bytes) mbar_arrive_expect_tx(kfull(stage), bytes);
          else mbar_arrive(kfull(stage));
        }
        {
          // every (box, chunk) of the tile from its own lane: the tile's loads
          // go out as one warp instruction, not one by one from lane 0 (a
          // box has >= 8 rows, so nbox * NCH <= 32)
          const int b = lane / C::NCH, c = lane % C::NCH;
          const int row = __shfl_sync(0xffffffffu, myrow, b & 31);
          const uint32_t dst = sbase + C::OFF_K + stage * C::KT_BYTES + c * 128 * C::ROWB + b * p.BH * C::ROWB;
          if (b < nbox && row >= 0) {
            if constexpr (kHint) tma_load_2d_hint(dst, &p.tm_keys, c * C::CH, row, kfull(stage), kpol);
            else tma_load_2d(dst, &p.tm_keys, c * C::CH, row, kfull(stage));
          }
        }
        if (++stage == C::STAGES) {
          stage = 0;
          kphase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t kphase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      int qb = -1, qcount = 0, cur_group = -1;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const IdxItem item = p.items[it];
        if (item.group != cur_group) {
          cur_group = item.group;
          qb = qcount % C::QBUF;
          const uint32_t use = qcount / C::QBUF;
          ++qcount;
          if (!mbar_wait(qfull(qb), use & 1, abort_flag, p.err)) break;
        }
        const uint32_t qaddr = sbase + C::OFF_Q + qb * C::Q_BYTES;
        for (int t = item.tile0; t < item.tile1; ++t) {
          if (!mbar_wait(kfull(stage), kphase, abort_flag, p.err)) { ok = false; break; }
          if (!mbar_wait(aempty(acc), aphase ^ 1, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = sbase + C::OFF_K + stage * C::KT_BYTES;
          const uint32_t d = tmem_base + acc * C::N;
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
            for (int k = 0; k < C::KSTEPS; ++k) {
              const uint64_t ad = smem_desc(kaddr + c * 128 * C::ROWB + k * 32, 16, C::SBO, C::SWZ);
              const uint64_t bd = smem_desc(qaddr + c * C::N * C::ROWB + k * 32, 16, C::SBO, C::SWZ);
              mma_f16_ss(d, ad, bd, C::IDESC, (c | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit(kempty(stage));
          mma_commit(afull(acc));
          if (++stage == C::STAGES) {
            stage = 0;
            kphase ^= 1;
          }
          acc ^= 1;
          if (acc == 0) aphase ^= 1;
        }
        // the query block is free once the group's last MMA completes
        const bool last_of_group = (it + 1 >= it1) || (p.items[it + 1].group != cur_group);
        if (last_of_group) mma_commit(qempty(qb));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;              // 0..127
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int m = quad * 32 + lane;               // key within the tile
    int acc = 0;
    uint32_t aphase = 0;
    int cur_group = -1;
    int64_t soff[G];
    int nrows = 0, pos0 = 0, lead = 0;
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      if (item.group != cur_group) {
        cur_group = item.group;
        const IdxGroup g = p.groups[item.group];
        nrows = g.nrows;
        pos0 = g.pos0;
        lead = g.lead;
        named_bar_sync(1, 32 * kEpiWarps);
        for (int i = et; i < G * HI; i += 32 * kEpiWarps)
          wsm[i] = (i < nrows * HI) ? p.w[static_cast<int64_t>(g.row0) * HI + i] : 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          soff[gg] = gg < nrows ? p.row_score_off[g.row0 + gg] : 0;
          if constexpr (BMAX) soff[gg] = block_key_base(soff[gg], g.row0 + gg, p.block);
        }
        named_bar_sync(1, 32 * kEpiWarps);
      }
      const uint64_t spol = (G == 1 && !BMAX) ? l2_policy_evict_last() : 0;
      bool ok = true;
      for (int t = item.tile0; t < item.tile1; ++t) {
        // warp-uniform, as the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(afull(acc), aphase, abort_flag, p.err))) { ok = false; break; }
        tc_fence_after();
        const int key = t * 128 + m - lead;   // < 0: a slot before the span's token 0
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::N;
        float sv[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          sv[gg] = 0.f;
          if (gg < nrows) {
            float s = 0.f;
            if constexpr (HI >= 16) {
              float v[HI];
#pragma unroll
              for (int h0 = 0; h0 < HI; h0 += 16) tmem_ld16(tbase + gg * HI + h0, *reinterpret_cast<float(*)[16]>(v + h0));
              tmem_ld_wait();
              s = weighted_relu_sum<HI>(wsm + gg * HI, v, 1.f);
            } else {
              float v[4];
#pragma unroll
              for (int h0 = 0; h0 < HI; h0 += 4) {
                tmem_ld4(tbase + gg * HI + h0, v);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 4; ++h) s = fmaf(wsm[gg * HI + h0 + h], fmaxf(v[h], 0.f), s);
              }
            }
            if constexpr (!BMAX) {
              if (key >= 0 && key <= pos0 + gg) {
                if constexpr (G == 1) st_global_hint(p.scores + soff[gg] + key, s, spol);
                else p.scores[soff[gg] + key] = s;
              }
            } else {
              sv[gg] = s;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(aempty(acc));   // the accumulator is read: the next tile's MMAs may take it
        if constexpr (BMAX) {
          // block maxima of the warp's 32 consecutive keys: a butterfly max
          // per row (the rows' shuffles interleave) and one atomic per row
          // and block; a warp that straddles a block edge (a lead or a block
          // size that is not a multiple of 32) takes one reduce per block
          const int kfirst = t * 128 + quad * 32 - lead;   // the key of lane 0
          const int klast = kfirst + 31;
          if (klast >= 0) {
            const int kmin = kfirst > 0 ? kfirst : 0;
            const int b_hi = klast / p.block;
            if (b_hi * p.block <= kmin) {   // one block (warp-uniform)
              float mx[G];
              uint32_t any[G];
#pragma unroll
              for (int gg = 0; gg < G; ++gg) {
                const bool vis = gg < nrows && key >= 0 && key <= pos0 + gg;
                mx[gg] = vis ? sv[gg] : -INFINITY;
                any[gg] = __ballot_sync(0xffffffffu, vis);
              }
#pragma unroll
              for (int o = 16; o; o >>= 1)
#pragma unroll
                for (int gg = 0; gg < G; ++gg) mx[gg] = fmaxf(mx[gg], __shfl_xor_sync(0xffffffffu, mx[gg], o));
              if (lane == 0) {
#pragma unroll
                for (int gg = 0; gg < G; ++gg)
                  if (any[gg]) atomicMax(p.block_keys + soff[gg] + b_hi, score_order_key(mx[gg]));
              }
            } else {
              const int b_lo = kmin / p.block;
#pragma unroll
              for (int gg = 0; gg < G; ++gg) {
                if (gg < nrows) {
                  const bool vis = key >= 0 && key <= pos0 + gg;
                  const uint32_t kk = vis ? score_order_key(sv[gg]) : 0u;
                  for (int b = b_lo; b <= b_hi; ++b) {   // warp-uniform bounds
                    const bool in = key >= b * p.block && key < (b + 1) * p.block;
                    const uint32_t mk = __reduce_max_sync(0xffffffffu, in ? kk : 0u);
                    if (lane == 0 && mk != 0u) atomicMax(p.block_keys + soff[gg] + b, mk);
                  }
                }
              }
            }
          }
        }
        acc ^= 1;
        if (acc == 0) aphase ^= 1;
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// CUDA-core fallback: one block of 128 threads per work item, thread = key.
// Handles any head count / dim and both index formats (fp8: code * scale).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) index_simt_kernel(const uint16_t *__restrict__ q, const float *__restrict__ w,
                                                          const uint8_t *__restrict__ cache,
                                                          const IdxGroup *__restrict__ groups,
                                                          const IdxItem *__restrict__ items,
                                                          const int32_t *__restrict__ pages,
                                                          const int64_t *__restrict__ row_score_off,
                                                          float *__restrict__ scores, int *err, int Hi, int Di,
                                                          int P, int fp8, int num_pages,
                                                          const int32_t *__restrict__ n_items_dev) {
  extern __shared__ float qs[];  // [Hi * Di] of one row, then [Hi] weights
  if (n_items_dev && static_cast<int>(blockIdx.x) >= *n_items_dev) return;   // capturable plan: past its items
  const IdxItem item = items[blockIdx.x];
  if (item.group < 0) return;   // padding of a capturable plan
  const IdxGroup g = groups[item.group];
  for (int gg = 0; gg < g.nrows; ++gg) {
    const int row = g.row0 + gg;
    __syncthreads();
    for (int i = threadIdx.x; i < Hi * Di; i += blockDim.x)
      qs[i] = __uint_as_float(static_cast<uint32_t>(q[static_cast<int64_t>(row) * Hi * Di + i]) << 16);
    for (int i = threadIdx.x; i < Hi; i += blockDim.x) qs[Hi * Di + i] = w[static_cast<int64_t>(row) * Hi + i];
    __syncthreads();
    const int pos = g.pos0 + gg;
    for (int t = item.tile0; t < item.tile1; ++t) {
      const int key = t * 128 + threadIdx.x - g.lead;
      if (key < 0 || key > pos) continue;
      const int64_t slot = static_cast<int64_t>(g.page_start) + key;
      const int64_t pi = slot / P;
      int page = -1;
      if (pi < g.npages) page = pages[g.page_off + pi];
      if (page < 0 || page >= num_pages) {
        atomicOr(err, kErrBounds);
        continue;
      }
      const int64_t prow = static_cast<int64_t>(page) * P + slot % P;
      float s = 0.f;
      if (!fp8) {
        const uint16_t *k = reinterpret_cast<const uint16_t *>(cache) + prow * Di;
        for (int h = 0; h < Hi; ++h) {
          float d = 0.f;
          for (int i = 0; i < Di; ++i) d = fmaf(qs[h * Di + i], __uint_as_float(static_cast<uint32_t>(k[i]) << 16), d);
          s = fmaf(qs[Hi * Di + h], fmaxf(d, 0.f), s);
        }
      } else {
        const uint8_t *base = cache + static_cast<int64_t>(page) * P * (Di + 4);
        const uint8_t *k = base + (slot % P) * Di;
        const float scale = *reinterpret_cast<const float *>(base + static_cast<int64_t>(P) * Di + (slot % P) * 4);
        for (int h = 0; h < Hi; ++h) {
          float d = 0.f;
          for (int i = 0; i < Di; ++i) {
            __nv_fp8_e4m3 c;
            c.__x = k[i];
            d = fmaf(qs[h * Di + i], static_cast<float>(c), d);
          }
          s = fmaf(qs[Hi * Di + h], fmaxf(d * scale, 0.f), s);
        }
      }
      scores[row_score_off[row] + key] = s;
    }
  }
}

template <int HI, int DI, int G>
cudaError_t run_tc(const dsa_ctx *ctx, const dsa_plan_t *plan, const IdxSet &set, const void *q, const float *w,
                   const void *cache, float *scores, cudaStream_t s, int BH, uint32_t *block_keys = nullptr,
                   int block = 0) {
  using C = IdxTraits<HI, DI, G>;
  IdxParams prm{};
  const dsa_config_t &c = ctx->cfg;
  const CUtensorMapSwizzle swz = C::ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!encode_tiled_2d(&prm.tm_keys, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(cache), DI,
                       static_cast<uint64_t>(plan->cache_pages) * c.page_size, DI * 2, C::CH, BH, swz))
    return cudaErrorInvalidValue;
  if (!encode_tiled_2d(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q), DI,
                       static_cast<uint64_t>(plan->T) * HI, DI * 2, C::CH, C::N, swz))
    return cudaErrorInvalidValue;
  prm.w = w;
  prm.groups = set.groups;
  prm.items = set.items;
  prm.cta_begin = set.cta_begin;
  prm.pages = plan->pages;
  prm.row_score_off = plan->row_score_off;
  prm.scores = scores;
  prm.block_keys = block_keys;
  prm.block = block;
  prm.err = ctx->err;
  prm.P = c.page_size;
  prm.BH = BH;
  prm.num_pages = plan->cache_pages;
  auto kern = block_keys ? index_tc_kernel<HI, DI, G, true> : index_tc_kernel<HI, DI, G, false>;
  static std::atomic<uint64_t> smem_limit_set[2] = {0, 0};
  if (cudaError_t e = ensure_smem_limit(kern, C::SMEM, ctx->device, smem_limit_set[block_keys ? 1 : 0]);
      e != cudaSuccess)
    return e;
  kern<<<set.n_ctas, kIdxThreads, C::SMEM, s>>>(prm);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// fp8 index keys on the tensor cores.  A 132-byte key is 128 e4m3 codes and
// one fp32 scale (LLMServingSim, "What the KV cache actually holds"), stored
// page-blocked: [P x 128 codes][P x fp32 scale] per page.  TMA brings each
// tile's code rows (3-D map: byte, slot, page) and scales (2-D map over the
// scale blocks) into a staging ring; four converter warps turn the codes into
// bf16 tiles (every e4m3 value is exactly a bf16 value), so the UMMA chain is
// the bf16 one.  The epilogue applies the key's scale:
//     relu(scale * d) = |scale| * relu(sign(scale) * d)
// so s = |scale| * sum_h w_h relu(+-d_h), one multiply per key instead of one
// per head.  For a power-of-two scale the two forms are equal; for any other
// scale (the quantiser writes amax / 448) they differ by where one fp32
// rounding falls, a relative difference of order 2^-24 in the score.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2-5
// epilogue, warps 6-9 converters (thread = key of the tile).
// ---------------------------------------------------------------------------
constexpr int kCvtWarps = 4;
constexpr int kFp8Threads = 64 + 32 * kEpiWarps + 32 * kCvtWarps;

template <int G>
struct IdxF8Traits {
  static constexpr int HI = 64, DI = 128;
  static constexpr int N = G * HI;
  static constexpr int CODE_BYTES = 128 * 128;           // staged codes of one tile (128-byte swizzle)
  static constexpr int SC_BYTES = 128 * 4;               // scales of one tile
  // Staged scales: a TMA destination in shared memory must be 128-byte
  // aligned, so box b of a tile lands at b * max(128, 4 * BH) bytes (up to 16
  // boxes of 8 keys: 2 KB per stage).
  static constexpr int SC8_BYTES = 2048;
  static constexpr int S8 = 4;                           // staging stages
  static constexpr int KT_BYTES = 128 * DI * 2;          // converted bf16 tile: 2 swizzled 64-column chunks
  static constexpr int QBUF = (G == 1) ? 2 : 1;
  static constexpr int S16 = (G == 1) ? 3 : 2;           // converted stages
  // Scale ring read by the epilogue.  The converter writes the scale of tile
  // n only after the MMA of tile n - S16 has finished, which waited for the
  // epilogue to release the accumulator of tile n - S16 - 2; S16 + 2 slots
  // keep a slot alive until the epilogue of its tile has read it.
  static constexpr int SCR = S16 + 2;
  static constexpr int Q_BYTES = N * DI * 2;
  static constexpr int TMEM_COLS = (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  static constexpr uint32_t IDESC = mma_idesc(128, N, 1u, false, false);
  static constexpr int OFF_C8 = 0;
  static constexpr int OFF_K = OFF_C8 + S8 * CODE_BYTES;
  static constexpr int OFF_Q = OFF_K + S16 * KT_BYTES;
  static constexpr int OFF_SC8 = OFF_Q + QBUF * Q_BYTES;
  static constexpr int OFF_SC = OFF_SC8 + S8 * SC8_BYTES;
  static constexpr int OFF_W = OFF_SC + SCR * SC_BYTES;
  static constexpr int OFF_BAR = OFF_W + G * HI * 4;
  static constexpr int NBAR = 2 * S8 + 2 * S16 + 2 * QBUF + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(N <= 256, "UMMA N");
};

struct IdxF8Params {
  CUtensorMap tm_codes;     // codes as [pages][P][128] uint8, box {128, BH, 1}, 128-byte swizzle
  CUtensorMap tm_scales;    // scales as [pages][P] fp32 (page stride P*132 bytes), box {BH, 1}
  CUtensorMap tm_q;         // q as [T*Hi, Di] bf16, box {64, N}
  const float *w;
  const IdxGroup *groups;
  const IdxItem *items;
  const int32_t *cta_begin;
  const int32_t *pages;
  const int64_t *row_score_off;
  float *scores;
  int *err;
  int P, BH, num_pages;
};

// e4m3 -> bf16 of the four codes of a 32-bit word (lowest byte first), two
// bf16 per output word
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  uint32_t o[2];
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    const __half2_raw hr =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((w >> (16 * hlf)) & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    o[hlf] = *reinterpret_cast<const uint32_t *>(&b);
  }
  return make_uint2(o[0], o[1]);
}

template <int G>
__global__ void __launch_bounds__(kFp8Threads, 1) index_fp8_tc_kernel(const __grid_constant__ IdxF8Params p) {
  using C = IdxF8Traits<G>;
  constexpr int HI = C::HI;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto c8full = [&](int s) { return bar0 + 8u * s; };
  auto c8empty = [&](int s) { return bar0 + 8u * (C::S8 + s); };
  auto kfull = [&](int s) { return bar0 + 8u * (2 * C::S8 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (2 * C::S8 + C::S16 + s); };
  auto qfull = [&](int b) { return bar0 + 8u * (2 * C::S8 + 2 * C::S16 + b); };
  auto qempty = [&](int b) { return bar0 + 8u * (2 * C::S8 + 2 * C::S16 + C::QBUF + b); };
  auto afull = [&](int b) { return bar0 + 8u * (2 * C::S8 + 2 * C::S16 + 2 * C::QBUF + b); };
  auto aempty = [&](int b) { return bar0 + 8u * (2 * C::S8 + 2 * C::S16 + 2 * C::QBUF + 2 + b); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *wsm = reinterpret_cast<float *>(smem + C::OFF_W);
  float *scr = reinterpret_cast<float *>(smem + C::OFF_SC);

  const int warp = threadIdx.x / 32;
  const int lane = lane_id();
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];
  const int sc_stride = max(32, p.BH);   // floats between the staged scale boxes of a tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S8; ++s) {
      mbar_init(c8full(s), 1);
      mbar_init(c8empty(s), 32 * kCvtWarps);
    }
    for (int s = 0; s < C::S16; ++s) {
      mbar_init(kfull(s), 32 * kCvtWarps);
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < C::QBUF; ++b) {
      mbar_init(qfull(b), 1);
      mbar_init(qempty(b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), 32 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_codes);
    tma_prefetch_desc(&p.tm_scales);
    tma_prefetch_desc(&p.tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int s8 = 0;
    uint32_t ph8 = 0;
    int qcount = 0, cur_group = -1;
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      const IdxGroup g = p.groups[item.group];
      if (item.group != cur_group) {
        cur_group = item.group;
        const int qb = qcount % C::QBUF;
        const uint32_t use = qcount / C::QBUF;
        ++qcount;
        bool qok = true;
        if (lane == 0) {
          qok = mbar_wait(qempty(qb), (use & 1) ^ 1, abort_flag, p.err);
          if (qok) {
            mbar_arrive_expect_tx(qfull(qb), C::Q_BYTES);
            for (int c = 0; c < C::DI / 64; ++c)
              tma_load_2d(sbase + C::OFF_Q + qb * C::Q_BYTES + c * C::N * 128, &p.tm_q, c * 64, g.row0 * HI,
                          qfull(qb));
          }
        }
        if (__shfl_sync(0xffffffffu, qok ? 1 : 0, 0) == 0) break;
      }
      const int nrows_total = g.lead + g.pos0 + g.nrows;  // tile rows: lead rows, then keys 0 .. pos0+nrows-1
      // raw page id of this lane's box of tile t (kNoBox: no box for this lane;
      // -1: past the request's pages), looked up four tiles ahead of its issue
      // (a shift queue in registers) and checked when the tile is issued
      auto box_page = [&](int t) -> int {
        const int nb = t < item.tile1 ? (min(128, nrows_total - t * 128) + p.BH - 1) / p.BH : 0;
        if (lane >= nb) return kNoBox;
        // (32-bit: a slot is the tile's first slot, page_start - lead >= 0, plus a row)
        const uint32_t pi = (static_cast<uint32_t>(g.page_start - g.lead) + static_cast<uint32_t>(t * 128 + lane * p.BH)) /
                            static_cast<uint32_t>(p.P);
        return pi < static_cast<uint32_t>(g.npages) ? __ldg(p.pages + g.page_off + pi) : -1;
      };
      // (page, slot) of this lane's box of tile t, page -1 if there is none
      auto box_at = [&](int t, int page, int &slot_out) -> int {
        slot_out = 0;
        if (page == kNoBox) return -1;
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.err, kErrBounds);
          return -1;
        }
        slot_out = static_cast<int>((static_cast<uint32_t>(g.page_start - g.lead) + static_cast<uint32_t>(t * 128 + lane * p.BH)) %
                                    static_cast<uint32_t>(p.P));
        return page;
      };
      int lp0 = box_page(item.tile0), lp1 = box_page(item.tile0 + 1), lp2 = box_page(item.tile0 + 2),
          lp3 = box_page(item.tile0 + 3);
      for (int t = item.tile0; t < item.tile1; ++t) {
        const int nkeys = min(128, nrows_total - t * 128);
        const int nbox = (nkeys + p.BH - 1) / p.BH;
        int myslot;
        const int mypage = box_at(t, lp0, myslot);
        lp0 = lp1;
        lp1 = lp2;
        lp2 = lp3;
        lp3 = box_page(t + 4);
        const uint32_t valid = __ballot_sync(0xffffffffu, mypage >= 0);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(c8empty(s8), ph8 ^ 1, abort_flag, p.err);
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
        const uint32_t bytes = __popc(valid) * p.BH * (128 + 4);
        if (lane == 0) {
          if (bytes) mbar_arrive_expect_tx(c8full(s8), bytes);
          else mbar_arrive(c8full(s8));
        }
        {
          // the codes and the scales of every box from their own lanes (a
          // box has >= 8 rows, so 2 * nbox <= 32)
          const int b = lane >> 1;
          const int page = __shfl_sync(0xffffffffu, mypage, b);
          const int slot = __shfl_sync(0xffffffffu, myslot, b);
          if (b < nbox && page >= 0) {
            if ((lane & 1) == 0)
              tma_load_3d(sbase + C::OFF_C8 + s8 * C::CODE_BYTES + b * p.BH * 128, &p.tm_codes, 0, slot, page,
                          c8full(s8));
            else
              tma_load_2d(sbase + C::OFF_SC8 + s8 * C::SC8_BYTES + b * sc_stride * 4, &p.tm_scales, slot, page,
                          c8full(s8));
          }
        }
        if (++s8 == C::S8) {
          s8 = 0;
          ph8 ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aphase = 0;
      int qb = 0, qcount = 0, cur_group = -1;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const IdxItem item = p.items[it];
        if (item.group != cur_group) {
          cur_group = item.group;
          qb = qcount % C::QBUF;
          const uint32_t use = qcount / C::QBUF;
          ++qcount;
          if (!mbar_wait(qfull(qb), use & 1, abort_flag, p.err)) break;
        }
        const uint32_t qaddr = sbase + C::OFF_Q + qb * C::Q_BYTES;
        for (int t = item.tile0; t < item.tile1; ++t) {
          if (!mbar_wait(kfull(st), ph, abort_flag, p.err)) { ok = false; break; }
          if (!mbar_wait(aempty(acc), aphase ^ 1, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = sbase + C::OFF_K + st * C::KT_BYTES;
          const uint32_t d = tmem_base + acc * C::N;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc(kaddr + c * 128 * 128 + k * 32, 16, 1024, kSwizzle128);
              const uint64_t bd = smem_desc(qaddr + c * C::N * 128 + k * 32, 16, 1024, kSwizzle128);
              mma_f16_ss(d, ad, bd, C::IDESC, (c | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit(kempty(st));
          mma_commit(afull(acc));
          if (++st == C::S16) {
            st = 0;
            ph ^= 1;
          }
          acc ^= 1;
          if (acc == 0) aphase ^= 1;
        }
        const bool last_of_group = (it + 1 >= it1) || (p.items[it + 1].group != cur_group);
        if (last_of_group) mma_commit(qempty(qb));
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    int acc = 0;
    uint32_t aphase = 0;
    int sc = 0;
    int cur_group = -1;
    int64_t soff[G];
    int nrows = 0, pos0 = 0, lead = 0;
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      if (item.group != cur_group) {
        cur_group = item.group;
        const IdxGroup g = p.groups[item.group];
        nrows = g.nrows;
        pos0 = g.pos0;
        lead = g.lead;
        named_bar_sync(1, 32 * kEpiWarps);
        for (int i = et; i < G * HI; i += 32 * kEpiWarps)
          wsm[i] = (i < nrows * HI) ? p.w[static_cast<int64_t>(g.row0) * HI + i] : 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) soff[gg] = gg < nrows ? p.row_score_off[g.row0 + gg] : 0;
        named_bar_sync(1, 32 * kEpiWarps);
      }
      bool ok = true;
      for (int t = item.tile0; t < item.tile1; ++t) {
        if (!__all_sync(0xffffffffu, mbar_wait(afull(acc), aphase, abort_flag, p.err))) { ok = false; break; }
        tc_fence_after();
        const float scale = scr[sc * 128 + m];
        const float mag = fabsf(scale);
        const bool neg = scale < 0.f;
        const bool all_pos = __all_sync(0xffffffffu, !neg);
        const int key = t * 128 + m - lead;   // < 0: a slot before the span's token 0
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::N;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          if (gg < nrows) {
            float v[HI];
#pragma unroll
            for (int h0 = 0; h0 < HI; h0 += 16)
              tmem_ld16(tbase + gg * HI + h0, *reinterpret_cast<float(*)[16]>(v + h0));
            tmem_ld_wait();
            // (the quantiser's scales are >= 0: a warp with no negative scale
            // takes the relu without the sign multiply)
            const float s = all_pos ? weighted_relu_sum<HI>(wsm + gg * HI, v, 1.f)
                                    : weighted_relu_sum<HI>(wsm + gg * HI, v, neg ? -1.f : 1.f);
            if (key >= 0 && key <= pos0 + gg) p.scores[soff[gg] + key] = s * mag;
          }
        }
        tc_fence_before();
        mbar_arrive(aempty(acc));
        acc ^= 1;
        if (acc == 0) aphase ^= 1;
        if (++sc == C::SCR) sc = 0;
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ converters
    // thread c converts key c of each tile: its 128 codes (staged with the
    // 128-byte swizzle) become 256 bytes of bf16 in two swizzled 64-column
    // chunks, the layout TMA gives a bf16 tile
    const int c = threadIdx.x - (64 + 32 * kEpiWarps);
    int s8 = 0, st = 0, sc = 0;
    uint32_t ph8 = 0, ph = 0;
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      bool ok = true;
      for (int t = item.tile0; t < item.tile1; ++t) {
        if (!mbar_wait(c8full(s8), ph8, abort_flag, p.err)) { ok = false; break; }
        const uint8_t *src = smem + C::OFF_C8 + s8 * C::CODE_BYTES + c * 128;
        uint4 in[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) in[i] = *reinterpret_cast<const uint4 *>(src + ((i ^ (c & 7)) << 4));
        const float scale = reinterpret_cast<const float *>(smem + C::OFF_SC8 + s8 * C::SC8_BYTES)
            [(c / p.BH) * sc_stride + c % p.BH];
        mbar_arrive(c8empty(s8));
        if (++s8 == C::S8) {
          s8 = 0;
          ph8 ^= 1;
        }
        if (!mbar_wait(kempty(st), ph ^ 1, abort_flag, p.err)) { ok = false; break; }
        const uint32_t row = sbase + C::OFF_K + st * C::KT_BYTES + c * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // codes 16i .. 16i+15 -> bf16 columns 16i .. 16i+15: chunk (16i)/64,
          // 16-byte pieces 2(i%4) and 2(i%4)+1 of the row
          const uint2 a = e4m3x4_to_bf16x4(in[i].x), b = e4m3x4_to_bf16x4(in[i].y);
          const uint2 e = e4m3x4_to_bf16x4(in[i].z), f = e4m3x4_to_bf16x4(in[i].w);
          const uint32_t chunk = row + (i / 4) * (128 * 128);
          const int piece = 2 * (i % 4);
          st_shared_v4(chunk + ((piece ^ (c & 7)) << 4), make_uint4(a.x, a.y, b.x, b.y));
          st_shared_v4(chunk + (((piece + 1) ^ (c & 7)) << 4), make_uint4(e.x, e.y, f.x, f.y));
        }
        scr[sc * 128 + c] = scale;
        fence_proxy_async_smem();
        mbar_arrive(kfull(st));
        if (++st == C::S16) {
          st = 0;
          ph ^= 1;
        }
        if (++sc == C::SCR) sc = 0;
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int G>
cudaError_t run_fp8(const dsa_ctx *ctx, const dsa_plan_t *plan, const IdxSet &set, const void *q, const float *w,
                    const void *cache, float *scores, cudaStream_t s, int BH) {
  using C = IdxF8Traits<G>;
  const dsa_config_t &c = ctx->cfg;
  IdxF8Params prm{};
  const uint64_t P = static_cast<uint64_t>(c.page_size);
  {
    const uint64_t dims[3] = {128, P, static_cast<uint64_t>(plan->cache_pages)};
    const uint64_t strides[2] = {128, P * 132};
    const uint32_t box[3] = {128, static_cast<uint32_t>(BH), 1};
    if (!encode_tiled_3d(&prm.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void *>(cache), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (!encode_tiled_2d(&prm.tm_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       static_cast<uint8_t *>(const_cast<void *>(cache)) + P * 128, P, plan->cache_pages, P * 132,
                       BH, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (!encode_tiled_2d(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q), C::DI,
                       static_cast<uint64_t>(plan->T) * C::HI, C::DI * 2, 64, C::N, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  prm.w = w;
  prm.groups = set.groups;
  prm.items = set.items;
  prm.cta_begin = set.cta_begin;
  prm.pages = plan->pages;
  prm.row_score_off = plan->row_score_off;
  prm.scores = scores;
  prm.err = ctx->err;
  prm.P = c.page_size;
  prm.BH = BH;
  prm.num_pages = plan->cache_pages;
  auto kern = index_fp8_tc_kernel<G>;
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(kern, C::SMEM, ctx->device, smem_limit_set); e != cudaSuccess) return e;
  kern<<<set.n_ctas, kFp8Threads, C::SMEM, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool indexer_tc_supported(const dsa_config_t &c, int G) {
  if (c.index_fmt == DSA_INDEX_FP8_132)
    return c.index_heads == 64 && c.index_dim == 128 && c.page_size % 8 == 0 && (G == 1 || G == 4);
  if (c.index_heads == 64 && c.index_dim == 128) return G == 1 || G == 4;
  if (c.index_heads == 4 && c.index_dim == 32) return G == 1 || G == 4;
  return false;
}

int indexer_group_rows(const dsa_config_t &c) { return indexer_tc_supported(c, 4) ? 4 : 1; }

int indexer_ctas_per_sm(const dsa_config_t &c, int G) { return (c.index_fmt == DSA_INDEX_BF16 && G == 1) ? 2 : 1; }

cudaError_t launch_index_scores(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                const void *cache, float *scores, cudaStream_t s, int32_t *launches) {
  const dsa_config_t &c = ctx->cfg;
  const int BH = plan->box_rows;
  for (int si = 0; si < 2; ++si) {
    const IdxSet &set = plan->idx[si];
    if (set.n_items == 0) continue;
    const bool tc = indexer_tc_supported(c, set.G) && BH >= 8;
    cudaError_t e = cudaSuccess;
    if (tc && c.index_fmt == DSA_INDEX_FP8_132) {
      e = set.G == 1 ? run_fp8<1>(ctx, plan, set, q, w, cache, scores, s, BH)
                     : run_fp8<4>(ctx, plan, set, q, w, cache, scores, s, BH);
    } else if (tc) {
      if (c.index_heads == 64 && set.G == 1) e = run_tc<64, 128, 1>(ctx, plan, set, q, w, cache, scores, s, BH);
      else if (c.index_heads == 64) e = run_tc<64, 128, 4>(ctx, plan, set, q, w, cache, scores, s, BH);
      else if (set.G == 1) e = run_tc<4, 32, 1>(ctx, plan, set, q, w, cache, scores, s, BH);
      else e = run_tc<4, 32, 4>(ctx, plan, set, q, w, cache, scores, s, BH);
    } else {
      const size_t sm = (static_cast<size_t>(c.index_heads) * c.index_dim + c.index_heads) * sizeof(float);
      if (sm > 48 * 1024) {
        e = cudaFuncSetAttribute(index_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
        if (e != cudaSuccess) return e;
      }
      index_simt_kernel<<<set.n_items, 128, sm, s>>>(static_cast<const uint16_t *>(q), w,
                                                     static_cast<const uint8_t *>(cache), set.groups, set.items,
                                                     plan->pages, plan->row_score_off, scores, ctx->err,
                                                     c.index_heads, c.index_dim, c.page_size,
                                                     c.index_fmt == DSA_INDEX_FP8_132, plan->cache_pages,
                                                     plan->capturable ? plan->counts + 1 : nullptr);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

// The block-maximum epilogue pays off where the indexer streams keys (single-
// row groups: the score writes and the selection's re-read are a real share
// of the traffic).  Multi-row groups are bound by the epilogue's arithmetic,
// where the extra cross-lane reduction costs more than the score stores it
// saves, so plans with such groups keep the score path.
bool index_block_keys_supported(const dsa_ctx *ctx, const dsa_plan_t *plan) {
  const dsa_config_t &c = ctx->cfg;
  if (c.index_fmt != DSA_INDEX_BF16 || plan->box_rows < 8 || plan->capturable) return false;
  if (plan->idx[1].n_items > 0) return false;
  return plan->idx[0].n_items == 0 || indexer_tc_supported(c, plan->idx[0].G);
}

cudaError_t launch_index_block_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                    const void *cache, uint32_t *block_keys, int block, cudaStream_t s,
                                    int32_t *launches) {
  if (!index_block_keys_supported(ctx, plan) || block <= 0) return cudaErrorNotSupported;
  const dsa_config_t &c = ctx->cfg;
  const int BH = plan->box_rows;
  for (int si = 0; si < 2; ++si) {
    const IdxSet &set = plan->idx[si];
    if (set.n_items == 0) continue;
    uint32_t *bk = block_keys;
    cudaError_t e;
    if (c.index_heads == 64 && set.G == 1) e = run_tc<64, 128, 1>(ctx, plan, set, q, w, cache, nullptr, s, BH, bk, block);
    else if (c.index_heads == 64) e = run_tc<64, 128, 4>(ctx, plan, set, q, w, cache, nullptr, s, BH, bk, block);
    else if (set.G == 1) e = run_tc<4, 32, 1>(ctx, plan, set, q, w, cache, nullptr, s, BH, bk, block);
    else e = run_tc<4, 32, 4>(ctx, plan, set, q, w, cache, nullptr, s, BH, bk, block);
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace dsa
