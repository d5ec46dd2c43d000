// plan_device.cu -- the device-side planner of capturable plans.
//
// The pages' follow-up gives selection and attention fixed-shape buffers so
// a decode step can be captured (mstar.engine.resources.dsa.manager, module
// overview); graph mode pads a layout to its bucket's ceiling with
// zero-length entries and sizes its index buffers for the worst case
// (mstar.engine.resources.attn.ragged.block_causal: RaggedBlockCausalWrapper,
// max_blocks, max_prefix_tokens).  plan_update_kernel recomputes, from spans
// in device memory, what dsa_plan computes on the host: each row's position
// and page list, the score offsets, the indexer groups (one row each), items
// and per-CTA item ranges, and the attention units and merges.  Rows past the
// step get position -1 and attention units / merges past its counts row -1,
// so their work exits at once; the counts themselves stay on the device.
//
// One CTA of 1024 threads.  The spans live in shared memory; each thread
// takes a contiguous run of spans or rows (at most kMaxRowsPerThread), and
// block-wide exclusive scans give the offsets, so the planner is a handful of
// passes with no chain of global-memory round trips.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMaxRowsPerThread = kPlanMaxRows / kPlanThreads;
static_assert(kPlanMaxRows % kPlanThreads == 0, "rows per thread");

struct PlanUpdateParams {
  const int32_t *num_spans;
  const dsa_device_span_t *spans;
  int64_t num_page_ids;
  int64_t max_scores;
  int32_t max_rows, max_spans, units_cap, combine_cap, idx_cap;
  int32_t P, align, topk, num_sms, box_rows;
  int32_t *row_pos, *row_page_off, *row_npages, *row_page_start;
  int64_t *row_score_off;
  IdxGroup *groups;
  IdxItem *items;
  int32_t *cta_begin;
  AttUnit *units;
  AttCombine *combine;
  AttCluster *clusters;           // [clusters_cap]
  int32_t clusters_cap;
  int32_t *counts;
  int *err;
};

// Exclusive scans of N values per thread over the block, in one pass (three
// barriers for all N): v[i] becomes the sum of the lower threads' v[i] and
// total[i] the sum over all threads.  sh holds 32 x N values.
template <int N>
__device__ void block_exclusive_scan(int64_t (&v)[N], int64_t (&total)[N], int64_t *sh) {
  static_assert(kPlanThreads == 32 * 32, "one scan level over 32 warps");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x[N];
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x[i], o);
      if (lane >= o) x[i] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < N; ++i) sh[i * 32 + warp] = x[i];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      int64_t t = sh[i * 32 + lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      sh[i * 32 + lane] = t;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    v[i] = (warp > 0 ? sh[i * 32 + warp - 1] : 0) + x[i] - v[i];
    total[i] = sh[i * 32 + 31];
  }
  __syncthreads();   // sh is free for the next scan
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__global__ void __launch_bounds__(kPlanThreads) plan_update_kernel(const PlanUpdateParams p) {
  extern __shared__ uint8_t smem_raw[];
  // shared memory: per span [max_spans + 1] first rows and [max_spans]
  // ctx_start, page_off, num_pages, page_start
  int32_t *s_q0 = reinterpret_cast<int32_t *>(smem_raw);
  int32_t *s_ctx = s_q0 + p.max_spans + 1;
  int32_t *s_poff = s_ctx + p.max_spans;
  int32_t *s_np = s_poff + p.max_spans;
  int32_t *s_ps = s_np + p.max_spans;
  __shared__ int64_t sh[32 * 3];
  const int tid = threadIdx.x;

  // ---- spans into shared memory, validity, rows and scores (the first span
  // of each thread is loaded together with the count: the span array holds
  // max_spans entries whatever the count says)
  dsa_device_span_t s0{};
  if (tid < p.max_spans) s0 = p.spans[tid];
  int n = *p.num_spans;
  bool ok = n >= 0 && n <= p.max_spans;
  if (!ok) n = 0;
  for (int i = tid; i < n; i += kPlanThreads) {
    const dsa_device_span_t s = i == tid ? s0 : p.spans[i];
    const int64_t end = static_cast<int64_t>(s.ctx_start) + s.q_len;   // tokens 0 .. end-1
    const bool v = s.q_len >= 1 && s.ctx_start >= 0 && s.page_start >= 0 && s.page_start % p.align == 0 &&
                   s.num_pages >= 0 && s.page_off >= 0 && s.reserved == 0 &&
                   static_cast<int64_t>(s.page_off) + s.num_pages <= p.num_page_ids && end <= INT32_MAX &&
                   static_cast<int64_t>(s.num_pages) * p.P >= s.page_start + end;
    ok = ok && v;
    s_q0[i] = v ? s.q_len : 0;
    s_ctx[i] = s.ctx_start;
    s_poff[i] = s.page_off;
    s_np[i] = s.num_pages;
    s_ps[i] = s.page_start;
  }
  ok = __syncthreads_and(ok) != 0;
  const int spt = (p.max_spans + kPlanThreads - 1) / kPlanThreads;
  const int sa = min(tid * spt, n), sb = min(sa + spt, n);
  int64_t my_rows = 0, my_scores = 0;
  for (int i = sa; i < sb; ++i) {
    const int64_t q = s_q0[i], c = s_ctx[i];
    my_rows += q;
    my_scores += (2 * c + 1 + q) * q / 2;   // rows at positions c .. c+q-1 score pos+1 keys each
  }
  int64_t sv[2] = {my_rows, my_scores}, st[2];
  block_exclusive_scan<2>(sv, st, sh);
  const int64_t row0 = sv[0];
  int64_t T = st[0];
  const int64_t total_scores = st[1];
  if (T > p.max_rows || total_scores > p.max_scores) ok = false;   // uniform: totals are block-wide
  if (!ok) {
    n = 0;
    T = 0;
    if (tid == 0) atomicOr(p.err, kErrSpans);
  } else {
    int64_t r = row0;
    for (int i = sa; i < sb; ++i) {
      const int32_t q = s_q0[i];
      s_q0[i] = static_cast<int32_t>(r);
      r += q;
    }
    if (tid == 0) s_q0[n] = static_cast<int32_t>(T);
  }
  __syncthreads();

  // ---- rows: position and page list (kept in registers for the later passes)
  const int rpt = (p.max_rows + kPlanThreads - 1) / kPlanThreads;
  const int ra = min(tid * rpt, p.max_rows), rn = min(rpt, p.max_rows - ra);
  int32_t pos[kMaxRowsPerThread];
  int64_t my_sc = 0, my_tiles = 0;
#pragma unroll
  for (int k = 0; k < kMaxRowsPerThread; ++k) {
    pos[k] = -1;
    if (k >= rn) continue;
    const int r = ra + k;
    int32_t poff = 0, np = 0, ps = 0;
    if (r < T) {
      int lo = 0, hi = n - 1;   // the last span whose first row is <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_q0[mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      pos[k] = s_ctx[lo] + (r - s_q0[lo]);
      poff = s_poff[lo];
      np = s_np[lo];
      ps = s_ps[lo];
      my_sc += static_cast<int64_t>(pos[k]) + 1;
      my_tiles += index_group_tiles(static_cast<int64_t>(pos[k]) + 1, index_tile_lead(ps, p.box_rows));
    }
    p.row_pos[r] = pos[k];
    p.row_page_off[r] = poff;
    p.row_npages[r] = np;
    p.row_page_start[r] = ps;
  }
  // (score offsets, indexer tiles and attention tiles in one scan)
  int64_t my_at = 0;
#pragma unroll
  for (int k = 0; k < kMaxRowsPerThread; ++k)
    if (pos[k] >= 0) my_at += att_row_tiles(pos[k], p.topk);
  int64_t rv[3] = {my_sc, my_tiles, my_at}, rt[3];
  block_exclusive_scan<3>(rv, rt, sh);
  int64_t sc = rv[0], tile = rv[1];
  const int64_t sc_total = rt[0], tiles_total = rt[1];
  const int64_t at_off0 = rv[2], at_total = rt[2];

  // ---- indexer items and attention units per row.  The attention schedule
  // cuts the rows' key tiles, in row order, into contiguous ranges, one per
  // persistent cluster (att_cluster_split, the host planner's function); a
  // row a cut crosses becomes one unit per piece, with partial slots and a
  // merge.
  // the indexer's tiles are split over n_cta CTAs exactly (index_cta_start,
  // the host planner's function); a row a CTA boundary crosses is one item
  // per piece
  const int32_t n_cta = static_cast<int32_t>(min64(tiles_total, p.idx_cap));
  auto idx_pieces = [&](int64_t off, int64_t n) -> int {
    return static_cast<int>(index_cta_of_tile(off + n - 1, tiles_total, n_cta) - index_cta_of_tile(off, tiles_total, n_cta) + 1);
  };
  int32_t ncl = 0;
  int64_t per = 1;
  att_cluster_split(at_total, p.num_sms, &ncl, &per);
  // counts packed two per scan: (items << 32 | units), (slots << 32 | merges)
  int64_t my_iu = 0, my_sm = 0;
  {
    int64_t off = at_off0, ioff = tile;
#pragma unroll
    for (int k = 0; k < kMaxRowsPerThread; ++k) {
      if (pos[k] < 0) continue;
      const int32_t tiles = index_group_tiles(static_cast<int64_t>(pos[k]) + 1,
                                              index_tile_lead(p.row_page_start[ra + k], p.box_rows));
      const int64_t n = att_row_tiles(pos[k], p.topk);
      const int u = static_cast<int>((off + n - 1) / per - off / per + 1);
      my_iu += (static_cast<int64_t>(idx_pieces(ioff, tiles)) << 32) + u;
      my_sm += u > 1 ? ((static_cast<int64_t>(u) << 32) + 1) : 0;
      off += n;
      ioff += tiles;
    }
  }
  int64_t uv[2] = {my_iu, my_sm}, ut[2];
  block_exclusive_scan<2>(uv, ut, sh);
  int64_t iu = uv[0], smc = uv[1];
  const int64_t iu_total = ut[0], sm_total = ut[1];
  const int32_t n_items = static_cast<int32_t>(iu_total >> 32), n_units = static_cast<int32_t>(iu_total & 0xffffffff);
  const int32_t n_slots = static_cast<int32_t>(sm_total >> 32), n_merge = static_cast<int32_t>(sm_total & 0xffffffff);
  // the plan's capacities bound these counts for every update the span checks
  // admit (see dsa_plan_capturable), so the writes below stay in bounds
  int64_t at_off = at_off0;
#pragma unroll
  for (int k = 0; k < kMaxRowsPerThread; ++k) {
    if (k >= rn) continue;
    const int r = ra + k;
    p.row_score_off[r] = sc;
    if (pos[k] < 0) continue;
    sc += static_cast<int64_t>(pos[k]) + 1;
    const int32_t lead = index_tile_lead(p.row_page_start[r], p.box_rows);
    const int32_t tiles = index_group_tiles(static_cast<int64_t>(pos[k]) + 1, lead);
    // the row is indexer group r (one row per group)
    IdxGroup g;
    g.row0 = r;
    g.nrows = 1;
    g.pos0 = pos[k];
    g.page_off = p.row_page_off[r];
    g.npages = p.row_npages[r];
    g.page_start = p.row_page_start[r];
    g.ntiles = tiles;
    g.lead = lead;
    p.groups[r] = g;
    int32_t item = static_cast<int32_t>(iu >> 32);
    {
      const int64_t b0 = index_cta_of_tile(tile, tiles_total, n_cta), b1 = index_cta_of_tile(tile + tiles - 1, tiles_total, n_cta);
      for (int64_t b = b0; b <= b1; ++b, ++item) {
        const int64_t cs = index_cta_start(b, tiles_total, n_cta);
        const int64_t a = tile > cs ? tile : cs;
        const int64_t ce = index_cta_start(b + 1, tiles_total, n_cta);
        const int64_t e = tile + tiles < ce ? tile + tiles : ce;
        if (a == cs) p.cta_begin[b] = item;   // the CTA's first item
        p.items[item] = IdxItem{r, static_cast<int32_t>(a - tile), static_cast<int32_t>(e - tile), 0};
      }
    }
    const int32_t n_idx_pieces = idx_pieces(tile, tiles);
    tile += tiles;
    // attention: one unit per piece of the row's tiles between cuts
    const int64_t nsel = min64(p.topk, static_cast<int64_t>(pos[k]) + 1);
    const int64_t n = att_row_tiles(pos[k], p.topk);
    const int64_t c0 = at_off / per, c1 = (at_off + n - 1) / per;
    const int u = static_cast<int>(c1 - c0 + 1);
    int32_t unit = static_cast<int32_t>(iu & 0xffffffff);
    const int32_t slot = static_cast<int32_t>(smc >> 32);
    if (u > 1) p.combine[static_cast<int32_t>(smc & 0xffffffff)] = AttCombine{r, slot, u, 0};
    for (int64_t cl = c0; cl <= c1; ++cl, ++unit) {
      const int64_t a = at_off > cl * per ? at_off : cl * per;
      const int64_t b = at_off + n < (cl + 1) * per ? at_off + n : (cl + 1) * per;
      if (a == cl * per) p.clusters[cl].u0 = unit;   // the cluster's first unit
      p.units[unit] = AttUnit{r, static_cast<int32_t>((a - at_off) * kAttTile),
                              static_cast<int32_t>(min64(nsel, (b - at_off) * kAttTile)),
                              u > 1 ? slot + static_cast<int32_t>(cl - c0) : -1};
    }
    if (u > 1) smc += (static_cast<int64_t>(u) << 32) + 1;
    iu += (static_cast<int64_t>(n_idx_pieces) << 32) + u;
    at_off += n;
  }
  // padding: units and merges past the step's counts exit at once
  for (int i = n_units + tid; i < p.units_cap; i += kPlanThreads) p.units[i] = AttUnit{-1, 0, 0, -1};
  for (int i = n_merge + tid; i < p.combine_cap; i += kPlanThreads) p.combine[i] = AttCombine{-1, 0, 0, 0};
  __syncthreads();   // every cluster's first unit is written
  // each cluster's unit range and tiles (thread = cluster; clusters_cap <=
  // kPlanThreads); clusters past the schedule are idle
  {
    AttCluster e{0, 0, 0, 0};
    if (tid < ncl) {
      e.u0 = p.clusters[tid].u0;
      e.u1 = tid + 1 < ncl ? p.clusters[tid + 1].u0 : n_units;
      e.tiles = static_cast<int32_t>(min64(per, at_total - static_cast<int64_t>(tid) * per));
    }
    __syncthreads();   // every u0 is read before any entry is rewritten
    if (tid < p.clusters_cap) p.clusters[tid] = e;
  }

  // ---- CTAs past the split (n_cta <= b <= idx_cap) start at the end
  for (int b = n_cta + tid; b <= p.idx_cap; b += kPlanThreads) p.cta_begin[b] = n_items;
  if (tid == 0) {
    p.counts[0] = static_cast<int32_t>(T);
    p.counts[1] = n_items;
    p.counts[2] = n_units;
    p.counts[3] = n_merge;
    p.counts[4] = n_slots;
    p.counts[5] = ok ? 1 : 0;
    p.counts[6] = ncl;
    p.counts[7] = static_cast<int32_t>(min64(sc_total, INT32_MAX));
  }
}

}  // namespace

static size_t plan_update_smem(int32_t /*max_rows*/, int32_t max_spans) {
  return static_cast<size_t>(max_spans + 1) * sizeof(int32_t) + static_cast<size_t>(max_spans) * 4 * sizeof(int32_t);
}

cudaError_t launch_plan_update(const dsa_ctx *ctx, dsa_plan_t *plan, const int32_t *num_spans,
                               const dsa_device_span_t *spans, int64_t num_page_ids, cudaStream_t s) {
  PlanUpdateParams p;
  p.num_spans = num_spans;
  p.spans = spans;
  p.num_page_ids = num_page_ids;
  p.max_scores = plan->num_scores;
  p.max_rows = plan->T;
  p.max_spans = plan->max_spans;
  p.units_cap = plan->n_units;
  p.combine_cap = plan->combine_cap;
  p.idx_cap = plan->idx[0].n_ctas;
  p.P = ctx->cfg.page_size;
  p.align = plan->page_start_align;
  p.box_rows = plan->box_rows;
  p.topk = ctx->cfg.topk;
  p.num_sms = ctx->num_sms;
  p.row_pos = plan->row_pos;
  p.row_page_off = plan->row_page_off;
  p.row_npages = plan->row_npages;
  p.row_page_start = plan->row_page_start;
  p.row_score_off = plan->row_score_off;
  p.groups = plan->idx[0].groups;
  p.items = plan->idx[0].items;
  p.cta_begin = plan->idx[0].cta_begin;
  p.units = plan->units;
  p.combine = plan->combine;
  p.clusters = plan->clusters;
  p.clusters_cap = plan->n_clusters;
  p.counts = plan->counts;
  p.err = ctx->err;
  plan_update_kernel<<<1, kPlanThreads, plan_update_smem(plan->T, plan->max_spans), s>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_plan_update(int32_t max_rows, int32_t max_spans) {
  static std::mutex mu;
  static size_t limit = 48 * 1024;
  const size_t smem = plan_update_smem(max_rows, max_spans);
  std::lock_guard<std::mutex> lock(mu);
  if (smem <= limit) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(plan_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) limit = smem;
  return e;
}

}  // namespace dsa
