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
// and per-CTA item ranges, and the attention units and merges.  Padding is
// marked so that its work exits at once: rows past the step get position -1,
// items and units past the step's counts group / row -1.
//
// One CTA of 1024 threads; each thread takes a contiguous run of spans or
// rows, and block-wide exclusive scans give the offsets.
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kPlanThreads = 1024;

struct PlanUpdateParams {
  const int32_t *num_spans;
  const dsa_device_span_t *spans;
  int64_t num_page_ids;
  int64_t max_scores;
  int32_t max_rows, max_spans, items_cap, units_cap, combine_cap, idx_cap;
  int32_t P, align, topk, num_sms;
  int32_t *span_q0;
  int32_t *row_pos, *row_page_off, *row_npages, *row_page_start;
  int64_t *row_score_off;
  IdxGroup *groups;
  IdxItem *items;
  int64_t *item_tile0;
  int32_t *cta_begin;
  AttUnit *units;
  AttCombine *combine;
  int32_t *counts;
  int *err;
};

// Exclusive scan of one value per thread over the block.  Returns the sum of
// the values of the lower threads; *total = the sum over all threads.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t *total, int64_t *sh) {
  static_assert(kPlanThreads == 32 * 32, "one scan level over 32 warps");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t t = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    sh[lane] = t;
  }
  __syncthreads();
  const int64_t before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
  *total = sh[31];
  __syncthreads();   // sh is free for the next scan
  return before;
}

__device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__global__ void __launch_bounds__(kPlanThreads) plan_update_kernel(const PlanUpdateParams p) {
  __shared__ int64_t sh[32];
  const int tid = threadIdx.x;

  // ---- spans: validity, rows and scores
  int n = *p.num_spans;
  bool ok = n >= 0 && n <= p.max_spans;
  if (!ok) n = 0;
  const int spt = (p.max_spans + kPlanThreads - 1) / kPlanThreads;
  const int sa = min(tid * spt, n), sb = min(sa + spt, n);
  int64_t my_rows = 0, my_scores = 0;
  for (int i = sa; i < sb; ++i) {
    const dsa_device_span_t s = p.spans[i];
    const int64_t end = static_cast<int64_t>(s.ctx_start) + s.q_len;   // tokens 0 .. end-1
    const bool v = s.q_len >= 1 && s.ctx_start >= 0 && s.page_start >= 0 && s.page_start % p.align == 0 &&
                   s.num_pages >= 0 && s.page_off >= 0 && s.reserved == 0 &&
                   static_cast<int64_t>(s.page_off) + s.num_pages <= p.num_page_ids && end <= INT32_MAX &&
                   static_cast<int64_t>(s.num_pages) * p.P >= s.page_start + end;
    ok = ok && v;
    if (v) {
      my_rows += s.q_len;
      // rows at positions ctx_start .. end-1 score pos+1 keys each
      my_scores += (static_cast<int64_t>(s.ctx_start) + 1 + end) * s.q_len / 2;
    }
  }
  ok = __syncthreads_and(ok) != 0;
  int64_t T = 0, total_scores = 0;
  const int64_t row0 = block_exclusive_scan(my_rows, &T, sh);
  const int64_t score0 = block_exclusive_scan(my_scores, &total_scores, sh);
  (void)score0;
  if (T > p.max_rows || total_scores > p.max_scores) ok = false;   // uniform: totals are block-wide
  if (!ok) {
    n = 0;
    T = 0;
    total_scores = 0;
    if (tid == 0) atomicOr(p.err, kErrSpans);
  } else {
    int64_t r = row0;
    for (int i = sa; i < sb; ++i) {
      p.span_q0[i] = static_cast<int32_t>(r);
      r += p.spans[i].q_len;
    }
    if (tid == 0) p.span_q0[n] = static_cast<int32_t>(T);
  }
  __syncthreads();   // span_q0 is visible to the block

  // ---- rows: position and page list; score and indexer-tile offsets
  const int rpt = (p.max_rows + kPlanThreads - 1) / kPlanThreads;
  const int ra = min(tid * rpt, p.max_rows), rb = min(ra + rpt, p.max_rows);
  int64_t my_sc = 0, my_tiles = 0;
  for (int r = ra; r < rb; ++r) {
    int32_t pos = -1, poff = 0, np = 0, ps = 0;
    if (r < T) {
      int lo = 0, hi = n - 1;   // the last span whose first row is <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.span_q0[mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      const dsa_device_span_t s = p.spans[lo];
      pos = s.ctx_start + (r - p.span_q0[lo]);
      poff = s.page_off;
      np = s.num_pages;
      ps = s.page_start;
      my_sc += static_cast<int64_t>(pos) + 1;
      my_tiles += ceil_div(static_cast<int64_t>(pos) + 1, kIndexTile);
    }
    p.row_pos[r] = pos;
    p.row_page_off[r] = poff;
    p.row_npages[r] = np;
    p.row_page_start[r] = ps;
  }
  int64_t sc_total = 0, tiles_total = 0;
  int64_t sc = block_exclusive_scan(my_sc, &sc_total, sh);
  int64_t tile = block_exclusive_scan(my_tiles, &tiles_total, sh);

  // ---- indexer items and attention units per row
  const int64_t tpi = index_tiles_per_item(tiles_total, p.idx_cap);
  const int splits = attention_splits(T, p.topk, p.num_sms);
  // counts packed two per scan: (items << 32 | units), (slots << 32 | merges)
  int64_t my_iu = 0, my_sm = 0;
  for (int r = ra; r < rb; ++r) {
    const int32_t pos = p.row_pos[r];
    if (pos < 0) continue;
    const int64_t tiles = ceil_div(static_cast<int64_t>(pos) + 1, kIndexTile);
    const int u = attention_row_units(pos, p.topk, splits);
    my_iu += (ceil_div(tiles, tpi) << 32) + u;
    my_sm += u > 1 ? ((static_cast<int64_t>(u) << 32) + 1) : 0;
  }
  int64_t iu_total = 0, sm_total = 0;
  int64_t iu = block_exclusive_scan(my_iu, &iu_total, sh);
  int64_t smc = block_exclusive_scan(my_sm, &sm_total, sh);
  int32_t n_items = static_cast<int32_t>(iu_total >> 32), n_units = static_cast<int32_t>(iu_total & 0xffffffff);
  int32_t n_slots = static_cast<int32_t>(sm_total >> 32), n_merge = static_cast<int32_t>(sm_total & 0xffffffff);
  // the capacities bound these counts for every update the span checks admit;
  // should one not fit, the plan is emptied rather than overrun
  if (n_items > p.items_cap || n_units > p.units_cap || n_merge > p.combine_cap || n_slots > p.units_cap) {
    if (tid == 0) atomicOr(p.err, kErrSpans);
    ok = false;
    T = 0;
    n_items = n_units = n_merge = n_slots = 0;
    tiles_total = 0;
    for (int r = ra; r < rb; ++r) p.row_pos[r] = -1;
  }
  for (int r = ra; r < rb; ++r) {
    const int32_t pos = p.row_pos[r];
    p.row_score_off[r] = sc;
    if (pos < 0) continue;
    sc += static_cast<int64_t>(pos) + 1;
    const int64_t tiles = ceil_div(static_cast<int64_t>(pos) + 1, kIndexTile);
    // the row is indexer group r (one row per group)
    IdxGroup g;
    g.row0 = r;
    g.nrows = 1;
    g.pos0 = pos;
    g.page_off = p.row_page_off[r];
    g.npages = p.row_npages[r];
    g.page_start = p.row_page_start[r];
    g.ntiles = static_cast<int32_t>(tiles);
    g.pad = 0;
    p.groups[r] = g;
    int32_t item = static_cast<int32_t>(iu >> 32);
    for (int64_t t0 = 0; t0 < tiles; t0 += tpi, ++item) {
      p.items[item] = IdxItem{r, static_cast<int32_t>(t0), static_cast<int32_t>(min64(tiles, t0 + tpi)), 0};
      p.item_tile0[item] = tile + t0;
    }
    tile += tiles;
    // attention: whole row, or `u` key ranges with partial slots and a merge
    const int64_t nsel = min64(p.topk, static_cast<int64_t>(pos) + 1);
    const int64_t atiles = ceil_div(nsel, kAttTile);
    const int u = attention_row_units(pos, p.topk, splits);
    const int32_t unit = static_cast<int32_t>(iu & 0xffffffff);
    if (u == 1) {
      p.units[unit] = AttUnit{r, 0, static_cast<int32_t>(nsel), -1};
    } else {
      const int32_t slot = static_cast<int32_t>(smc >> 32);
      p.combine[static_cast<int32_t>(smc & 0xffffffff)] = AttCombine{r, slot, u, 0};
      for (int k = 0; k < u; ++k) {
        const int64_t t0 = atiles * k / u, t1 = atiles * (k + 1) / u;
        p.units[unit + k] = AttUnit{r, static_cast<int32_t>(t0 * kAttTile),
                                    static_cast<int32_t>(min64(nsel, t1 * kAttTile)), slot + k};
      }
      smc += (static_cast<int64_t>(u) << 32) + 1;
    }
    iu += (ceil_div(tiles, tpi) << 32) + u;
  }
  // padding: work past the step's counts exits at once
  for (int i = n_items + tid; i < p.items_cap; i += kPlanThreads) p.items[i] = IdxItem{-1, 0, 0, 0};
  for (int i = n_units + tid; i < p.units_cap; i += kPlanThreads) p.units[i] = AttUnit{-1, 0, 0, -1};
  for (int i = n_merge + tid; i < p.combine_cap; i += kPlanThreads) p.combine[i] = AttCombine{-1, 0, 0, 0};
  if (tid == 0) p.item_tile0[n_items] = tiles_total;
  __syncthreads();   // item_tile0 is visible to the block

  // ---- per-CTA item ranges of the persistent indexer: CTA b starts at the
  // first item that begins at or after tile tiles_total * b / idx_cap
  for (int b = tid; b <= p.idx_cap; b += kPlanThreads) {
    int32_t k = n_items;
    if (b < p.idx_cap) {
      const int64_t target = tiles_total * b / p.idx_cap;
      int lo = 0, hi = n_items;   // first k in [0, n_items] with item_tile0[k] >= target
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (p.item_tile0[mid] < target) lo = mid + 1;
        else hi = mid;
      }
      k = lo;
    }
    p.cta_begin[b] = k;
  }
  if (tid == 0) {
    p.counts[0] = static_cast<int32_t>(T);
    p.counts[1] = n_items;
    p.counts[2] = n_units;
    p.counts[3] = n_merge;
    p.counts[4] = n_slots;
    p.counts[5] = ok ? 1 : 0;
    p.counts[6] = splits;
    p.counts[7] = static_cast<int32_t>(min64(sc_total, INT32_MAX));
  }
}

}  // namespace

cudaError_t launch_plan_update(const dsa_ctx *ctx, dsa_plan_t *plan, const int32_t *num_spans,
                               const dsa_device_span_t *spans, int64_t num_page_ids, cudaStream_t s) {
  PlanUpdateParams p;
  p.num_spans = num_spans;
  p.spans = spans;
  p.num_page_ids = num_page_ids;
  p.max_scores = plan->num_scores;
  p.max_rows = plan->T;
  p.max_spans = plan->max_spans;
  p.items_cap = plan->items_cap;
  p.units_cap = plan->n_units;
  p.combine_cap = plan->combine_cap;
  p.idx_cap = plan->idx[0].n_ctas;
  p.P = ctx->cfg.page_size;
  p.align = plan->page_start_align;
  p.topk = ctx->cfg.topk;
  p.num_sms = ctx->num_sms;
  p.span_q0 = plan->span_q0;
  p.row_pos = plan->row_pos;
  p.row_page_off = plan->row_page_off;
  p.row_npages = plan->row_npages;
  p.row_page_start = plan->row_page_start;
  p.row_score_off = plan->row_score_off;
  p.groups = plan->idx[0].groups;
  p.items = plan->idx[0].items;
  p.item_tile0 = plan->item_tile0;
  p.cta_begin = plan->idx[0].cta_begin;
  p.units = plan->units;
  p.combine = plan->combine;
  p.counts = plan->counts;
  p.err = ctx->err;
  plan_update_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
