// api.cu -- the C ABI (include/dsa.h): contexts, plans, validation, scratch
// management and the calls that launch the kernels.
//
// Planning follows mstar DSAManager.plan / DSAPlan / DSASpan
// ("mstar.engine.resources.dsa.manager"): each span contributes q_len rows
// starting at row q_start, the first at position ctx_start; a row's page list
// is its span's, and its token 0 sits page_start slots into it.  The plan
// flattens all of that into device arrays once, so no kernel of the step
// needs the host again.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "dsa_internal.h"

using namespace dsa;

namespace {

bool valid_config(const dsa_config_t &c) {
  if (c.index_heads <= 0 || c.index_dim <= 0 || c.topk <= 0 || c.heads <= 0 || c.kv_lora_rank <= 0 ||
      c.rope_dim < 0 || c.page_size <= 0)
    return false;
  if (c.latent_fmt != DSA_LATENT_BF16 && c.latent_fmt != DSA_LATENT_FP8_656) return false;
  if (c.index_fmt != DSA_INDEX_BF16 && c.index_fmt != DSA_INDEX_FP8_132) return false;
  return true;
}

dsa_status supported_config(const dsa_config_t &c) {
  // 16-byte vector copies of key rows and of latent rows
  if ((c.index_dim * 2) % 16 != 0) return DSA_ERR_UNSUPPORTED;
  if (c.index_fmt == DSA_INDEX_FP8_132 && c.index_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (c.latent_fmt == DSA_LATENT_FP8_656 && (c.kv_lora_rank % 128 != 0)) return DSA_ERR_UNSUPPORTED;
  if (((c.kv_lora_rank + c.rope_dim) * 2) % 16 != 0) return DSA_ERR_UNSUPPORTED;
  if (c.kv_lora_rank % 8 != 0 || c.rope_dim % 8 != 0) return DSA_ERR_UNSUPPORTED;
  if (c.kv_lora_rank > 1024 || c.index_heads > 256 || c.heads > 1024) return DSA_ERR_UNSUPPORTED;
  // the attention schedule cuts a row into at most kAttMaxPieces pieces
  if (c.topk > 16384) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

template <typename T>
size_t align_up(size_t x) {
  return (x + alignof(T) - 1) / alignof(T) * alignof(T);
}

// Bump allocator over the staging vector: records offsets, fills pointers later.
struct Layout {
  size_t bytes = 0;
  template <typename T>
  size_t take(size_t n) {
    bytes = (bytes + 255) / 256 * 256;
    size_t off = bytes;
    bytes += n * sizeof(T);
    return off;
  }
};

bool is_host_only(const dsa_ctx *ctx) { return ctx == nullptr || ctx->device < 0; }

// DSA_OK, or DSA_ERR_CUDA with the CUDA error recorded in the context.
dsa_status cuda_status(dsa_ctx *ctx, cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  snprintf(ctx->last_cuda_error, sizeof(ctx->last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

dsa_status ensure_scratch(dsa_ctx *ctx, size_t scores, size_t slots) {
  if (scores > ctx->scores_cap) {
    size_t cap = std::max(scores, ctx->scores_cap * 3 / 2);
    if (ctx->scores) cudaFree(ctx->scores);
    ctx->scores = nullptr;
    ctx->scores_cap = 0;
    if (cudaMalloc(&ctx->scores, cap * sizeof(float)) != cudaSuccess) return DSA_ERR_OOM;
    ctx->scores_cap = cap;
  }
  if (slots > ctx->part_cap) {
    size_t cap = std::max(slots, ctx->part_cap * 3 / 2);
    if (ctx->opart) cudaFree(ctx->opart);
    if (ctx->mlpart) cudaFree(ctx->mlpart);
    ctx->opart = ctx->mlpart = nullptr;
    ctx->part_cap = 0;
    const size_t hl = static_cast<size_t>(ctx->cfg.heads) * ctx->cfg.kv_lora_rank;
    if (cudaMalloc(&ctx->opart, cap * hl * sizeof(float)) != cudaSuccess) return DSA_ERR_OOM;
    if (cudaMalloc(&ctx->mlpart, cap * ctx->cfg.heads * 2 * sizeof(float)) != cudaSuccess) return DSA_ERR_OOM;
    ctx->part_cap = cap;
  }
  return DSA_OK;
}

}  // namespace

// ----------------------------------------------------------------------------
// tensor maps
// ----------------------------------------------------------------------------
namespace dsa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

bool encode_tiled_2d(CUtensorMap *tm, CUtensorMapDataType dtype, void *base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tiled_3d(CUtensorMap *tm, CUtensorMapDataType dtype, void *base, const uint64_t dims[3],
                     const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, dtype, 3, base, d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa

// ----------------------------------------------------------------------------
// C ABI
// ----------------------------------------------------------------------------
extern "C" {

const char *dsa_status_str(dsa_status s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_SHORT_HISTORY: return "span pages do not reach the positions the step needs";
    case DSA_ERR_OOM: return "out of memory";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_BOUNDS: return "device bounds check failed (selection or page id out of range)";
    case DSA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case DSA_ERR_SCRATCH_LIMIT: return "plan needs more scores than the static score array holds (DSA_STATIC_SCORES_MAX)";
    case DSA_ERR_BAD_SPANS: return "a capturable plan's update found invalid spans or exceeded its capacities; the plan was emptied";
    default: return "unknown status";
  }
}

dsa_status dsa_create(const dsa_config_t *cfg, int device, dsa_ctx_t **out) {
  if (!cfg || !out) return DSA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_config(*cfg)) return DSA_ERR_INVALID_ARG;
  dsa_status sup = supported_config(*cfg);
  if (sup != DSA_OK) return sup;
  dsa_ctx *ctx = new (std::nothrow) dsa_ctx();
  if (!ctx) return DSA_ERR_OOM;
  ctx->cfg = *cfg;
  ctx->device = device;
  if (device >= 0) {
    if (cudaSetDevice(device) != cudaSuccess) { delete ctx; return DSA_ERR_CUDA; }
    if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      delete ctx;
      return DSA_ERR_CUDA;
    }
    if (cudaMalloc(&ctx->err, sizeof(int)) != cudaSuccess) { delete ctx; return DSA_ERR_OOM; }
    if (cudaMemset(ctx->err, 0, sizeof(int)) != cudaSuccess) { cudaFree(ctx->err); delete ctx; return DSA_ERR_CUDA; }
    // the fixed score array of dsa_index_topk_static: looking up its address
    // loads the module that holds it, so the array is on the device from here
    // on and the static entry point never makes the driver allocate
    if (static_scores_address(device, &ctx->static_scores) != cudaSuccess) {
      cudaFree(ctx->err);
      delete ctx;
      return DSA_ERR_CUDA;
    }
  } else {
    ctx->num_sms = 152;
  }
  *out = ctx;
  return DSA_OK;
}

void dsa_destroy(dsa_ctx_t *ctx) {
  if (!ctx) return;
  if (ctx->device >= 0) {
    cudaSetDevice(ctx->device);
    cudaFree(ctx->err);
    cudaFree(ctx->scores);
    cudaFree(ctx->opart);
    cudaFree(ctx->mlpart);
    cudaFree(ctx->block_keys);
  }
  delete ctx;
}

dsa_status dsa_plan(dsa_ctx_t *ctx, const dsa_span_t *spans, int32_t num_spans, int32_t cache_pages,
                    dsa_stream_t stream, dsa_plan_t **out) {
  if (!ctx || !out || num_spans < 0 || (num_spans > 0 && !spans) || cache_pages < 0) return DSA_ERR_INVALID_ARG;
  *out = nullptr;
  const dsa_config_t &c = ctx->cfg;
  const int64_t P = c.page_size;

  // ---- validate spans (they must tile rows [0, T) in order)
  int64_t T = 0, total_pages = 0, num_scores = 0;
  int32_t max_pos = 0;
  for (int32_t i = 0; i < num_spans; ++i) {
    const dsa_span_t &s = spans[i];
    if (s.q_start != T || s.q_len <= 0 || s.ctx_start < 0 || s.page_start < 0 || s.num_pages < 0)
      return DSA_ERR_INVALID_ARG;
    if (s.num_pages > 0 && !s.pages) return DSA_ERR_INVALID_ARG;
    const int64_t end = static_cast<int64_t>(s.ctx_start) + s.q_len;     // tokens 0 .. end-1
    if (end > INT32_MAX) return DSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(s.num_pages) * P < s.page_start + end) return DSA_ERR_SHORT_HISTORY;
    for (int32_t k = 0; k < s.num_pages; ++k)
      if (s.pages[k] < 0 || s.pages[k] >= cache_pages) return DSA_ERR_INVALID_ARG;
    T += s.q_len;
    total_pages += s.num_pages;
    // rows at positions ctx_start .. end-1 each score pos+1 keys
    num_scores += (static_cast<int64_t>(s.ctx_start) + 1 + end) * s.q_len / 2;
    max_pos = std::max<int32_t>(max_pos, static_cast<int32_t>(end - 1));
    if (T > INT32_MAX / 2 || total_pages > INT32_MAX / 2) return DSA_ERR_INVALID_ARG;
  }

  dsa_plan_t *plan = new (std::nothrow) dsa_plan_t();
  if (!plan) return DSA_ERR_OOM;
  plan->ctx = ctx;
  plan->stream = reinterpret_cast<cudaStream_t>(stream);
  plan->T = static_cast<int32_t>(T);
  plan->n_spans = num_spans;
  plan->cache_pages = cache_pages;
  plan->num_scores = num_scores;
  plan->max_pos = max_pos;
  plan->box_rows = index_box_rows(c.page_size);

  // ---- indexer groups: single rows (decode spans) and runs of G rows (chunks)
  const int Gm = indexer_group_rows(c);
  std::vector<IdxGroup> groups[2];
  int32_t page_off = 0;
  for (int32_t i = 0; i < num_spans; ++i) {
    const dsa_span_t &s = spans[i];
    const int set = (s.q_len > 1 && Gm > 1) ? 1 : 0;
    const int G = set ? Gm : 1;
    for (int32_t r = 0; r < s.q_len; r += G) {
      IdxGroup g{};
      g.row0 = s.q_start + r;
      g.nrows = std::min<int32_t>(G, s.q_len - r);
      g.pos0 = s.ctx_start + r;
      g.page_off = page_off;
      g.npages = s.num_pages;
      g.page_start = s.page_start;
      g.lead = index_tile_lead(s.page_start, plan->box_rows);
      g.ntiles = index_group_tiles(static_cast<int64_t>(g.pos0) + g.nrows, g.lead);
      groups[set].push_back(g);
    }
    page_off += s.num_pages;
  }
  std::vector<IdxItem> items[2];
  std::vector<int32_t> cta_begin[2];
  int64_t n_index_items = 0;
  for (int set = 0; set < 2; ++set) {
    int64_t tiles = 0;
    for (auto &g : groups[set]) tiles += g.ntiles;
    if (tiles == 0) continue;
    const int G = set ? Gm : 1;
    // CTAs take exactly balanced tile ranges (floor or ceil of tiles / CTAs);
    // a group a range boundary crosses is one item per piece
    const int n_ctas = static_cast<int>(std::min<int64_t>(tiles, std::max(1, ctx->num_sms * indexer_ctas_per_sm(c, G))));
    cta_begin[set].assign(n_ctas + 1, 0);
    int64_t off = 0;
    for (int32_t gi = 0; gi < static_cast<int32_t>(groups[set].size()); ++gi) {
      const IdxGroup &g = groups[set][gi];
      if (g.ntiles <= 0) continue;
      const int64_t b0 = index_cta_of_tile(off, tiles, n_ctas), b1 = index_cta_of_tile(off + g.ntiles - 1, tiles, n_ctas);
      for (int64_t b = b0; b <= b1; ++b) {
        const int64_t a = std::max<int64_t>(off, index_cta_start(b, tiles, n_ctas));
        const int64_t e = std::min<int64_t>(off + g.ntiles, index_cta_start(b + 1, tiles, n_ctas));
        if (a == index_cta_start(b, tiles, n_ctas)) cta_begin[set][b] = static_cast<int32_t>(items[set].size());
        items[set].push_back(IdxItem{gi, static_cast<int32_t>(a - off), static_cast<int32_t>(e - off), 0});
      }
      off += g.ntiles;
    }
    const int n_items = static_cast<int>(items[set].size());
    cta_begin[set][n_ctas] = n_items;
    plan->idx[set].G = G;
    plan->idx[set].n_groups = static_cast<int>(groups[set].size());
    plan->idx[set].n_items = n_items;
    plan->idx[set].n_ctas = n_ctas;
    n_index_items += n_items;
  }
  plan->n_index_items = static_cast<int32_t>(n_index_items);

  // ---- attention: the rows' key tiles, in row order, cut into contiguous
  // ranges, one per persistent two-CTA cluster; a row a cut crosses becomes
  // one unit per piece, each with a partial slot, merged afterwards
  std::vector<AttUnit> units;
  std::vector<AttCombine> combines;
  std::vector<AttCluster> clusters;
  {
    const int64_t K = c.topk;
    int64_t S = 0;
    for (int32_t i = 0; i < num_spans; ++i)
      for (int32_t r = 0; r < spans[i].q_len; ++r) S += att_row_tiles(static_cast<int64_t>(spans[i].ctx_start) + r, K);
    int32_t ncl = 0;
    int64_t per = 1;
    att_cluster_split(S, ctx->num_sms, &ncl, &per);
    clusters.assign(ncl, AttCluster{0, 0, 0, 0});
    int32_t slot = 0;
    int32_t row = 0;
    int64_t off = 0;
    for (int32_t i = 0; i < num_spans; ++i) {
      const dsa_span_t &s = spans[i];
      for (int32_t r = 0; r < s.q_len; ++r, ++row) {
        const int64_t pos = s.ctx_start + r;
        const int64_t nsel = std::min<int64_t>(K, pos + 1);
        const int64_t n = att_row_tiles(pos, K);
        const int64_t c0 = off / per, c1 = (off + n - 1) / per;
        const int32_t pieces = static_cast<int32_t>(c1 - c0 + 1);
        if (pieces > 1) combines.push_back(AttCombine{row, slot, pieces, 0});
        for (int64_t cl = c0; cl <= c1; ++cl) {
          const int64_t a = std::max<int64_t>(off, cl * per), b = std::min<int64_t>(off + n, (cl + 1) * per);
          if (a == cl * per) clusters[cl].u0 = static_cast<int32_t>(units.size());   // the cluster starts here
          units.push_back(AttUnit{row, static_cast<int32_t>((a - off) * kAttTile),
                                  static_cast<int32_t>(std::min<int64_t>(nsel, (b - off) * kAttTile)),
                                  pieces > 1 ? slot++ : -1});
        }
        plan->splits_max = std::max(plan->splits_max, pieces);
        off += n;
      }
    }
    for (int32_t cl = 0; cl < ncl; ++cl) {
      clusters[cl].u1 = cl + 1 < ncl ? clusters[cl + 1].u0 : static_cast<int32_t>(units.size());
      clusters[cl].tiles = static_cast<int32_t>(std::min<int64_t>(per, S - cl * per));
    }
    plan->n_units = static_cast<int32_t>(units.size());
    plan->n_combine = static_cast<int32_t>(combines.size());
    plan->n_slots = slot;
    plan->n_clusters = ncl;
  }

  // needs_selection: some row sees more than topk keys (mstar DSAPlan)
  plan->needs_selection = (max_pos + 1 > c.topk) ? 1 : 0;

  // ---- device metadata in one buffer
  Layout lay;
  const size_t o_pos = lay.take<int32_t>(T), o_poff = lay.take<int32_t>(T), o_np = lay.take<int32_t>(T),
               o_ps = lay.take<int32_t>(T), o_soff = lay.take<int64_t>(T), o_pages = lay.take<int32_t>(total_pages);
  size_t o_g[2], o_i[2], o_c[2];
  for (int set = 0; set < 2; ++set) {
    o_g[set] = lay.take<IdxGroup>(groups[set].size());
    o_i[set] = lay.take<IdxItem>(items[set].size());
    o_c[set] = lay.take<int32_t>(cta_begin[set].size());
  }
  const size_t o_u = lay.take<AttUnit>(units.size()), o_cb = lay.take<AttCombine>(combines.size()),
               o_cl = lay.take<AttCluster>(clusters.size());
  const size_t bytes = std::max<size_t>(lay.bytes, 256);
  try {
    plan->host.assign(bytes, 0);
  } catch (...) {
    delete plan;
    return DSA_ERR_OOM;
  }
  char *h = plan->host.data();
  {
    auto *pos = reinterpret_cast<int32_t *>(h + o_pos);
    auto *poff = reinterpret_cast<int32_t *>(h + o_poff);
    auto *np = reinterpret_cast<int32_t *>(h + o_np);
    auto *ps = reinterpret_cast<int32_t *>(h + o_ps);
    auto *soff = reinterpret_cast<int64_t *>(h + o_soff);
    auto *pg = reinterpret_cast<int32_t *>(h + o_pages);
    int32_t row = 0, poff_acc = 0;
    int64_t sacc = 0;
    for (int32_t i = 0; i < num_spans; ++i) {
      const dsa_span_t &s = spans[i];
      if (s.num_pages) std::memcpy(pg + poff_acc, s.pages, sizeof(int32_t) * s.num_pages);
      for (int32_t r = 0; r < s.q_len; ++r, ++row) {
        pos[row] = s.ctx_start + r;
        poff[row] = poff_acc;
        np[row] = s.num_pages;
        ps[row] = s.page_start;
        soff[row] = sacc;
        sacc += static_cast<int64_t>(pos[row]) + 1;
      }
      poff_acc += s.num_pages;
    }
    for (int set = 0; set < 2; ++set) {
      if (!groups[set].empty()) std::memcpy(h + o_g[set], groups[set].data(), groups[set].size() * sizeof(IdxGroup));
      if (!items[set].empty()) std::memcpy(h + o_i[set], items[set].data(), items[set].size() * sizeof(IdxItem));
      if (!cta_begin[set].empty())
        std::memcpy(h + o_c[set], cta_begin[set].data(), cta_begin[set].size() * sizeof(int32_t));
    }
    if (!units.empty()) std::memcpy(h + o_u, units.data(), units.size() * sizeof(AttUnit));
    if (!combines.empty()) std::memcpy(h + o_cb, combines.data(), combines.size() * sizeof(AttCombine));
    if (!clusters.empty()) std::memcpy(h + o_cl, clusters.data(), clusters.size() * sizeof(AttCluster));
  }

  if (is_host_only(ctx)) {
    *out = plan;
    return DSA_OK;
  }
  if (cudaSetDevice(ctx->device) != cudaSuccess) { delete plan; return DSA_ERR_CUDA; }
  dsa_status st = ensure_scratch(ctx, static_cast<size_t>(num_scores), static_cast<size_t>(plan->n_slots));
  if (st != DSA_OK) { delete plan; return st; }
  if (cudaMallocAsync(reinterpret_cast<void **>(&plan->dev), bytes, plan->stream) != cudaSuccess) {
    delete plan;
    return DSA_ERR_OOM;
  }
  if (cudaMemcpyAsync(plan->dev, h, bytes, cudaMemcpyHostToDevice, plan->stream) != cudaSuccess) {
    cudaFreeAsync(plan->dev, plan->stream);
    delete plan;
    return DSA_ERR_CUDA;
  }
  char *d = plan->dev;
  plan->row_pos = reinterpret_cast<int32_t *>(d + o_pos);
  plan->row_page_off = reinterpret_cast<int32_t *>(d + o_poff);
  plan->row_npages = reinterpret_cast<int32_t *>(d + o_np);
  plan->row_page_start = reinterpret_cast<int32_t *>(d + o_ps);
  plan->row_score_off = reinterpret_cast<int64_t *>(d + o_soff);
  plan->pages = reinterpret_cast<int32_t *>(d + o_pages);
  for (int set = 0; set < 2; ++set) {
    plan->idx[set].groups = reinterpret_cast<IdxGroup *>(d + o_g[set]);
    plan->idx[set].items = reinterpret_cast<IdxItem *>(d + o_i[set]);
    plan->idx[set].cta_begin = reinterpret_cast<int32_t *>(d + o_c[set]);
  }
  plan->units = reinterpret_cast<AttUnit *>(d + o_u);
  plan->combine = reinterpret_cast<AttCombine *>(d + o_cb);
  plan->clusters = reinterpret_cast<AttCluster *>(d + o_cl);
  *out = plan;
  return DSA_OK;
}

void dsa_plan_destroy(dsa_plan_t *plan) {
  if (!plan) return;
  if (plan->capturable) {
    cudaSetDevice(plan->ctx->device);
    cudaFree(plan->dev);
    cudaFree(plan->own_scores);
    cudaFree(plan->own_opart);
    cudaFree(plan->own_mlpart);
  } else if (plan->dev && !is_host_only(plan->ctx)) {
    cudaSetDevice(plan->ctx->device);
    cudaFreeAsync(plan->dev, plan->stream);
  }
  delete plan;
}

dsa_status dsa_plan_capturable(dsa_ctx_t *ctx, int32_t max_rows, int32_t max_spans, int64_t max_scores,
                               int32_t page_start_align, int32_t cache_pages, dsa_stream_t stream,
                               dsa_plan_t **out) {
  if (!out) return DSA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!ctx || is_host_only(ctx) || max_rows <= 0 || max_spans <= 0 || max_rows > kPlanMaxRows ||
      max_spans > kPlanMaxSpans || max_scores < max_rows || max_scores > (int64_t(1) << 40) || page_start_align <= 0 ||
      cache_pages < 0)
    return DSA_ERR_INVALID_ARG;
  const dsa_config_t &c = ctx->cfg;
  // worst-case work for any update within the capacities
  // indexer items: one per row plus one per CTA boundary inside a row, and
  // the CTAs are at most the key tiles (max_scores / 128 + 2 per row)
  const int idx_ctas = std::max(1, ctx->num_sms * indexer_ctas_per_sm(c, 1));
  const int64_t items_cap =
      static_cast<int64_t>(max_rows) + std::min<int64_t>(idx_ctas, max_scores / kIndexTile + 2 * static_cast<int64_t>(max_rows)) + 1;
  // attention: at most one cluster per two SMs; each cut between clusters
  // adds one unit and at most one split row, and each split row's pieces are
  // its cuts plus one
  const int32_t clusters_cap = std::max(1, std::min(ctx->num_sms / 2, 1024));   // the device planner: one thread each
  const int64_t units_cap = static_cast<int64_t>(max_rows) + clusters_cap;
  const int32_t combine_cap = std::min(max_rows, clusters_cap);
  const int32_t slots_cap = 2 * clusters_cap;
  if (items_cap > INT32_MAX / 2 || units_cap > INT32_MAX / 2) return DSA_ERR_INVALID_ARG;
  const int idx_cap = idx_ctas;

  dsa_plan_t *plan = new (std::nothrow) dsa_plan_t();
  if (!plan) return DSA_ERR_OOM;
  plan->ctx = ctx;
  plan->stream = reinterpret_cast<cudaStream_t>(stream);
  plan->capturable = true;
  plan->T = max_rows;
  plan->n_spans = max_spans;
  plan->max_spans = max_spans;
  plan->needs_selection = 1;
  plan->cache_pages = cache_pages;
  plan->num_scores = max_scores;
  plan->max_pos = INT32_MAX;
  plan->page_start_align = page_start_align;
  plan->box_rows = index_box_rows(c.page_size);
  plan->items_cap = static_cast<int32_t>(items_cap);
  plan->combine_cap = combine_cap;
  plan->n_units = static_cast<int32_t>(units_cap);
  plan->n_combine = combine_cap;
  plan->n_slots = slots_cap;
  plan->n_clusters = clusters_cap;
  plan->n_index_items = plan->items_cap;
  plan->splits_max = clusters_cap;
  IdxSet &set = plan->idx[0];
  set.G = 1;
  set.n_groups = max_rows;
  set.n_items = plan->items_cap;
  set.n_ctas = idx_cap;

  Layout lay;
  const size_t o_pos = lay.take<int32_t>(max_rows), o_poff = lay.take<int32_t>(max_rows),
               o_np = lay.take<int32_t>(max_rows), o_ps = lay.take<int32_t>(max_rows),
               o_soff = lay.take<int64_t>(max_rows), o_g = lay.take<IdxGroup>(max_rows),
               o_i = lay.take<IdxItem>(items_cap), o_c = lay.take<int32_t>(idx_cap + 1),
               o_u = lay.take<AttUnit>(units_cap), o_cb = lay.take<AttCombine>(combine_cap), o_n = lay.take<int32_t>(8),
               o_cl = lay.take<AttCluster>(clusters_cap);
  auto fail = [&](dsa_status st) {
    dsa_plan_destroy(plan);
    return st;
  };
  if (cudaSetDevice(ctx->device) != cudaSuccess) return fail(DSA_ERR_CUDA);
  if (prepare_plan_update(max_rows, max_spans) != cudaSuccess) return fail(DSA_ERR_CUDA);
  const size_t hl = static_cast<size_t>(c.heads) * c.kv_lora_rank;
  if (cudaMalloc(reinterpret_cast<void **>(&plan->dev), lay.bytes) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void **>(&plan->own_scores), static_cast<size_t>(max_scores) * sizeof(float)) !=
          cudaSuccess ||
      cudaMalloc(reinterpret_cast<void **>(&plan->own_opart), static_cast<size_t>(slots_cap) * hl * sizeof(float)) !=
          cudaSuccess ||
      cudaMalloc(reinterpret_cast<void **>(&plan->own_mlpart),
                 static_cast<size_t>(slots_cap) * c.heads * 2 * sizeof(float)) != cudaSuccess)
    return fail(DSA_ERR_OOM);
  char *d = plan->dev;
  plan->row_pos = reinterpret_cast<int32_t *>(d + o_pos);
  plan->row_page_off = reinterpret_cast<int32_t *>(d + o_poff);
  plan->row_npages = reinterpret_cast<int32_t *>(d + o_np);
  plan->row_page_start = reinterpret_cast<int32_t *>(d + o_ps);
  plan->row_score_off = reinterpret_cast<int64_t *>(d + o_soff);
  set.groups = reinterpret_cast<IdxGroup *>(d + o_g);
  set.items = reinterpret_cast<IdxItem *>(d + o_i);
  set.cta_begin = reinterpret_cast<int32_t *>(d + o_c);
  plan->units = reinterpret_cast<AttUnit *>(d + o_u);
  plan->combine = reinterpret_cast<AttCombine *>(d + o_cb);
  plan->counts = reinterpret_cast<int32_t *>(d + o_n);
  plan->clusters = reinterpret_cast<AttCluster *>(d + o_cl);
  // an empty plan until the first update: every row is padding, no work
  std::vector<char> h(lay.bytes, 0);
  std::fill_n(reinterpret_cast<int32_t *>(h.data() + o_pos), max_rows, -1);
  for (int64_t i = 0; i < items_cap; ++i) reinterpret_cast<IdxItem *>(h.data() + o_i)[i] = IdxItem{-1, 0, 0, 0};
  for (int64_t i = 0; i < units_cap; ++i) reinterpret_cast<AttUnit *>(h.data() + o_u)[i] = AttUnit{-1, 0, 0, -1};
  for (int32_t i = 0; i < combine_cap; ++i) reinterpret_cast<AttCombine *>(h.data() + o_cb)[i] = AttCombine{-1, 0, 0, 0};
  // (clusters start idle: zero-filled, u0 == u1)
  if (cudaMemcpy(plan->dev, h.data(), lay.bytes, cudaMemcpyHostToDevice) != cudaSuccess) return fail(DSA_ERR_CUDA);
  *out = plan;
  return DSA_OK;
}

dsa_status dsa_plan_update(dsa_ctx_t *ctx, dsa_plan_t *plan, const int32_t *num_spans,
                           const dsa_device_span_t *spans, const int32_t *pages, int64_t num_page_ids,
                           dsa_stream_t stream) {
  if (!ctx || !plan || plan->ctx != ctx || !plan->capturable || is_host_only(ctx)) return DSA_ERR_INVALID_ARG;
  if (!num_spans || !spans || !pages || num_page_ids < 0) return DSA_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  plan->pages = const_cast<int32_t *>(pages);
  plan->page_ids = num_page_ids;
  ctx->last_launches = 1;
  return cuda_status(ctx, launch_plan_update(ctx, plan, num_spans, spans, num_page_ids,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

dsa_status dsa_plan_read_counts(const dsa_plan_t *plan, int32_t counts[8]) {
  if (!plan || !counts || !plan->capturable) return DSA_ERR_INVALID_ARG;
  if (cudaSetDevice(plan->ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpy(counts, plan->counts, 8 * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

dsa_status dsa_plan_get_info(const dsa_plan_t *plan, dsa_plan_info_t *info) {
  if (!plan || !info) return DSA_ERR_INVALID_ARG;
  info->num_rows = plan->T;
  info->num_spans = plan->n_spans;
  info->needs_selection = plan->needs_selection;
  info->index_items = plan->n_index_items;
  info->num_scores = plan->num_scores;
  info->attend_units = plan->n_units;
  info->attend_splits_max = plan->splits_max;
  bool tc = plan->box_rows >= 8;
  for (int set = 0; set < 2; ++set)
    if (plan->idx[set].n_items > 0 && !indexer_tc_supported(plan->ctx->cfg, plan->idx[set].G)) tc = false;
  info->index_tensor_cores = tc ? 1 : 0;
  info->index_box_rows = plan->box_rows;
  return DSA_OK;
}

static dsa_status check_call(dsa_ctx_t *ctx, const dsa_plan_t *plan) {
  if (!ctx || !plan || plan->ctx != ctx || is_host_only(ctx)) return DSA_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

dsa_status dsa_store_keys(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *keys, void *index_cache,
                          dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!keys || !index_cache) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_store_keys(ctx, plan, keys, index_cache, reinterpret_cast<cudaStream_t>(stream),
                                    &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_quantize_store_keys(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *keys_bf16,
                                   void *index_cache, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (ctx->cfg.index_fmt != DSA_INDEX_FP8_132 || ctx->cfg.index_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!keys_bf16 || !index_cache) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_keys(ctx, plan, keys_bf16, index_cache, reinterpret_cast<cudaStream_t>(stream),
                                       &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_quantize_store_latents(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *latents_bf16,
                                      void *latent_cache, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (ctx->cfg.latent_fmt != DSA_LATENT_FP8_656 || ctx->cfg.kv_lora_rank != 512 || ctx->cfg.rope_dim != 64)
    return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!latents_bf16 || !latent_cache) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_latents(ctx, plan, latents_bf16, latent_cache,
                                          reinterpret_cast<cudaStream_t>(stream), &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_index_scores(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                            const void *index_cache, float *scores, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!q || !w || !index_cache || !scores) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_index_scores(ctx, plan, q, w, index_cache, scores, reinterpret_cast<cudaStream_t>(stream),
                                      &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_topk_from_scores(dsa_ctx_t *ctx, const dsa_plan_t *plan, const float *scores, int32_t *selection,
                                dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!scores || !selection) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_topk(ctx, plan, scores, selection, reinterpret_cast<cudaStream_t>(stream),
                              &ctx->last_launches);
  if (e == cudaSuccess) plan->last_selection = selection;
  return cuda_status(ctx, e);
}

dsa_status dsa_index_topk(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                          const void *index_cache, int32_t *selection, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!q || !w || !index_cache || !selection) return DSA_ERR_INVALID_ARG;
  if (!plan->own_scores && static_cast<size_t>(plan->num_scores) > ctx->scores_cap)
    return DSA_ERR_INVALID_ARG;  // plan of another size
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t n = 0;
  float *scores = plan_scores(ctx, plan);
  cudaError_t e = launch_index_scores(ctx, plan, q, w, index_cache, scores, s, &n);
  if (e == cudaSuccess) e = launch_topk(ctx, plan, scores, selection, s, &n);
  if (e == cudaSuccess) plan->last_selection = selection;
  ctx->last_launches = n;
  return cuda_status(ctx, e);
}

static bool f8q_ok(const dsa_ctx_t *ctx, const dsa_plan_t *plan) {
  return ctx->cfg.index_fmt == DSA_INDEX_FP8_132 && ctx->cfg.index_heads == 64 && ctx->cfg.index_dim == 128 &&
         indexer_f8q_supported(ctx->cfg, plan);
}

dsa_status dsa_quantize_q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_bf16, void *q_codes, float *q_scale,
                          dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (ctx->cfg.index_heads != 64 || ctx->cfg.index_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!q_bf16 || !q_codes || !q_scale) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_q(ctx, plan, q_bf16, q_codes, q_scale, reinterpret_cast<cudaStream_t>(stream),
                                    &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_index_scores_fp8q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_codes, const float *q_scale,
                                 const float *w, const void *index_cache, float *scores, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (!f8q_ok(ctx, plan)) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!q_codes || !q_scale || !w || !index_cache || !scores) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_index_scores_f8q(ctx, plan, q_codes, q_scale, w, index_cache, scores,
                                          reinterpret_cast<cudaStream_t>(stream), &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_index_topk_fp8q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_codes, const float *q_scale,
                               const float *w, const void *index_cache, int32_t *selection, dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (!f8q_ok(ctx, plan)) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!q_codes || !q_scale || !w || !index_cache || !selection) return DSA_ERR_INVALID_ARG;
  if (!plan->own_scores && static_cast<size_t>(plan->num_scores) > ctx->scores_cap) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t n = 0;
  float *scores = plan_scores(ctx, plan);
  cudaError_t e = launch_index_scores_f8q(ctx, plan, q_codes, q_scale, w, index_cache, scores, s, &n);
  if (e == cudaSuccess) e = launch_topk(ctx, plan, scores, selection, s, &n);
  if (e == cudaSuccess) plan->last_selection = selection;
  ctx->last_launches = n;
  return cuda_status(ctx, e);
}

dsa_status dsa_attend(dsa_ctx_t *ctx, const dsa_plan_t *plan, const int32_t *selection, const void *q_nope,
                      const void *q_pe, const void *latent_cache, const float *sink, float sm_scale, void *out,
                      dsa_stream_t stream) {
  dsa_status st = check_call(ctx, plan);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!selection || !q_nope || !latent_cache || !out || (!q_pe && ctx->cfg.rope_dim > 0)) return DSA_ERR_INVALID_ARG;
  if (!plan->own_opart && static_cast<size_t>(plan->n_slots) > ctx->part_cap) return DSA_ERR_INVALID_ARG;
  cudaError_t e = launch_attend(ctx, plan, selection, q_nope, q_pe, latent_cache, sink, sm_scale, out,
                                reinterpret_cast<cudaStream_t>(stream), &ctx->last_launches);
  return cuda_status(ctx, e);
}

dsa_status dsa_attend_shared(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_nope, const void *q_pe,
                             const void *latent_cache, const float *sink, float sm_scale, void *out,
                             dsa_stream_t stream) {
  if (plan && plan->T > 0 && !plan->last_selection) return DSA_ERR_INVALID_ARG;   // no FULL layer yet
  return dsa_attend(ctx, plan, plan ? plan->last_selection : nullptr, q_nope, q_pe, latent_cache, sink, sm_scale,
                    out, stream);
}

dsa_status dsa_get_error(dsa_ctx_t *ctx, dsa_stream_t stream) {
  if (!ctx || is_host_only(ctx)) return DSA_ERR_INVALID_ARG;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ctx->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  if (word && cudaMemset(ctx->err, 0, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (word & kErrTimeout) return DSA_ERR_TIMEOUT;
  if (word & kErrSpans) return DSA_ERR_BAD_SPANS;
  if (word & kErrBounds) return DSA_ERR_BOUNDS;
  return DSA_OK;
}

int32_t dsa_last_launch_count(const dsa_ctx_t *ctx) { return ctx ? ctx->last_launches : 0; }

const char *dsa_last_cuda_error(const dsa_ctx_t *ctx) { return ctx ? ctx->last_cuda_error : ""; }

}  // extern "C"
