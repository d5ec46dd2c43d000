// dsa_internal.h -- host/device structures shared by the C-ABI layer and the
// kernel launchers.  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <vector>

#include "dsa.h"
#include "errors.h"

namespace dsa {

// A group of consecutive rows of one span that the indexer scores together
// (1 row for decode rows, up to 4 for prefill chunks).
struct IdxGroup {
  int32_t row0;        // first row
  int32_t nrows;       // rows in the group (positions pos0 .. pos0+nrows-1)
  int32_t pos0;        // position of the first row
  int32_t page_off;    // offset of the span's page list in the plan's pages[]
  int32_t npages;      // length of that list
  int32_t page_start;  // slot of token 0
  int32_t ntiles;      // key tiles of 128 covering positions 0 .. pos0+nrows-1 (index_group_tiles)
  int32_t lead;        // tile rows before token 0: tile t holds positions t*128 - lead .. t*128 - lead + 127
};

// A contiguous run of key tiles of one group.
struct IdxItem {
  int32_t group;
  int32_t tile0;
  int32_t tile1;
  int32_t pad;
};

// An attention work unit: selection entries [k0, k1) of one row; `slot` >= 0
// when the row is split and the unit writes a partial result.
struct AttUnit {
  int32_t row;
  int32_t k0;
  int32_t k1;
  int32_t slot;
};

// A row whose attention was split over `nsplit` units with partial slots
// first_slot .. first_slot + nsplit - 1.
struct AttCombine {
  int32_t row;
  int32_t first_slot;
  int32_t nsplit;
  int32_t pad;
};

// The work of one persistent attention cluster: units [u0, u1), `tiles` key
// tiles in all.  u0 == u1: an idle cluster (capturable plans' padding).
struct AttCluster {
  int32_t u0;
  int32_t u1;
  int32_t tiles;
  int32_t pad;
};

constexpr int kIndexTile = 128;   // keys per indexer tile (UMMA M)
constexpr int kAttTile = 64;      // keys per attention tile (UMMA N of QK)
constexpr int kNoBox = -0x7fffffff - 1;   // index producers: a lane with no key box in the tile
constexpr int kPlanMaxRows = 8192;   // capturable plans: rows and spans the device planner holds in shared memory
constexpr int kPlanMaxSpans = 4096;

// Height of the indexer's TMA key boxes: the largest power of two <= 128 that
// divides the page size.  Key tiles start on a multiple of it in slot space
// (a span's page_start rounded down), so every box of a tile lies inside one
// page whatever the span's page_start.
__host__ __device__ inline int index_box_rows(int page_size) {
  int bh = 1;
  while (bh < kIndexTile && page_size % (bh * 2) == 0) bh *= 2;
  return bh;
}
// Tile rows ahead of a span's token 0: page_start's distance above the box
// boundary below it.
__host__ __device__ inline int32_t index_tile_lead(int32_t page_start, int box_rows) {
  return page_start % box_rows;
}
// Key tiles of a group whose rows see positions 0 .. nkeys-1.
__host__ __device__ inline int32_t index_group_tiles(int64_t nkeys, int32_t lead) {
  return static_cast<int32_t>((lead + nkeys + kIndexTile - 1) / kIndexTile);
}

// Raises a kernel's dynamic shared-memory limit on the current device once.
// The limit belongs to the device, so each GPU the process uses gets its own
// bit in `done` (devices past 63 set it on every launch); two host threads
// racing here both set the same value, which is harmless.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kern, int bytes, int device, std::atomic<uint64_t> &done) {
  const uint64_t bit = (device >= 0 && device < 64) ? (uint64_t(1) << device) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// The persistent indexer's split of a launch set's `total` key tiles (its
// groups' tiles in order) over `cap` CTAs: CTA b takes tiles
// [index_cta_start(b), index_cta_start(b + 1)), ceil(total * b / cap), so
// every CTA has floor or ceil of total / cap tiles and tile t belongs to CTA
// floor(t * cap / total).  A group a boundary crosses is one work item per
// piece.  The host planner and the device planner share these functions.
__host__ __device__ inline int64_t index_cta_start(int64_t b, int64_t total, int cap) {
  return (total * b + cap - 1) / cap;
}
__host__ __device__ inline int64_t index_cta_of_tile(int64_t t, int64_t total, int cap) {
  return t * cap / total;
}

// Order-preserving 32-bit key of a score (larger score, larger key; -0.0
// ranks as +0.0).  Every score, -inf included, has a key above 0, so 0 can
// stand for "no score".
__host__ __device__ inline uint32_t score_order_key(float f) {
  union {
    float f;
    uint32_t u;
  } v{f};
  uint32_t u = v.u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// First word of row r's block maxima in a packed block-key array: rows are
// laid out by their score offsets, off / block + r, which keeps the rows'
// ranges of pos / block + 1 words disjoint (the array needs
// num_scores / block + rows + 1 words).
__host__ __device__ inline int64_t block_key_base(int64_t score_off, int64_t row, int block) {
  return score_off / block + row;
}

// Persistent attention schedule (the host planner and the device planner share
// these functions, so both make the same units).  The step's rows, in order, are a sequence
// of S key tiles (ceil(min(topk, pos+1) / kAttTile) per row).  It is cut
// into n_clusters contiguous ranges of `per` tiles (the last one shorter), one
// per two-CTA cluster; a row that a cut crosses becomes one unit per piece,
// each writing a partial result that attend_combine_kernel merges.  Clusters
// take at least kAttMinClusterTiles tiles, and there are at most one per two
// SMs.
constexpr int kAttMinClusterTiles = 16;
// Ranges hold at least 8 tiles once S >= kAttMinClusterTiles (S / ceil(S / 16)),
// so a row has at most ceil(tiles / 8) + 1 pieces: 33 at the largest topk
// the library takes (16,384 keys, 256 tiles); the merge holds this many.
constexpr int kAttMaxPieces = 64;

__host__ __device__ inline void att_cluster_split(int64_t S, int num_sms, int32_t *n_clusters, int64_t *per) {
  const int64_t cap = num_sms / 2 > 1 ? num_sms / 2 : 1;
  int64_t n = (S + kAttMinClusterTiles - 1) / kAttMinClusterTiles;
  n = n < 1 ? 1 : (n > cap ? cap : n);
  int64_t q = (S + n - 1) / n;
  if (q < 1) q = 1;
  *per = q;
  *n_clusters = static_cast<int32_t>(S > 0 ? (S + q - 1) / q : 0);
}

// Key tiles of a row at position pos (>= 0).
__host__ __device__ inline int64_t att_row_tiles(int64_t pos, int64_t topk) {
  const int64_t nsel = pos + 1 < topk ? pos + 1 : topk;
  return (nsel + kAttTile - 1) / kAttTile;
}

// Indexer launch set: groups with the same row-group size.
struct IdxSet {
  int G = 1;                      // rows per group
  int n_groups = 0;
  int n_items = 0;
  int n_ctas = 0;                 // persistent grid
  IdxGroup *groups = nullptr;     // device
  IdxItem *items = nullptr;       // device
  int32_t *cta_begin = nullptr;   // device [n_ctas + 1]: item range of each CTA
};

}  // namespace dsa

struct dsa_ctx {
  dsa_config_t cfg;
  int device = -1;
  int num_sms = 0;
  int *err = nullptr;             // device error word
  float *scores = nullptr;        // score scratch
  size_t scores_cap = 0;          // floats
  float *opart = nullptr;         // attention partial outputs [slots][H][L]
  float *mlpart = nullptr;        // attention partial (m, l) [slots][H][2]
  size_t part_cap = 0;            // slots
  int32_t last_launches = 0;
  char last_cuda_error[160] = {0};  // name and text of the last CUDA error a call returned DSA_ERR_CUDA for
  float *static_scores = nullptr; // device address of the library's fixed score array (dsa_index_topk_static)
  uint32_t *block_keys = nullptr; // MSA block maxima scratch (dsa_msa_index_select)
  size_t block_keys_cap = 0;      // words
};

struct dsa_plan {
  dsa_ctx *ctx = nullptr;
  cudaStream_t stream = nullptr;
  int32_t T = 0, n_spans = 0, needs_selection = 0, cache_pages = 0, max_pos = 0;
  int32_t box_rows = 1;           // TMA box height of the indexer's key tiles (index_box_rows of the page size)
  int64_t num_scores = 0;
  std::vector<char> host;         // staging copy of the device metadata
  char *dev = nullptr;
  // device views
  int32_t *row_pos = nullptr, *row_page_off = nullptr, *row_npages = nullptr, *row_page_start = nullptr;
  int64_t *row_score_off = nullptr;
  int32_t *pages = nullptr;
  dsa::IdxSet idx[2];             // [0]: single-row groups, [1]: multi-row groups
  dsa::AttUnit *units = nullptr;
  int32_t n_units = 0, splits_max = 1;
  dsa::AttCluster *clusters = nullptr;  // persistent attention clusters (the grid is two CTAs per entry)
  int32_t n_clusters = 0;
  dsa::AttCombine *combine = nullptr;
  int32_t n_combine = 0, n_slots = 0;
  int32_t n_index_items = 0;
  // the selection the last FULL layer's dsa_index_topk / dsa_topk_from_scores
  // wrote for this plan (mstar DSAPlan.last_selection), for SHARED layers
  mutable const int32_t *last_selection = nullptr;
  // capturable plans (dsa_plan_capturable): the host fields above hold the
  // capacities, the device metadata is rewritten by dsa_plan_update, and the
  // plan owns its scratch
  bool capturable = false;
  int32_t max_spans = 0, items_cap = 0, combine_cap = 0, page_start_align = 1;
  int64_t page_ids = 0;                 // length of the page array of the last update
  float *own_scores = nullptr, *own_opart = nullptr, *own_mlpart = nullptr;
  int32_t *counts = nullptr;            // device [8], see dsa_plan_read_counts
};

namespace dsa {
inline float *plan_scores(const dsa_ctx *c, const dsa_plan_t *p) { return p->own_scores ? p->own_scores : c->scores; }
inline float *plan_opart(const dsa_ctx *c, const dsa_plan_t *p) { return p->own_opart ? p->own_opart : c->opart; }
inline float *plan_mlpart(const dsa_ctx *c, const dsa_plan_t *p) { return p->own_mlpart ? p->own_mlpart : c->mlpart; }
}  // namespace dsa

namespace dsa {

// Launchers (each returns cudaGetLastError() after its launches and adds the
// number of kernels it launched to *launches).
cudaError_t launch_quantize_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *keys, void *cache,
                                 cudaStream_t s, int32_t *launches);
cudaError_t launch_quantize_latents(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *latents, void *cache,
                                    cudaStream_t s, int32_t *launches);
cudaError_t launch_quantize_q(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, void *codes, float *scales,
                              cudaStream_t s, int32_t *launches);
cudaError_t launch_index_scores_f8q(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q_codes,
                                    const float *q_scale, const float *w, const void *cache, float *scores,
                                    cudaStream_t s, int32_t *launches);
bool indexer_f8q_supported(const dsa_config_t &c, const dsa_plan_t *plan);
cudaError_t launch_store_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *keys, void *cache,
                              cudaStream_t s, int32_t *launches);
cudaError_t launch_index_scores(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                const void *cache, float *scores, cudaStream_t s, int32_t *launches);
// The indexer with a block-maximum epilogue instead of the score store: for
// every row r and block b of `block` positions, block_keys[block_key_base(r) + b]
// is raised (atomicMax) to the largest score_order_key of the row's visible
// scores in that block.  The words must start at zero.  Only the bf16
// tensor-core kernels have this epilogue (index_block_keys_supported).
cudaError_t launch_index_block_keys(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                    const void *cache, uint32_t *block_keys, int block, cudaStream_t s,
                                    int32_t *launches);
bool index_block_keys_supported(const dsa_ctx *ctx, const dsa_plan_t *plan);
cudaError_t launch_topk(const dsa_ctx *ctx, const dsa_plan_t *plan, const float *scores, int32_t *sel,
                        cudaStream_t s, int32_t *launches);
cudaError_t launch_plan_update(const dsa_ctx *ctx, dsa_plan_t *plan, const int32_t *num_spans,
                               const dsa_device_span_t *spans, int64_t num_page_ids, cudaStream_t s);
// Shared memory the device planner needs for these capacities; sets the
// kernel's limit (call when the plan is made, outside any stream capture).
cudaError_t prepare_plan_update(int32_t max_rows, int32_t max_spans);
cudaError_t launch_attend(const dsa_ctx *ctx, const dsa_plan_t *plan, const int32_t *sel, const void *q_nope,
                          const void *q_pe, const void *latent, const float *sink, float sm_scale, void *out,
                          cudaStream_t s, int32_t *launches);

// Device address of the fixed score array behind dsa_index_topk_static on the
// current device (loads the module that holds it, so the array is taken when
// the context is created rather than at the first call).
cudaError_t static_scores_address(int device, float **out);

// Shapes the tensor-core kernels implement (others run the simple kernels).
bool indexer_tc_supported(const dsa_config_t &c, int G);
bool attend_tc_supported(const dsa_config_t &c);
int indexer_group_rows(const dsa_config_t &c);   // rows per multi-row group (4 or 1)
int indexer_ctas_per_sm(const dsa_config_t &c, int G);

// Tensor-map encoding through the driver entry point (no libcuda link).
bool encode_tiled_2d(CUtensorMap *tm, CUtensorMapDataType dtype, void *base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

bool encode_tiled_3d(CUtensorMap *tm, CUtensorMapDataType dtype, void *base, const uint64_t dims[3],
                     const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swz);

}  // namespace dsa
