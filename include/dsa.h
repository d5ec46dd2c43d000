/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention library.
 *
 * The operation (mstar page "mstar.engine.resources.dsa.manager", module
 * summary, index_topk, select_topk_causal and DSAManager.attend):
 *
 *   1. indexer score   s[r, j] = sum_h w[r,h] * relu(q[r,h] . k[j]), in fp32,
 *                      for every key j = 0 .. pos(r) of row r's request
 *                      (a row sees the keys up to its own position, itself included);
 *   2. causal top-k    the topk highest-scoring positions of each row, int32,
 *                      ties to the earlier position, -1 padded;
 *   3. sparse MLA      absorbed MLA over the selected latents only:
 *                      out[r,h] = softmax_j((q_nope[r,h] . c_j + q_pe[r,h] . kpe_j) * sm_scale) . c_j,
 *                      shape (T, H, kv_lora_rank).
 *
 * Everything here is asynchronous on the caller's stream except dsa_create,
 * dsa_plan (host work, then one host-to-device copy on the stream) and
 * dsa_get_error (synchronises the stream).  All tensor arguments are DEVICE
 * pointers owned by the caller, row-major and densely packed, unless stated
 * otherwise.  Every call returns a dsa_status; no call aborts the process.
 *
 * Paged layout (DSASpan / DSAPlan on the mstar page): a request's token at
 * position p lives at slot = page_start + p of its page list, i.e. in page
 * pages[slot / page_size] at offset slot % page_size.  The latent cache and the
 * index-key cache share page ids.
 *
 * Cache formats (per token, per layer):
 *   latent  DSA_LATENT_BF16    : [kv_lora_rank | rope_dim] bf16 (1,152 B at 512+64)
 *           DSA_LATENT_FP8_656 : [512 e4m3 | 4 fp32 scales, one per 128 | 64 bf16 rope]
 *                                (656 B; ttnn.transformer.sparse_sdpa "kv" parameter;
 *                                 LLMServingSim "What the KV cache actually holds")
 *   index   DSA_INDEX_BF16     : index_dim bf16 per token, cache [pages][page_size][index_dim]
 *           DSA_INDEX_FP8_132  : 128 e4m3 + one fp32 scale per token (132 B; LLMServingSim,
 *                                same section), stored page-blocked: each page is
 *                                [page_size x 128 codes][page_size x fp32 scale].
 */
#ifndef DSA_GB300_DSA_H_
#define DSA_GB300_DSA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t).  NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *dsa_stream_t;

typedef int32_t dsa_status;
enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, spans that do not tile the rows */
  DSA_ERR_SHORT_HISTORY = 2,  /* a span's pages cannot hold positions 0 .. ctx_start+q_len-1
                                 (mstar IndexKeyStore.history raises in this case) */
  DSA_ERR_OOM = 3,            /* device or host allocation failed */
  DSA_ERR_CUDA = 4,           /* a CUDA runtime call failed */
  DSA_ERR_BOUNDS = 5,         /* device side: a selected position outside 0..pos(r), or a
                                 page id outside the cache; the access was skipped */
  DSA_ERR_TIMEOUT = 6,        /* device side: a pipeline wait gave up after its time limit */
  DSA_ERR_UNSUPPORTED = 7     /* shape or format the library does not implement */
};

enum { DSA_LATENT_BF16 = 0, DSA_LATENT_FP8_656 = 1 };
enum { DSA_INDEX_BF16 = 0, DSA_INDEX_FP8_132 = 1 };

/* Problem shape, fixed for a context. */
typedef struct dsa_config {
  int32_t index_heads;   /* indexer heads Hi (64 for DeepSeek-V3.2) */
  int32_t index_dim;     /* indexer head dim Di (128) */
  int32_t topk;          /* positions kept per row (2048; at most 16384) */
  int32_t heads;         /* MLA query heads H (128) */
  int32_t kv_lora_rank;  /* latent width L (512); also the output width */
  int32_t rope_dim;      /* rope width R (64) */
  int32_t page_size;     /* tokens per cache page */
  int32_t latent_fmt;    /* DSA_LATENT_* */
  int32_t index_fmt;     /* DSA_INDEX_* */
} dsa_config_t;

/* One request's rows of a step (mstar DSASpan): q_len rows from row q_start,
 * the first at request-local position ctx_start; the request's token p sits
 * at slot page_start + p of `pages` (num_pages HOST int32 page ids).  Spans
 * must tile rows [0, T) in order. */
typedef struct dsa_span {
  int64_t request_id;    /* caller's id, carried for diagnostics only */
  int32_t q_start;
  int32_t q_len;         /* > 0 */
  int32_t ctx_start;     /* >= 0 */
  int32_t page_start;    /* >= 0 */
  const int32_t *pages;  /* host memory, read during dsa_plan only */
  int32_t num_pages;
  int32_t reserved;      /* set to 0 */
} dsa_span_t;

typedef struct dsa_ctx dsa_ctx_t;
typedef struct dsa_plan dsa_plan_t;

/* Plan statistics (host-side copy). */
typedef struct dsa_plan_info {
  int32_t num_rows;          /* T */
  int32_t num_spans;
  int32_t needs_selection;   /* 1 when some row sees more than topk keys (mstar DSAPlan) */
  int32_t index_items;       /* indexer work items (tiles of 128 keys, grouped) */
  int64_t num_scores;        /* sum over rows of pos(r)+1: the score scratch length */
  int32_t attend_units;      /* attention work units (row x key split) */
  int32_t attend_splits_max; /* largest key split count of any row */
  int32_t index_tensor_cores;/* 1 when the plan's index scores run on the tensor-core kernels (any
                                page_start, page_size a multiple of 8), 0 for the CUDA-core kernel */
  int32_t index_box_rows;    /* height of the indexer's TMA key boxes (a power of two dividing page_size) */
} dsa_plan_info_t;

/* Create a context on CUDA device `device` (>= 0).  device = -1 creates a
 * host-only context: dsa_plan validates spans and fills dsa_plan_info but
 * makes no CUDA call, and every compute entry point returns
 * DSA_ERR_INVALID_ARG.  Returns DSA_ERR_UNSUPPORTED for shapes outside the
 * library's kernels (see DSA_ERR_UNSUPPORTED below each entry point). */
dsa_status dsa_create(const dsa_config_t *cfg, int device, dsa_ctx_t **out);
void dsa_destroy(dsa_ctx_t *ctx);

/* Build a plan from host spans (mstar DSAManager.plan / DSAPlan): validates
 * the spans, computes every row's position and page list, the indexer work
 * items and the attention units, and copies them to the device on `stream`
 * (stream-ordered allocation).  cache_pages is the number of pages in the
 * caches (page ids must be < cache_pages).  The plan may grow the context's
 * scratch (cudaMalloc; synchronous when it grows).  Errors:
 * DSA_ERR_INVALID_ARG (spans do not tile the rows in order, q_len <= 0,
 * negative ctx_start/page_start, null pages, page id out of range),
 * DSA_ERR_SHORT_HISTORY (too few pages for ctx_start + q_len tokens). */
dsa_status dsa_plan(dsa_ctx_t *ctx, const dsa_span_t *spans, int32_t num_spans, int32_t cache_pages,
                    dsa_stream_t stream, dsa_plan_t **out);
/* Frees the plan's device metadata in order on the plan's stream. */
void dsa_plan_destroy(dsa_plan_t *plan);
dsa_status dsa_plan_get_info(const dsa_plan_t *plan, dsa_plan_info_t *info);

/* Store the step's index keys (mstar DSAManager.store_keys): row r's key goes
 * to the slot of its own position.  keys: (T, index_dim) bf16, or (T, 132)
 * uint8 rows [128 e4m3 | fp32 scale] for DSA_INDEX_FP8_132.  index_cache: the
 * page-resident index cache in the context's index format.  Must precede
 * dsa_index_topk for the same step (the current chunk is stored before
 * selection). */
dsa_status dsa_store_keys(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *keys, void *index_cache,
                          dsa_stream_t stream);

/* Quantize-on-store (an extension: the pages store rows already in cache
 * format, mstar DSAManager.store_keys; the fp8 row layouts are LLMServingSim's
 * "What the KV cache actually holds").  Each row is quantised into the slot
 * of its own position, like dsa_store_keys:
 *   per group: scale = amax / 448 in fp32 (1 for an all-zero group);
 *   code = E4M3(x / scale), the fp32 quotient rounded to nearest with ties to
 *   even, saturating at 448 (the largest finite E4M3 value).
 * dsa_quantize_store_keys: keys_bf16 (T, 128) bf16 -> 132-byte rows (one group
 *   per row) in the page-blocked index cache; needs DSA_INDEX_FP8_132 and
 *   index_dim 128.
 * dsa_quantize_store_latents: latents_bf16 (T, 512 + 64) bf16 -> 656-byte rows
 *   (four groups of 128 columns; the 64 rope values copied as bf16); needs
 *   DSA_LATENT_FP8_656, kv_lora_rank 512, rope_dim 64.
 * Device pointers, caller-owned; the caches are written in place.  Errors:
 * DSA_ERR_UNSUPPORTED for other formats or shapes, DSA_ERR_INVALID_ARG for
 * null pointers; a page id outside the cache sets the device error word
 * (DSA_ERR_BOUNDS at the next dsa_get_error) and the row is skipped. */
dsa_status dsa_quantize_store_keys(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *keys_bf16,
                                   void *index_cache, dsa_stream_t stream);
dsa_status dsa_quantize_store_latents(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *latents_bf16,
                                      void *latent_cache, dsa_stream_t stream);

/* Score and select (mstar index_topk + select_topk_causal): q (T, Hi, Di)
 * bf16, w (T, Hi) fp32 (any scales folded in), index_cache as above;
 * selection (T, topk) int32 out: each row's selected positions in ascending
 * order, then -1 (rows that see fewer than topk keys keep them all).  Ties
 * go to the earlier position.  Scores are fp32 and live in the context's
 * scratch. */
dsa_status dsa_index_topk(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                          const void *index_cache, int32_t *selection, dsa_stream_t stream);

/* The indexer score alone (step 1): scores out, fp32, row r's pos(r)+1
 * scores starting at offset sum_{i<r} (pos(i)+1) (dsa_plan_info.num_scores
 * in total). */
dsa_status dsa_index_scores(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                            const void *index_cache, float *scores, dsa_stream_t stream);

/* The selection alone (step 2) over caller-provided scores in the layout
 * dsa_index_scores writes. */
dsa_status dsa_topk_from_scores(dsa_ctx_t *ctx, const dsa_plan_t *plan, const float *scores,
                                int32_t *selection, dsa_stream_t stream);

/* Sparse absorbed MLA (mstar DSAManager.attend; V = the first kv_lora_rank
 * columns of each latent row as in ttnn sparse_sdpa): selection (T, topk)
 * int32 request-local positions, -1 entries skipped (entries outside
 * 0..pos(r) set DSA_ERR_BOUNDS and are skipped); q_nope (T, H, L) bf16;
 * q_pe (T, H, R) bf16; latent_cache in the context's latent format with this
 * step's latents already written; sink (H) fp32 logits already in scaled
 * units that join only the softmax denominator, or NULL; out (T, H, L) bf16.
 * A row with nothing selected and no sink gets zeros. */
dsa_status dsa_attend(dsa_ctx_t *ctx, const dsa_plan_t *plan, const int32_t *selection, const void *q_nope,
                      const void *q_pe, const void *latent_cache, const float *sink, float sm_scale, void *out,
                      dsa_stream_t stream);

/* A SHARED layer (mstar DSAManager.shared_selection, DSAPlan.last_selection:
 * "SHARED layers reuse the last FULL layer's pick this forward", IndexShare):
 * dsa_attend over the selection buffer that the last dsa_index_topk or
 * dsa_topk_from_scores call with this plan wrote.  The plan keeps only the
 * pointer: the caller keeps that buffer alive and unchanged for the SHARED
 * layers of the step.  dsa_index_topk_static does not record its output here
 * (pass its selection to dsa_attend).  Same arguments and errors as
 * dsa_attend, plus DSA_ERR_INVALID_ARG when no selection has been recorded for
 * this plan. */
dsa_status dsa_attend_shared(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_nope, const void *q_pe,
                             const void *latent_cache, const float *sink, float sm_scale, void *out,
                             dsa_stream_t stream);

/* dsa_index_topk for callers that cannot allocate device memory at step time
 * (a process that reserves HBM up front in its own pool and permits no driver
 * allocation while serving).  The pages have no counterpart to this call.
 * Same arguments, results and errors as dsa_index_topk, but the fp32 scores
 * live in a fixed array inside the library (DSA_STATIC_SCORES_MAX floats,
 * 16 MiB) instead of the context's scratch; the call itself allocates
 * nothing.  The array is taken on a GPU when the first context on it is
 * created: dsa_create looks up its device address (cudaGetSymbolAddress),
 * which loads the module holding it even under lazy module loading, and it
 * stays until the process exits.  A plan with more than
 * DSA_STATIC_SCORES_MAX scores (the sum over rows of pos+1) is rejected with
 * DSA_ERR_SCRATCH_LIMIT before anything runs.  All calls share the array:
 * calls whose kernels overlap on the GPU race and must be serialised by the
 * caller. */
#define DSA_STATIC_SCORES_MAX (4 * 1024 * 1024)
enum { DSA_ERR_SCRATCH_LIMIT = 8 };
dsa_status dsa_index_topk_static(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q, const float *w,
                                 const void *index_cache, int32_t *selection, dsa_stream_t stream);

/* ---- fp8 query for the indexer -----------------------------------------
 * The indexer score with an e4m3 query over the fp8 index cache
 * (DSA_INDEX_FP8_132, index_heads 64, index_dim 128): ttnn
 * .transformer.sparse_sdpa takes its q as "bf16 or fp8_e4m3"; the index row
 * is LLMServingSim's 132-byte [128 e4m3 | fp32 scale] ("What the KV cache
 * actually holds").  Here the query of (row r, head h) is
 *   q[r,h,d] = e4m3(q_codes[r,h,d]) * q_scale[r,h],
 * and the score is the same definition as dsa_index_scores:
 *   s[r,j] = sum_h w[r,h] * relu(q[r,h] . k[j]),  k[j,d] = e4m3(code) * scale,
 * computed with e4m3 x e4m3 tensor-core products accumulated in fp32.
 *
 * dsa_quantize_q: q_bf16 (T, 64, 128) bf16 -> q_codes (T, 64, 128) uint8 e4m3
 *   and q_scale (T, 64) fp32 with the quantize-on-store rule per (row, head):
 *   scale = amax / 448 in fp32 (1 for an all-zero head), code = E4M3(x /
 *   scale), round to nearest even, saturating at 448.
 * dsa_index_scores_fp8q / dsa_index_topk_fp8q: as dsa_index_scores /
 *   dsa_index_topk with (q_codes, q_scale) in place of q (q_scale may have
 *   any sign; the quantiser writes scales >= 0).
 * Device pointers, caller-owned.  DSA_ERR_UNSUPPORTED for other index formats
 * or shapes, or a page size that is not a multiple of 8 (any page_start is
 * accepted); DSA_ERR_INVALID_ARG for null pointers. */
dsa_status dsa_quantize_q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_bf16, void *q_codes, float *q_scale,
                          dsa_stream_t stream);
dsa_status dsa_index_scores_fp8q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_codes, const float *q_scale,
                                 const float *w, const void *index_cache, float *scores, dsa_stream_t stream);
dsa_status dsa_index_topk_fp8q(dsa_ctx_t *ctx, const dsa_plan_t *plan, const void *q_codes, const float *q_scale,
                               const float *w, const void *index_cache, int32_t *selection, dsa_stream_t stream);

/* ---- Capturable plans --------------------------------------------------
 * The pages' follow-up gives selection and attention fixed-shape buffers "so
 * a decode can capture" (mstar.engine.resources.dsa.manager, module
 * overview), and graph mode pads a layout to its bucket's ceiling with
 * zero-length entries and sizes index buffers for the worst prefix sum the
 * bucket allows (mstar.engine.resources.attn.ragged.block_causal:
 * RaggedBlockCausalWrapper, max_blocks, max_prefix_tokens).
 *
 * dsa_plan_capturable allocates a plan for at most max_rows (<= 8192) rows in
 * at most max_spans (<= 4096) spans whose rows score at most max_scores keys
 * in total (the sum over rows of pos+1), with every span's page_start a
 * multiple of page_start_align (>= 1; a validation constraint only, the
 * kernels take any page_start); the device planner is one CTA that holds
 * the spans and rows in shared memory.  The plan owns its metadata and score/partial
 * scratch (plain cudaMalloc, so a captured graph may keep pointing at them)
 * and starts empty.  dsa_plan_update recomputes it ON THE DEVICE, enqueued
 * on `stream`, from spans in device memory:
 *   num_spans  device int32 scalar, 0 .. max_spans;
 *   spans      device dsa_device_span_t[max_spans] (all max_spans entries are
 *              read; the first num_spans are used);
 *   pages      device int32 page ids; span s uses pages[page_off ..
 *              page_off + num_pages); num_page_ids is the array's length.
 * The rows are the spans' rows in order (row 0 = span 0's first row).  The
 * update makes no allocation, copy or synchronisation, so it and every call
 * that follows with this plan can be captured in a CUDA graph and replayed
 * after the caller rewrites num_spans / spans / pages in place (the plan
 * keeps the `pages` pointer: pass the same array to every update of a
 * captured sequence).
 *
 * With a capturable plan every entry point above takes max_rows rows of
 * per-row input and output (q, w, keys, q_nope, q_pe, selection, out) and
 * treats rows at or after the update's row count as padding: nothing of a
 * padding row is read or written.  Work is launched for the plan's
 * capacity; padded work items exit at once.  The indexer scores every row
 * with the single-row kernel (a host plan groups the rows of a prefill chunk
 * four at a time), so scores can differ from a host plan's in the last bit
 * for chunk rows; decode rows get identical results.  dsa_plan_get_info
 * returns the capacities (num_rows = max_rows, num_scores = max_scores,
 * attend_units = the most units any update can make, needs_selection = 1).
 *
 * A span is invalid when q_len < 1, ctx_start < 0, page_start < 0 or not a
 * multiple of page_start_align, num_pages < 0, page_off < 0, page_off +
 * num_pages > num_page_ids, or num_pages * page_size < page_start +
 * ctx_start + q_len; the update is invalid when num_spans is outside 0 ..
 * max_spans, the rows exceed max_rows or the scores exceed max_scores.
 * Then the plan is left empty (every later call does nothing) and the
 * device error word records it: DSA_ERR_BAD_SPANS at the next dsa_get_error.
 * Page ids themselves are checked where they are used (DSA_ERR_BOUNDS).
 * Host-side errors: DSA_ERR_INVALID_ARG (host-only context, capacities out
 * of range, non-positive alignment, max_scores < max_rows, null pointers, a
 * plan that is not capturable), DSA_ERR_OOM. */
typedef struct dsa_device_span {
  int32_t q_len;
  int32_t ctx_start;
  int32_t page_start;
  int32_t page_off;
  int32_t num_pages;
  int32_t reserved;      /* set to 0 */
} dsa_device_span_t;
enum { DSA_ERR_BAD_SPANS = 9 };
dsa_status dsa_plan_capturable(dsa_ctx_t *ctx, int32_t max_rows, int32_t max_spans, int64_t max_scores,
                               int32_t page_start_align, int32_t cache_pages, dsa_stream_t stream,
                               dsa_plan_t **out);
dsa_status dsa_plan_update(dsa_ctx_t *ctx, dsa_plan_t *plan, const int32_t *num_spans,
                           const dsa_device_span_t *spans, const int32_t *pages, int64_t num_page_ids,
                           dsa_stream_t stream);
/* The counts the last update of a capturable plan computed, copied to the
 * host after synchronising the device: counts[0] rows, [1] indexer items,
 * [2] attention units, [3] split rows, [4] partial slots, [5] 1 when the
 * spans were valid, [6] the key split of the rows, [7] the scored keys
 * (clamped to INT32_MAX).  DSA_ERR_INVALID_ARG for a host plan. */
dsa_status dsa_plan_read_counts(const dsa_plan_t *plan, int32_t counts[8]);

/* Synchronise `stream`, read and clear the context's device error word.
 * Returns DSA_OK, DSA_ERR_BOUNDS, DSA_ERR_TIMEOUT, DSA_ERR_BAD_SPANS or
 * DSA_ERR_CUDA. */
dsa_status dsa_get_error(dsa_ctx_t *ctx, dsa_stream_t stream);

/* ---- Block-sparse MSA -----------------------------------------------------
 * LLMServingSim, "Sparse attention (DSA and block-sparse MSA)", table "Two
 * shapes, three checkpoints", MiniMax-M3 column: each row keeps the top 16
 * blocks of 128 tokens and attends over them with plain GQA; the index cache
 * holds one bf16 vector per token.  The pages give no block-scoring formula;
 * these calls implement the reading: a token's score is the DSA indexer score
 * (dsa_index_scores over the context's index cache and shape), a block's
 * score is the largest score among the positions the row sees, the selection
 * is the causal top-k over blocks (ties to the lower block), and attention
 * covers the positions <= the row's own in the kept blocks.
 *
 * Blocks are counted in request positions: block b of a request holds
 * positions b*block_size .. (b+1)*block_size - 1.  The calls use the context's
 * index format, index shape and page size and a HOST plan (dsa_plan; its topk
 * and MLA fields are not read); capturable plans get DSA_ERR_UNSUPPORTED.
 *
 * dsa_msa_select_blocks: scores as from dsa_index_scores (each row's pos+1
 *   scores at the plan's offsets) -> block_sel (T, topk_blocks) int32: the
 *   kept block ids in ascending order, then -1 (rows that see at most
 *   topk_blocks blocks keep them all).  DSA_ERR_UNSUPPORTED when a row has more
 *   than 16,384 blocks or topk_blocks > 64.
 * dsa_msa_index_select: dsa_index_scores into the context's scratch, then
 *   dsa_msa_select_blocks.
 * dsa_msa_attend: block_sel (T, topk_blocks) int32 (any order, -1 skipped; an
 *   id outside 0 .. pos/block_size sets DSA_ERR_BOUNDS and is skipped);
 *   q (T, q_heads, head_dim) bf16; kv_cache [pages][page_size][2 * kv_heads *
 *   head_dim] bf16 per token: K of kv heads 0..kv_heads-1, then V of the same
 *   heads; query head h reads kv head h / (q_heads / kv_heads);
 *   out (T, q_heads, head_dim) bf16 = softmax((q . k_j) * sm_scale) . v_j over
 *   the kept positions j, fp32 accumulation.  block_size 128 and head_dim 128
 *   with a group of at most 64 query heads, at most 8 kv heads and a page size
 *   that is a multiple of 8 run on the tensor cores
 *   (dsa_msa_attend_on_tensor_cores); other shapes run a CUDA-core kernel.
 * Device pointers, caller-owned.  DSA_ERR_INVALID_ARG for null pointers, a
 * q_heads that is not a multiple of kv_heads or a nonzero reserved field. */
typedef struct dsa_msa_shape {
  int32_t block_size;    /* tokens per block (128 on the pages' MiniMax-M3 row) */
  int32_t topk_blocks;   /* blocks kept per row (16), at most 64 */
  int32_t q_heads;       /* query heads */
  int32_t kv_heads;      /* key/value heads (GQA groups) */
  int32_t head_dim;      /* per-head width of q, K and V */
  int32_t reserved;      /* set to 0 */
} dsa_msa_shape_t;
dsa_status dsa_msa_select_blocks(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape,
                                 const float *scores, int32_t *block_sel, dsa_stream_t stream);
dsa_status dsa_msa_index_select(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape, const void *q,
                                const float *w, const void *index_cache, int32_t *block_sel, dsa_stream_t stream);
dsa_status dsa_msa_attend(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape,
                          const int32_t *block_sel, const void *q, const void *kv_cache, float sm_scale, void *out,
                          dsa_stream_t stream);
/* 1 when dsa_msa_attend runs this shape on the tensor cores, else 0 (host-side query). */
int dsa_msa_attend_on_tensor_cores(const dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape);

/* Drive the pipeline's bounded wait to its limit, for testing the failure
 * path (mstar IndexKeyStore.history: a failure is reported to the caller, not
 * fatal).  One CTA takes tensor memory, waits on an mbarrier that nothing
 * arrives on with a limit of limit_ns nanoseconds (the kernels' own limit is
 * one second), then waits on it again, frees the tensor memory and exits.
 * result: DEVICE int64[5], caller-owned: [0] 1 if the first wait succeeded,
 * [1] its duration in ns, [2] 1 if the second wait succeeded, [3] its
 * duration in ns, [4] the CTA's abort flag at the end.  Expected: the first
 * wait gives up after about limit_ns and sets DSA_ERR_TIMEOUT in the error
 * word (read by dsa_get_error), the abort flag it raises ends the second wait
 * at once, and the context stays usable.  DSA_ERR_INVALID_ARG for a
 * host-only context, a null result or limit_ns outside 1 .. 1e9. */
dsa_status dsa_selftest_wait_timeout(dsa_ctx_t *ctx, uint64_t limit_ns, int64_t *result, dsa_stream_t stream);

/* Number of kernels the last compute call on this context launched (for
 * accounting; host-side counter, no synchronisation). */
int32_t dsa_last_launch_count(const dsa_ctx_t *ctx);

const char *dsa_status_str(dsa_status s);

/* Name and text of the CUDA error behind the context's last DSA_ERR_CUDA
 * ("" when there was none); owned by the context. */
const char *dsa_last_cuda_error(const dsa_ctx_t *ctx);

#ifdef __cplusplus
}
#endif
#endif /* DSA_GB300_DSA_H_ */
