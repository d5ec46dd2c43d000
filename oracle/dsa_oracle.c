/*
 * dsa_oracle.c -- plain, slow CPU oracle for DeepSeek Sparse Attention (DSA)
 * over a paged MLA cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py may build, load or call this file.  It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * loads it: the library fails loudly when its CUDA build is missing.
 *
 * Source of the method: the mstar page "mstar.engine.resources.dsa.manager"
 * (module summary; index_topk; select_topk_causal; DSAManager.attend; DSASpan;
 * DSAPlan), the Tenstorrent page "ttnn.transformer.sparse_sdpa" (packed 656-byte
 * latent row, attention sink, sentinel tail) and the LLMServingSim page "Sparse
 * attention (DSA and block-sparse MSA)" (132-byte fp8 index row).
 *
 * Everything is computed the direct way, in double precision:
 *   score  s[r, j] = sum_h w[r,h] * relu(q[r,h] . k[j])      for j = 0 .. pos(r)
 *          accumulated in double and rounded once to fp32
 *   select the top `topk` positions of s[r, 0..pos(r)], ties to the lower position,
 *          -1 padded when the row sees fewer than topk keys
 *   attend o[r,h] = sum_j e^{l_j - m} c_j / (sum_j e^{l_j - m} [+ e^{sink_h - m}])
 *          with l_j = (q_nope[r,h] . c_j + q_pe[r,h] . kpe_j) * sm_scale over the
 *          selected j, m the maximum of the l_j (and of the sink)
 *
 * Block-sparse MSA (LLMServingSim, the MiniMax-M3 column of "Two shapes,
 * three checkpoints"): block scores are the largest token score of each block
 * of block_size positions the row sees, the top topk_blocks blocks are kept
 * (the same causal top-k, over blocks), and GQA attention runs over the
 * visible positions of the kept blocks.
 *
 * Paged layout (DSASpan / DSAPlan): a row at request-local position p finds
 * token j at slot = page_start + j of its span's page list,
 * physical row = pages[slot / page_size] * page_size + slot % page_size.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC (oracle/build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_SHORT_HISTORY = 2, OR_BAD_PAGE = 3, OR_BAD_SELECTION = 4, OR_NOMEM = 5 };
enum { FMT_BF16 = 0, FMT_FP8 = 1 };

/* ------------------------------------------------------------------------ */
/* number formats                                                            */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double f32_at(const uint8_t *p) {
  float f;
  memcpy(&f, p, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn": finite, no infinities):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * exponent field 0      -> subnormal, (m / 8) * 2^(1 - 7)
 * exponent field 1..15  -> normal, (1 + m / 8) * 2^(e - 7)
 * S.1111.111            -> NaN (the only non-finite encoding). */
double oracle_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 0xF, m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* rows and pages                                                            */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t T;                 /* rows this step */
  int32_t page_size;
  int32_t num_pages;         /* pages in the cache */
  const int64_t *pos;        /* [T] request-local position of each row */
  const int64_t *page_off;   /* [T] offset of the row's page list in `pages` */
  const int64_t *npages;     /* [T] length of the row's page list */
  const int64_t *page_start; /* [T] slot of token 0 within the page list */
  const int32_t *pages;      /* concatenated page lists */
} oracle_rows;

/* Physical cache row of token j of row r, or -1 (with *err set) when the
 * span's pages do not reach it or a page id is outside the cache. */
static int64_t phys_row(const oracle_rows *R, int64_t r, int64_t j, int *err) {
  int64_t slot = R->page_start[r] + j;
  int64_t pi = slot / R->page_size;
  if (j < 0 || pi >= R->npages[r]) { *err = OR_SHORT_HISTORY; return -1; }
  int64_t page = R->pages[R->page_off[r] + pi];
  if (page < 0 || page >= R->num_pages) { *err = OR_BAD_PAGE; return -1; }
  return page * R->page_size + slot % R->page_size;
}

/* ------------------------------------------------------------------------ */
/* store_keys: each row's index key goes to the slot of its own position     */
/* ------------------------------------------------------------------------ */

/* keys: T rows in cache format (bf16: 2*index_dim bytes; fp8: index_dim codes
 * followed by a 4-byte fp32 scale).  bf16 cache: [pages][page_size][index_dim].
 * fp8 cache, page-blocked: each page holds page_size*index_dim codes, then
 * page_size fp32 scales. */
int oracle_store_keys(const oracle_rows *R, int index_fmt, int index_dim, const uint8_t *keys, uint8_t *cache) {
  int err = OR_OK;
  for (int64_t r = 0; r < R->T; r++) {
    int64_t row = phys_row(R, r, R->pos[r], &err);
    if (row < 0) return err;
    int64_t page = row / R->page_size, s = row % R->page_size;
    if (index_fmt == FMT_BF16) {
      memcpy(cache + row * 2 * index_dim, keys + r * 2 * index_dim, 2 * (size_t)index_dim);
    } else {
      size_t page_bytes = (size_t)R->page_size * (index_dim + 4);
      uint8_t *base = cache + page * page_bytes;
      const uint8_t *src = keys + r * (index_dim + 4);
      memcpy(base + s * index_dim, src, (size_t)index_dim);
      memcpy(base + (size_t)R->page_size * index_dim + s * 4, src + index_dim, 4);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* quantize-on-store (an extension past the pages: they store rows that are  */
/* already in cache format)                                                  */
/* ------------------------------------------------------------------------ */

/* fp32 -> E4M3 code, round to nearest with ties to even.  The representable
 * magnitudes of a binade [2^E, 2^(E+1)) are multiples of 2^(E-3); below 2^-6
 * (the subnormal range) they are multiples of 2^-9.  Magnitudes at or above
 * the largest finite value, 448, encode as 448 (the quantiser scales groups so
 * that nothing exceeds it).  The sign is the sign bit of the input (-0 gives
 * code 0x80). */
uint8_t oracle_e4m3_encode(float xf) {
  const double x = (double)xf;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs(x);
  if (isnan(a)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  int E = (a < ldexp(1.0, -6)) ? -6 : ilogb(a);
  const double steps = nearbyint(a / ldexp(1.0, E - 3)); /* exact quotient, rounded to even */
  int k = (int)steps;
  if (E == -6 && k < 8) return sign | (uint8_t)k;        /* subnormal (or zero) */
  if (k == 16) {                                          /* rounded up into the next binade */
    E += 1;
    k = 8;
  }
  return sign | (uint8_t)(((E + 7) << 3) | (k - 8));
}

/* One group: scale = amax / 448 in fp32 (1 when the group is all zeros),
 * codes = E4M3(x / scale) with the quotient rounded to fp32 first. */
static float quantize_group(const uint16_t *src, int n, uint8_t *codes) {
  float amax = 0.0f;
  for (int i = 0; i < n; i++) {
    float v = (float)bf16_value(src[i]);
    if (fabsf(v) > amax) amax = fabsf(v);
  }
  const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int i = 0; i < n; i++) {
    const float q = (float)bf16_value(src[i]) / scale;
    codes[i] = oracle_e4m3_encode(q);
  }
  return scale;
}

/* keys: T rows of index_dim bf16 -> the page-blocked 132-byte layout at the
 * slot of each row's own position (one scale per row). */
int oracle_quantize_store_keys(const oracle_rows *R, int index_dim, const uint16_t *keys, uint8_t *cache) {
  int err = OR_OK;
  uint8_t *codes = (uint8_t *)malloc((size_t)index_dim);
  if (!codes) return OR_NOMEM;
  for (int64_t r = 0; r < R->T; r++) {
    int64_t row = phys_row(R, r, R->pos[r], &err);
    if (row < 0) {
      free(codes);
      return err;
    }
    int64_t page = row / R->page_size, s = row % R->page_size;
    uint8_t *base = cache + page * (size_t)R->page_size * (index_dim + 4);
    const float scale = quantize_group(keys + r * index_dim, index_dim, codes);
    memcpy(base + s * index_dim, codes, (size_t)index_dim);
    memcpy(base + (size_t)R->page_size * index_dim + s * 4, &scale, 4);
  }
  free(codes);
  return OR_OK;
}

/* latents: T rows of (L + Rd) bf16 -> 656-byte rows [L codes | L/128 fp32
 * scales, one per group of 128 | Rd bf16 rope, copied] at each row's slot. */
int oracle_quantize_store_latents(const oracle_rows *R, int L, int Rd, const uint16_t *lat, uint8_t *cache) {
  int err = OR_OK;
  const size_t row_bytes = (size_t)L + 4 * (size_t)(L / 128) + 2 * (size_t)Rd;
  for (int64_t r = 0; r < R->T; r++) {
    int64_t row = phys_row(R, r, R->pos[r], &err);
    if (row < 0) return err;
    uint8_t *dst = cache + row * row_bytes;
    const uint16_t *src = lat + r * (L + Rd);
    for (int g = 0; g < L / 128; g++) {
      const float scale = quantize_group(src + 128 * g, 128, dst + 128 * g);
      memcpy(dst + L + 4 * g, &scale, 4);
    }
    memcpy(dst + L + 4 * (L / 128), src + L, 2 * (size_t)Rd);
  }
  return OR_OK;
}

/* The index key of token j of row r, as doubles. */
static int load_index_key(const oracle_rows *R, int64_t r, int64_t j, int index_fmt, int index_dim,
                          const uint8_t *cache, double *k) {
  int err = OR_OK;
  int64_t row = phys_row(R, r, j, &err);
  if (row < 0) return err;
  if (index_fmt == FMT_BF16) {
    const uint16_t *src = (const uint16_t *)cache + row * index_dim;
    for (int d = 0; d < index_dim; d++) k[d] = bf16_value(src[d]);
  } else {
    int64_t page = row / R->page_size, s = row % R->page_size;
    const uint8_t *base = cache + page * (size_t)R->page_size * (index_dim + 4);
    double scale = f32_at(base + (size_t)R->page_size * index_dim + s * 4);
    for (int d = 0; d < index_dim; d++) k[d] = oracle_e4m3_value(base[s * index_dim + d]) * scale;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* indexer score                                                             */
/* ------------------------------------------------------------------------ */

/* q: [T][index_heads][index_dim] bf16 (q_codes == NULL), or e4m3 codes
 * q_codes [T][index_heads][index_dim] with one fp32 scale per (row, head)
 * q_scale [T][index_heads]: q = e4m3(code) * scale.  w: [T][index_heads] fp32.
 * scores: row r's pos(r)+1 scores start at score_off[r]. */
static int index_scores(const oracle_rows *R, int index_heads, int index_dim, int index_fmt,
                        const uint16_t *q, const uint8_t *q_codes, const float *q_scale, const float *w,
                        const uint8_t *cache, const int64_t *score_off, float *scores) {
  int status = OR_OK;
#pragma omp parallel
  {
    double *k = (double *)malloc(sizeof(double) * index_dim);
    double *qd = (double *)malloc(sizeof(double) * index_heads * index_dim);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < R->T; r++) {
      if (!k || !qd) { status = OR_NOMEM; continue; }
      for (int64_t i = 0; i < (int64_t)index_heads * index_dim; i++) {
        const int64_t at = r * index_heads * index_dim + i;
        qd[i] = q_codes ? oracle_e4m3_value(q_codes[at]) * (double)q_scale[r * index_heads + i / index_dim]
                        : bf16_value(q[at]);
      }
      for (int64_t j = 0; j <= R->pos[r]; j++) {
        int e = load_index_key(R, r, j, index_fmt, index_dim, cache, k);
        if (e != OR_OK) { status = e; break; }
        double s = 0.0;
        for (int h = 0; h < index_heads; h++) {
          double dot = 0.0;
          for (int d = 0; d < index_dim; d++) dot += qd[h * index_dim + d] * k[d];
          double relu = dot > 0.0 ? dot : 0.0;
          s += (double)w[r * index_heads + h] * relu;
        }
        scores[score_off[r] + j] = (float)s;
      }
    }
    free(k);
    free(qd);
  }
  return status;
}

int oracle_index_scores(const oracle_rows *R, int index_heads, int index_dim, int index_fmt,
                        const uint16_t *q, const float *w, const uint8_t *cache,
                        const int64_t *score_off, float *scores) {
  return index_scores(R, index_heads, index_dim, index_fmt, q, NULL, NULL, w, cache, score_off, scores);
}

/* The same score with an fp8 query (e4m3 codes x one fp32 scale per head). */
int oracle_index_scores_fp8q(const oracle_rows *R, int index_heads, int index_dim, int index_fmt,
                             const uint8_t *q_codes, const float *q_scale, const float *w, const uint8_t *cache,
                             const int64_t *score_off, float *scores) {
  return index_scores(R, index_heads, index_dim, index_fmt, NULL, q_codes, q_scale, w, cache, score_off, scores);
}

/* n_rows rows of `width` bf16 -> e4m3 codes and one scale per row, by the
 * quantize-on-store rule (fp8 query). */
int oracle_quantize_rows(int64_t n_rows, int width, const uint16_t *src, uint8_t *codes, float *scales) {
  for (int64_t r = 0; r < n_rows; r++) scales[r] = quantize_group(src + r * width, width, codes + r * width);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* causal top-k with ties to the lower position                              */
/* ------------------------------------------------------------------------ */

/* true when position a ranks before position b */
static int ranks_before(const float *s, int64_t a, int64_t b) {
  if (s[a] != s[b]) return s[a] > s[b];
  return a < b;
}

/* stable merge sort of positions by (score descending, position ascending) */
static void sort_positions(const float *s, int64_t *idx, int64_t *tmp, int64_t n) {
  for (int64_t width = 1; width < n; width *= 2) {
    for (int64_t lo = 0; lo < n; lo += 2 * width) {
      int64_t mid = lo + width < n ? lo + width : n;
      int64_t hi = lo + 2 * width < n ? lo + 2 * width : n;
      int64_t a = lo, b = mid, o = lo;
      while (a < mid && b < hi) tmp[o++] = ranks_before(s, idx[b], idx[a]) ? idx[b++] : idx[a++];
      while (a < mid) tmp[o++] = idx[a++];
      while (b < hi) tmp[o++] = idx[b++];
    }
    memcpy(idx, tmp, sizeof(int64_t) * n);
  }
}

/* sel: [T][topk] int32, valid positions first in rank order, then -1. */
int oracle_topk(int64_t T, int topk, const int64_t *pos, const float *scores, const int64_t *score_off,
                int32_t *sel) {
  int status = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < T; r++) {
    int64_t n = pos[r] + 1;
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * n);
    int64_t *tmp = (int64_t *)malloc(sizeof(int64_t) * n);
    if (!idx || !tmp) { status = OR_NOMEM; free(idx); free(tmp); continue; }
    for (int64_t j = 0; j < n; j++) idx[j] = j;
    sort_positions(scores + score_off[r], idx, tmp, n);
    for (int64_t i = 0; i < topk; i++) sel[r * topk + i] = i < n ? (int32_t)idx[i] : -1;
    free(idx);
    free(tmp);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* absorbed MLA over the selected latents                                    */
/* ------------------------------------------------------------------------ */

/* Latent row of token j: c[0..L) and kpe[0..R) as doubles.
 * bf16 row: (L+R) bf16.  fp8 row (656 B at L=512, R=64): L e4m3 codes, L/128
 * fp32 scales (scale i covers codes 128i .. 128i+127), R bf16 rope values. */
static int load_latent(const oracle_rows *Rw, int64_t r, int64_t j, int latent_fmt, int L, int Rd,
                       const uint8_t *cache, double *c, double *kpe) {
  int err = OR_OK;
  int64_t row = phys_row(Rw, r, j, &err);
  if (row < 0) return err;
  if (latent_fmt == FMT_BF16) {
    const uint16_t *src = (const uint16_t *)cache + row * (L + Rd);
    for (int i = 0; i < L; i++) c[i] = bf16_value(src[i]);
    for (int i = 0; i < Rd; i++) kpe[i] = bf16_value(src[L + i]);
  } else {
    size_t row_bytes = (size_t)L + 4 * (L / 128) + 2 * (size_t)Rd;
    const uint8_t *src = cache + row * row_bytes;
    for (int i = 0; i < L; i++) c[i] = oracle_e4m3_value(src[i]) * f32_at(src + L + 4 * (i / 128));
    const uint8_t *rope = src + L + 4 * (L / 128);
    for (int i = 0; i < Rd; i++) {
      uint16_t b;
      memcpy(&b, rope + 2 * i, 2);
      kpe[i] = bf16_value(b);
    }
  }
  return OR_OK;
}

/* sel: [T][topk]; entries -1 are skipped; any other entry must lie in 0..pos(r).
 * q_nope [T][H][L], q_pe [T][H][R] bf16; sink [H] fp32 or NULL; out [T][H][L]. */
int oracle_attend(const oracle_rows *Rw, int H, int L, int Rd, int topk, int latent_fmt,
                  const int32_t *sel, const uint16_t *q_nope, const uint16_t *q_pe, const uint8_t *cache,
                  const float *sink, double sm_scale, double *out) {
  int status = OR_OK;
#pragma omp parallel
  {
    double *c = (double *)malloc(sizeof(double) * (size_t)topk * L);
    double *kpe = (double *)malloc(sizeof(double) * (size_t)topk * (Rd > 0 ? Rd : 1));
    double *logit = (double *)malloc(sizeof(double) * topk);
    double *qn = (double *)malloc(sizeof(double) * L);
    double *qp = (double *)malloc(sizeof(double) * (Rd > 0 ? Rd : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < Rw->T; r++) {
      if (!c || !kpe || !logit || !qn || !qp) { status = OR_NOMEM; continue; }
      int n = 0;
      int bad = OR_OK;
      for (int i = 0; i < topk; i++) {
        int64_t j = sel[r * topk + i];
        if (j == -1) continue;
        if (j < 0 || j > Rw->pos[r]) { bad = OR_BAD_SELECTION; break; }
        int e = load_latent(Rw, r, j, latent_fmt, L, Rd, cache, c + (size_t)n * L, kpe + (size_t)n * Rd);
        if (e != OR_OK) { bad = e; break; }
        n++;
      }
      if (bad != OR_OK) { status = bad; continue; }
      for (int h = 0; h < H; h++) {
        const uint16_t *qnr = q_nope + ((size_t)r * H + h) * L;
        const uint16_t *qpr = q_pe + ((size_t)r * H + h) * Rd;
        for (int i = 0; i < L; i++) qn[i] = bf16_value(qnr[i]);
        for (int i = 0; i < Rd; i++) qp[i] = bf16_value(qpr[i]);
        double m = -INFINITY;
        for (int t = 0; t < n; t++) {
          double a = 0.0, b = 0.0;
          for (int i = 0; i < L; i++) a += qn[i] * c[(size_t)t * L + i];
          for (int i = 0; i < Rd; i++) b += qp[i] * kpe[(size_t)t * Rd + i];
          logit[t] = (a + b) * sm_scale;
          if (logit[t] > m) m = logit[t];
        }
        if (sink && (double)sink[h] > m) m = (double)sink[h];
        double den = sink ? exp((double)sink[h] - m) : 0.0;
        for (int t = 0; t < n; t++) den += exp(logit[t] - m);
        double *o = out + ((size_t)r * H + h) * L;
        for (int i = 0; i < L; i++) o[i] = 0.0;
        if (n == 0) continue; /* nothing selected: the output row is zero */
        for (int t = 0; t < n; t++) {
          double p = exp(logit[t] - m) / den;
          for (int i = 0; i < L; i++) o[i] += p * c[(size_t)t * L + i];
        }
      }
    }
    free(c);
    free(kpe);
    free(logit);
    free(qn);
    free(qp);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* block-sparse MSA (LLMServingSim, "Sparse attention (DSA and block-sparse  */
/* MSA)", table "Two shapes, three checkpoints", MiniMax-M3 column: the top  */
/* 16 blocks of 128 tokens, over plain GQA, one bf16 index vector per token) */
/* ------------------------------------------------------------------------ */

/* Block scores.  Block b of row r holds positions b*block_size ..
 * (b+1)*block_size - 1; its score is the largest token score (the DSA indexer
 * score above) among the positions the row sees, 0 .. pos(r).  Row r has
 * pos(r)/block_size + 1 blocks, its scores starting at block_off[r].  The
 * selection is then the causal top-k above over these block scores (ties to
 * the lower block). */
int oracle_msa_block_scores(int64_t T, int block_size, const int64_t *pos, const float *scores,
                            const int64_t *score_off, const int64_t *block_off, float *block_scores) {
  if (block_size <= 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < T; r++) {
    int64_t nblk = pos[r] / block_size + 1;
    for (int64_t b = 0; b < nblk; b++) {
      int64_t j0 = b * block_size, j1 = j0 + block_size - 1;
      if (j1 > pos[r]) j1 = pos[r];
      float m = scores[score_off[r] + j0];
      for (int64_t j = j0 + 1; j <= j1; j++)
        if (scores[score_off[r] + j] > m) m = scores[score_off[r] + j];
      block_scores[block_off[r] + b] = m;
    }
  }
  return OR_OK;
}

/* GQA attention over the tokens of the selected blocks.
 * kv cache: one row per token, [K of kv heads 0..kv_heads-1 | V of the same
 * heads], head_dim bf16 each (2 * kv_heads * head_dim * 2 bytes), in the
 * paged layout of oracle_rows.  sel: [T][topk_blocks] block ids, -1 skipped;
 * any other id must lie in 0 .. pos(r)/block_size.  q: [T][q_heads][head_dim]
 * bf16; query head h reads kv head h / (q_heads / kv_heads).
 * out[r][h] = sum_j e^{l_j - m} v_j / sum_j e^{l_j - m}, l_j = (q . k_j) * sm_scale,
 * over the positions j <= pos(r) of the selected blocks, in double. */
int oracle_msa_attend(const oracle_rows *R, int q_heads, int kv_heads, int head_dim, int block_size,
                      int topk_blocks, const int32_t *sel, const uint16_t *q, const uint8_t *kv, double sm_scale,
                      double *out) {
  if (kv_heads <= 0 || q_heads % kv_heads != 0 || block_size <= 0 || topk_blocks <= 0) return OR_BAD_ARG;
  const int group = q_heads / kv_heads;
  const size_t row_elems = 2 * (size_t)kv_heads * head_dim;
  const int64_t max_tokens = (int64_t)topk_blocks * block_size;
  int status = OR_OK;
#pragma omp parallel
  {
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * max_tokens);
    double *logit = (double *)malloc(sizeof(double) * max_tokens);
    double *qd = (double *)malloc(sizeof(double) * head_dim);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < R->T; r++) {
      if (!rows || !logit || !qd) { status = OR_NOMEM; continue; }
      int64_t n = 0;
      int bad = OR_OK;
      for (int i = 0; i < topk_blocks && bad == OR_OK; i++) {
        int64_t b = sel[r * topk_blocks + i];
        if (b == -1) continue;
        if (b < 0 || b > R->pos[r] / block_size) { bad = OR_BAD_SELECTION; break; }
        for (int64_t j = b * block_size; j < (b + 1) * block_size && j <= R->pos[r]; j++) {
          int e = OR_OK;
          int64_t row = phys_row(R, r, j, &e);
          if (row < 0) { bad = e; break; }
          rows[n++] = row;
        }
      }
      if (bad != OR_OK) { status = bad; continue; }
      for (int h = 0; h < q_heads; h++) {
        const int g = h / group;
        const uint16_t *qr = q + ((size_t)r * q_heads + h) * head_dim;
        for (int d = 0; d < head_dim; d++) qd[d] = bf16_value(qr[d]);
        double m = -INFINITY;
        for (int64_t t = 0; t < n; t++) {
          const uint16_t *k = (const uint16_t *)kv + rows[t] * row_elems + (size_t)g * head_dim;
          double a = 0.0;
          for (int d = 0; d < head_dim; d++) a += qd[d] * bf16_value(k[d]);
          logit[t] = a * sm_scale;
          if (logit[t] > m) m = logit[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < n; t++) den += exp(logit[t] - m);
        double *o = out + ((size_t)r * q_heads + h) * head_dim;
        for (int d = 0; d < head_dim; d++) o[d] = 0.0;
        for (int64_t t = 0; t < n; t++) {
          const uint16_t *v = (const uint16_t *)kv + rows[t] * row_elems + ((size_t)kv_heads + g) * head_dim;
          double p = exp(logit[t] - m) / den;
          for (int d = 0; d < head_dim; d++) o[d] += p * bf16_value(v[d]);
        }
      }
    }
    free(rows);
    free(logit);
    free(qd);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
