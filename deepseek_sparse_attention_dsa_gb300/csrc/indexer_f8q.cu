// indexer_f8q.cu -- the indexer score with an fp8 query over the fp8 index
// cache, e4m3 x e4m3 on the tensor cores (tcgen05.mma kind::f8f6f4).
//
//   q[r,h,d] = e4m3(qc[r,h,d]) * qs[r,h],   k[j,d] = e4m3(kc[j,d]) * ks[j]
//   s[r,j]   = sum_h w[r,h] * relu(q[r,h] . k[j])
//            = |ks[j]| * sum_h (w[r,h] |qs[r,h]|) * relu(sgn(ks[j] qs[r,h]) * (qc[r,h] . kc[j]))
//
// The index row is the 132-byte fp8 key (LLMServingSim, "What the KV cache
// actually holds": 128 e4m3 codes + one fp32 scale, page-blocked), and an
// e4m3 query is the sparse_sdpa option (ttnn.transformer.sparse_sdpa, q
// "bf16 or fp8_e4m3") carried over to the indexer's query with one scale per
// (row, head), written by dsa_quantize_q with the quantize-on-store rule.
//
// The staged key codes ARE the A operand: M = 128 keys, K = 128 codes in one
// 128-byte swizzled row per key (four K = 32 steps), N = G rows x 64 heads;
// nothing is converted.  The epilogue applies the key scale staged beside the
// codes, so a stage is released by the MMA commit (codes read) and by the
// epilogue (scale read).
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread) and TMEM owner, warps 2-5 epilogue (thread = key = TMEM lane).
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {


__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int G>
struct F8qTraits {
  static constexpr int HI = 64, DI = 128;
  static constexpr int N = G * HI;
  // epilogue warps: two per TMEM lane quadrant for row groups, each taking
  // half of the group's rows (the MMAs of a group tile are half the
  // epilogue's work); one per quadrant for single rows
  static constexpr int EPI = (G == 4) ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI;
  static constexpr int RPH = G / (EPI / 4);              // rows per epilogue warp
  static constexpr int CODE_BYTES = 128 * 128;           // one tile of key codes, 128-byte swizzle
  // staged scales: a TMA destination must be 128-byte aligned, so box b of a
  // tile lands at b * max(128, 4 * BH) bytes (up to 16 boxes of 8 keys)
  static constexpr int SC_BYTES = 2048;
  static constexpr int STAGE = CODE_BYTES + SC_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int QBUF = (G == 1) ? 2 : 1;
  static constexpr int Q_BYTES = N * 128;                // query codes, 128-byte swizzle
  static constexpr int TMEM_COLS = (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  static constexpr uint32_t IDESC = mma_idesc(128, N, 0u, false, false);   // kind::f8f6f4: format 0 = e4m3
  static constexpr int OFF_ST = 0;
  static constexpr int OFF_Q = OFF_ST + STAGES * STAGE;
  static constexpr int OFF_W = OFF_Q + QBUF * Q_BYTES;   // [G*HI] w |qs|, then [G*HI] sgn(qs)
  static constexpr int OFF_BAR = OFF_W + 2 * G * HI * 4;
  static constexpr int NBAR = 2 * STAGES + 2 * QBUF + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(STAGE % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(N <= 256, "UMMA N");
};

struct F8qParams {
  CUtensorMap tm_codes;     // key codes as [pages][P][128] uint8, box {128, BH, 1}, 128-byte swizzle
  CUtensorMap tm_scales;    // key scales as [pages][P] fp32 (page stride P*132 bytes), box {BH, 1}
  CUtensorMap tm_q;         // query codes as [T*Hi, 128] uint8, box {128, N}, 128-byte swizzle
  const float *q_scale;     // [T, Hi]
  const float *w;           // [T, Hi]
  const IdxGroup *groups;
  const IdxItem *items;
  const int32_t *cta_begin;
  const int32_t *pages;
  const int64_t *row_score_off;
  float *scores;
  int *err;
  int P, BH, num_pages;
};

template <int G>
__global__ void __launch_bounds__(F8qTraits<G>::THREADS, 1) index_f8q_kernel(const __grid_constant__ F8qParams p) {
  using C = F8qTraits<G>;
  constexpr int HI = C::HI;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto sfull = [&](int s) { return bar0 + 8u * s; };
  auto sempty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto qfull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto qempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + C::QBUF + b); };
  auto afull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * C::QBUF + b); };
  auto aempty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * C::QBUF + 2 + b); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *wsm = reinterpret_cast<float *>(smem + C::OFF_W);
  float *ssm = wsm + G * HI;

  const int warp = threadIdx.x / 32;
  const int lane = lane_id();
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];
  const int sc_stride = max(32, p.BH);   // floats between the staged scale boxes of a tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(sfull(s), 1);
      mbar_init(sempty(s), 1 + C::EPI);   // the MMA commit and one lane of each epilogue warp
    }
    for (int b = 0; b < C::QBUF; ++b) {
      mbar_init(qfull(b), 1);
      mbar_init(qempty(b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), C::EPI);
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
    int st = 0;
    uint32_t ph = 0;
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
            tma_load_2d(sbase + C::OFF_Q + qb * C::Q_BYTES, &p.tm_q, 0, g.row0 * HI, qfull(qb));
          }
        }
        if (__shfl_sync(0xffffffffu, qok ? 1 : 0, 0) == 0) break;
      }
      const int nrows_total = g.lead + g.pos0 + g.nrows;  // tile rows: lead rows, then keys 0 .. pos0+nrows-1
      // raw page id of this lane's box of tile t (kNoBox: no box for this lane;
      // -1: past the request's pages), looked up four tiles ahead of its issue
      // and checked when the tile is issued
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
      // four lookups in flight: the loop is unrolled by four so that every
      // looked-up page id stays in its own register until its tile is issued
      int lp[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) lp[u] = box_page(item.tile0 + u);
      bool stop = false;
      for (int t0 = item.tile0; t0 < item.tile1 && !stop; t0 += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + u;
          if (t >= item.tile1) break;
          int myslot;
          const int mypage = box_at(t, lp[u], myslot);
          lp[u] = box_page(t + 4);
          const uint32_t valid = __ballot_sync(0xffffffffu, mypage >= 0);
          bool ok = true;
          if (lane == 0) ok = mbar_wait(sempty(st), ph ^ 1, abort_flag, p.err);
          if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) {
            stop = true;
            break;
          }
          const uint32_t bytes = __popc(valid) * p.BH * (128 + 4);
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(sfull(st), bytes);
            else mbar_arrive(sfull(st));
          }
          // every box from the lane that looked it up (lane b holds box b):
          // the tile's loads go out as one warp instruction
          const uint32_t stage = sbase + C::OFF_ST + st * C::STAGE;
          if (mypage >= 0) {
            tma_load_3d(stage + lane * p.BH * 128, &p.tm_codes, 0, myslot, mypage, sfull(st));
            tma_load_2d(stage + C::CODE_BYTES + lane * sc_stride * 4, &p.tm_scales, myslot, mypage, sfull(st));
          }
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
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
          if (!mbar_wait(sfull(st), ph, abort_flag, p.err)) { ok = false; break; }
          if (!mbar_wait(aempty(acc), aphase ^ 1, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = sbase + C::OFF_ST + st * C::STAGE;
          const uint32_t d = tmem_base + acc * C::N;
#pragma unroll
          for (int k = 0; k < 4; ++k)   // K = 32 codes (32 bytes) per step
            mma_f8_ss(d, smem_desc(kaddr + k * 32, 16, 1024, kSwizzle128),
                      smem_desc(qaddr + k * 32, 16, 1024, kSwizzle128), C::IDESC, k != 0 ? 1u : 0u);
          mma_commit(sempty(st));   // the codes are read; the epilogue still reads the scales
          mma_commit(afull(acc));
          if (++st == C::STAGES) {
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;            // which of the group's rows this warp takes
    const int m = quad * 32 + lane;
    int acc = 0, st = 0;
    uint32_t aphase = 0, ph = 0;
    int cur_group = -1;
    int64_t soff[G];
    int nrows = 0, pos0 = 0, lead = 0;
    bool signed_q = false;   // some head of the group has a negative query scale
    for (int it = it0; it < it1 && !*abort_flag; ++it) {
      const IdxItem item = p.items[it];
      if (item.group != cur_group) {
        cur_group = item.group;
        const IdxGroup g = p.groups[item.group];
        nrows = g.nrows;
        pos0 = g.pos0;
        lead = g.lead;
        named_bar_sync(1, 32 * C::EPI);
        bool neg = false;
        for (int i = et; i < G * HI; i += 32 * C::EPI) {
          float wv = 0.f, qs = 0.f;
          if (i < nrows * HI) {
            wv = p.w[static_cast<int64_t>(g.row0) * HI + i];
            qs = p.q_scale[static_cast<int64_t>(g.row0) * HI + i];
          }
          wsm[i] = wv * fabsf(qs);
          ssm[i] = qs < 0.f ? -1.f : 1.f;
          neg = neg || qs < 0.f;
        }
#pragma unroll
        for (int gg = 0; gg < G; ++gg) soff[gg] = gg < nrows ? p.row_score_off[g.row0 + gg] : 0;
        signed_q = named_bar_any(1, 32 * C::EPI, neg);   // also the barrier after the writes
      }
      bool ok = true;
      for (int t = item.tile0; t < item.tile1; ++t) {
        // waits are made warp-uniform: each warp arrives once, by lane 0
        if (!__all_sync(0xffffffffu, mbar_wait(afull(acc), aphase, abort_flag, p.err))) { ok = false; break; }
        tc_fence_after();
        // the key scales of this tile's stage (the stage filled phase `ph`;
        // it is not refilled before this warp releases it below)
        if (!__all_sync(0xffffffffu, mbar_wait(sfull(st), ph, abort_flag, p.err))) { ok = false; break; }
        const float ks = reinterpret_cast<const float *>(smem + C::OFF_ST + st * C::STAGE + C::CODE_BYTES)
            [(m / p.BH) * sc_stride + m % p.BH];
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty(st));
        if (++st == C::STAGES) {
          st = 0;
          ph ^= 1;
        }
        const float mag = fabsf(ks);
        const float ksign = ks < 0.f ? -1.f : 1.f;
        // the quantiser's scales are >= 0: then relu needs no sign at all
        const bool unsigned_tile = __all_sync(0xffffffffu, ks >= 0.f) && !signed_q;
        const int key = t * 128 + m - lead;   // < 0: a slot before the span's token 0
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::N;
#pragma unroll
        for (int j = 0; j < C::RPH; ++j) {
          const int gg = half * C::RPH + j;
          if (gg < nrows) {
            float v[HI];
#pragma unroll
            for (int h0 = 0; h0 < HI; h0 += 16)
              tmem_ld16(tbase + gg * HI + h0, *reinterpret_cast<float(*)[16]>(v + h0));
            tmem_ld_wait();
            const float4 *w4 = reinterpret_cast<const float4 *>(wsm + gg * HI);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            if (unsigned_tile) {
#pragma unroll
              for (int h = 0; h < HI; h += 4) {
                const float4 ww = w4[h / 4];
                a0 = fmaf(ww.x, fmaxf(v[h], 0.f), a0);
                a1 = fmaf(ww.y, fmaxf(v[h + 1], 0.f), a1);
                a2 = fmaf(ww.z, fmaxf(v[h + 2], 0.f), a2);
                a3 = fmaf(ww.w, fmaxf(v[h + 3], 0.f), a3);
              }
            } else if (!signed_q) {   // one sign per key
#pragma unroll
              for (int h = 0; h < HI; h += 4) {
                const float4 ww = w4[h / 4];
                a0 = fmaf(ww.x, fmaxf(ksign * v[h], 0.f), a0);
                a1 = fmaf(ww.y, fmaxf(ksign * v[h + 1], 0.f), a1);
                a2 = fmaf(ww.z, fmaxf(ksign * v[h + 2], 0.f), a2);
                a3 = fmaf(ww.w, fmaxf(ksign * v[h + 3], 0.f), a3);
              }
            } else {
              const float4 *s4 = reinterpret_cast<const float4 *>(ssm + gg * HI);
#pragma unroll
              for (int h = 0; h < HI; h += 4) {
                const float4 ww = w4[h / 4], sg = s4[h / 4];
                a0 = fmaf(ww.x, fmaxf(ksign * sg.x * v[h], 0.f), a0);
                a1 = fmaf(ww.y, fmaxf(ksign * sg.y * v[h + 1], 0.f), a1);
                a2 = fmaf(ww.z, fmaxf(ksign * sg.z * v[h + 2], 0.f), a2);
                a3 = fmaf(ww.w, fmaxf(ksign * sg.w * v[h + 3], 0.f), a3);
              }
            }
            if (key >= 0 && key <= pos0 + gg) p.scores[soff[gg] + key] = ((a0 + a1) + (a2 + a3)) * mag;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty(acc));
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

template <int G>
cudaError_t run_f8q(const dsa_ctx *ctx, const dsa_plan_t *plan, const IdxSet &set, const void *q_codes,
                    const float *q_scale, const float *w, const void *cache, float *scores, cudaStream_t s, int BH) {
  using C = F8qTraits<G>;
  const dsa_config_t &c = ctx->cfg;
  F8qParams prm{};
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
  if (!encode_tiled_2d(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void *>(q_codes), 128,
                       static_cast<uint64_t>(plan->T) * C::HI, 128, 128, C::N, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  prm.q_scale = q_scale;
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
  auto kern = index_f8q_kernel<G>;
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(kern, C::SMEM, ctx->device, smem_limit_set); e != cudaSuccess) return e;
  kern<<<set.n_ctas, C::THREADS, C::SMEM, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool indexer_f8q_supported(const dsa_config_t &c, const dsa_plan_t *plan) {
  return c.index_fmt == DSA_INDEX_FP8_132 && c.index_heads == 64 && c.index_dim == 128 && c.page_size % 8 == 0 &&
         plan->box_rows >= 8;
}

cudaError_t launch_index_scores_f8q(const dsa_ctx *ctx, const dsa_plan_t *plan, const void *q_codes,
                                    const float *q_scale, const float *w, const void *cache, float *scores,
                                    cudaStream_t s, int32_t *launches) {
  for (int si = 0; si < 2; ++si) {
    const IdxSet &set = plan->idx[si];
    if (set.n_items == 0) continue;
    cudaError_t e = set.G == 1 ? run_f8q<1>(ctx, plan, set, q_codes, q_scale, w, cache, scores, s, plan->box_rows)
                               : run_f8q<4>(ctx, plan, set, q_codes, q_scale, w, cache, scores, s, plan->box_rows);
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace dsa
