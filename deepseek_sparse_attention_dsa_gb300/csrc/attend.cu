// attend.cu -- sparse absorbed-MLA attention over the selected latents.
//
//   out[r, h] = sum_j softmax_j(l_j) c_j,   l_j = (q_nope[r,h] . c_j + q_pe[r,h] . kpe_j) * sm_scale
//
// over the positions j that row r selected (mstar DSAManager.attend: absorbed
// MLA over just the picked latents, (T, H, kv_lora_rank); ttnn sparse_sdpa: V
// is the leading kv_lora_rank columns of the same latent row, and an optional
// per-head sink joins only the softmax denominator).
//
// Tensor-core kernel (bf16 latents, H <= 128, kv_lora_rank in {128, 256,
// 512}, rope 64): a cluster of two CTAs handles one (row, key range).  CTA c
// owns latent columns [c*L/2, (c+1)*L/2) and rope columns [32c, 32c+32).  At
// the start of a unit the producers resolve every selected position of the
// unit to its physical cache row (one table in shared memory).  Then, per tile
// of 64 selected keys, both CTAs
//   * gather their 576 bytes of each of the 64 latent rows (cp.async, 128- and
//     64-byte swizzled tiles; completion signalled to an mbarrier, three
//     tiles in flight),
//   * compute partial logits S_c = Q[:, cols_c] . C[:, cols_c]^T on the tensor
//     core (M = 128 heads, N = 64 keys, fp32 in TMEM),
//   * swap the partials through distributed shared memory so both hold the
//     same full S and run the same online softmax (base 2, the reference max
//     moves only when it grows by more than 2^8, so O is rarely rescaled),
//   * write P as bf16 into tensor memory over the S tile it came from, and
//   * accumulate O_c += P . C[:, cols_c] (A from TMEM, B = the gathered tile
//     read MN-major; M = 128, N = L/2, fp32 in TMEM).
// The MMA work is split between the pair, not duplicated, and each latent byte
// is read once.  Rows split over several key ranges write fp32 partials (O,
// max, sum) that attend_combine_kernel merges.
//
// Other shapes and the fp8 latent format run attend_simt_kernel.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kNegBig = -1.0e30f;

// warp roles
// (8 warps: registers are handed out per group of four warps, so a ninth
// warp would cost as much register file as twelve)
constexpr int kMmaWarp = 0;
constexpr int kProdWarp0 = 1;               // warps 1-3: producers (96 threads)
constexpr int kSoftWarp0 = 4;               // warps 4-7: softmax, thread = head
constexpr int kProdThreads = 96;
constexpr int kAttThreads = 8 * 32;

template <int L>
struct AttTraits {
  static constexpr int HALF = L / 2;                     // latent columns per CTA
  static constexpr int NPV = HALF / 64;                  // 64-column (128-byte) chunks per CTA
  static constexpr int TILE = kAttTile;                  // keys per tile
  static constexpr int CHUNK = TILE * 128;               // [64 keys x 64 cols] bf16, 128-byte swizzle
  static constexpr int RCHUNK = TILE * 64;               // [64 keys x 32 rope cols], 64-byte swizzle
  static constexpr int STAGE = NPV * CHUNK + RCHUNK;
  static constexpr int STAGES = 3;
  static constexpr int PIECES = NPV * 8 + 4;             // 16-byte pieces per key per CTA
  static constexpr int QCHUNK = 128 * 128;               // [128 heads x 64 cols]
  static constexpr int QRCHUNK = 128 * 64;               // [128 heads x 32 rope cols]
  static constexpr int QBYTES = NPV * QCHUNK + QRCHUNK;
  static constexpr int XBYTES = 128 * TILE * 4;          // partial-logit exchange, fp32
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QBYTES;
  static constexpr int OFF_X = OFF_K + STAGES * STAGE;
  static constexpr int OFF_ROWS = OFF_X + XBYTES;        // int32 [topk]: physical row of each entry
  static constexpr int NBAR = 16;
  // the row table holds topk entries rounded up to whole tiles
  __host__ __device__ static constexpr int rows_bytes(int topk) { return (topk + TILE - 1) / TILE * TILE * 4; }
  static constexpr uint32_t IDESC_QK = mma_idesc(128, TILE, 1u, false, false);
  static constexpr uint32_t IDESC_PV = mma_idesc(128, HALF, 1u, false, true);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0;                   // two S tiles: cols 0..63, 64..127 (P over their first 32)
  static constexpr uint32_t O_COL = 256;                 // O half: cols 256 .. 256+HALF-1
  static_assert(HALF % 64 == 0 && HALF <= 256, "latent width");
};

// Shared-memory bytes of the tensor-core kernel for a given topk.
template <int L>
constexpr int att_smem_bytes(int topk) {
  return AttTraits<L>::OFF_ROWS + AttTraits<L>::rows_bytes(topk) + AttTraits<L>::NBAR * 8 + 16 + 1024;
}

struct AttParams {
  CUtensorMap tm_qn;       // q_nope as [T*H, L] bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tm_qp;       // q_pe as [T*H, R] bf16, box {32, 128}, 64-byte swizzle
  const int32_t *sel;
  const uint8_t *latent;   // [pages*P][L+R] bf16
  const float *sink;
  const AttUnit *units;
  const int32_t *row_pos, *row_page_off, *row_npages, *row_page_start, *pages;
  __nv_bfloat16 *out;      // [T][H][L]
  float *opart;            // [slots][H][L]
  float *mlpart;           // [slots][H][2]
  int *err;
  int H, K, P, num_pages;
  float scale_log2;        // sm_scale * log2(e)
};

// Physical latent row of selection entry j for a row, or -1 (masked).  -1 is
// the padding value; any other value outside 0..pos is a bounds error.
__device__ __forceinline__ int64_t latent_row(int j, int pos, int page_off, int npages, int page_start,
                                              const int32_t *pages, int P, int num_pages, int *err) {
  if (j < 0 || j > pos) {
    if (j != -1) atomicOr(err, kErrBounds);
    return -1;
  }
  const int64_t slot = static_cast<int64_t>(page_start) + j;
  const int64_t pi = slot / P;
  if (pi >= npages) {
    atomicOr(err, kErrBounds);
    return -1;
  }
  const int page = pages[page_off + pi];
  if (page < 0 || page >= num_pages) {
    atomicOr(err, kErrBounds);
    return -1;
  }
  return static_cast<int64_t>(page) * P + slot % P;
}

template <int L>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttThreads, 1)
    attend_tc_kernel(const __grid_constant__ AttParams p) {
  using C = AttTraits<L>;
  constexpr int R = 64;
  constexpr int ROWB = (L + R) * 2;        // bytes per latent row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int off_bar = C::OFF_ROWS + C::rows_bytes(p.K);
  const uint32_t bar0 = sbase + off_bar;
  const uint32_t b_qfull = bar0 + 0;
  auto kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (4 + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (7 + b); };
  auto sempty = [&](int b) { return bar0 + 8u * (9 + b); };
  const uint32_t b_pfull = bar0 + 8u * 11, b_pvdone = bar0 + 8u * 12;
  const uint32_t b_xfull = bar0 + 8u * 13, b_xfree = bar0 + 8u * 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + off_bar + C::NBAR * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + off_bar + C::NBAR * 8 + 4);
  int32_t *rows_sm = reinterpret_cast<int32_t *>(smem + C::OFF_ROWS);

  const int warp = threadIdx.x / 32, lane = lane_id();
  const uint32_t crank = cluster_rank();
  const uint32_t peer = crank ^ 1u;
  const AttUnit unit = p.units[blockIdx.x >> 1];
  const int row = unit.row;
  const int pos = p.row_pos[row];
  const int nent = unit.k1 - unit.k0;
  const int ntiles = (nent + C::TILE - 1) / C::TILE;

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kfull(s), kProdThreads);
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull(b), 1);
      mbar_init(sempty(b), 1);
    }
    mbar_init(b_pfull, 128);
    mbar_init(b_pvdone, 1);
    mbar_init(b_xfull, 1);   // armed locally with the exchange bytes; filled by the partner's st.async
    mbar_init(b_xfree, 4);   // one arrival per partner softmax warp once it has read its copy
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      mbar_arrive_expect_tx(b_qfull, C::QBYTES);
      for (int ch = 0; ch < C::NPV; ++ch)
        tma_load_2d(sbase + C::OFF_Q + ch * C::QCHUNK, &p.tm_qn, static_cast<int>(crank) * C::HALF + ch * 64,
                    row * p.H, b_qfull);
      tma_load_2d(sbase + C::OFF_Q + C::NPV * C::QCHUNK, &p.tm_qp, static_cast<int>(crank) * 32, row * p.H,
                  b_qfull);
      bool ok = mbar_wait(b_qfull, 0, abort_flag, p.err);
      const uint32_t o_tmem = tmem_base + C::O_COL;
      const uint32_t qst = sbase + C::OFF_Q;
      for (int t = 0; ok && t <= ntiles; ++t) {
        if (t < ntiles) {
          const int st = t % C::STAGES, sb = t & 1;
          if (!mbar_wait(kfull(st), (t / C::STAGES) & 1, abort_flag, p.err)) break;
          fence_proxy_async_smem();   // the gathered tile (generic-proxy writes) feeds the tensor core
          if (!mbar_wait(sempty(sb), ((t >> 1) & 1) ^ 1, abort_flag, p.err)) break;
          tc_fence_after();
          const uint32_t s_tmem = tmem_base + C::S_COL + sb * C::TILE;
          const uint32_t kst = sbase + C::OFF_K + st * C::STAGE;
#pragma unroll
          for (int ch = 0; ch < C::NPV; ++ch) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc(qst + ch * C::QCHUNK + k * 32, 16, 1024, kSwizzle128);
              const uint64_t bd = smem_desc(kst + ch * C::CHUNK + k * 32, 16, 1024, kSwizzle128);
              mma_f16_ss(s_tmem, ad, bd, C::IDESC_QK, (ch | k) ? 1u : 0u);
            }
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {   // this CTA's 32 rope columns
            const uint64_t ad = smem_desc(qst + C::NPV * C::QCHUNK + k * 32, 16, 512, kSwizzle64);
            const uint64_t bd = smem_desc(kst + C::NPV * C::CHUNK + k * 32, 16, 512, kSwizzle64);
            mma_f16_ss(s_tmem, ad, bd, C::IDESC_QK, 1u);
          }
          mma_commit(sfull(sb));
        }
        if (t >= 1) {
          const int u = t - 1;
          if (!mbar_wait(b_pfull, u & 1, abort_flag, p.err)) break;
          tc_fence_after();
          const uint32_t p_tmem = tmem_base + C::S_COL + (u & 1) * C::TILE;
          const uint32_t kst = sbase + C::OFF_K + (u % C::STAGES) * C::STAGE;
#pragma unroll
          for (int k = 0; k < C::TILE / 16; ++k) {
            const uint64_t bd = smem_desc(kst + k * 16 * 128, C::CHUNK, 1024, kSwizzle128);
            mma_f16_ts(o_tmem, p_tmem + k * 8, bd, C::IDESC_PV, (u > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(b_pvdone);
          mma_commit(kempty(u % C::STAGES));
          mma_commit(sempty(u & 1));
        }
      }
    }
    __syncwarp();
  } else if (warp < kSoftWarp0) {
    // ------------------------------------------------------------ producers
    const int pt = threadIdx.x - 32 * kProdWarp0;  // 0..95
    {
      const int page_off = p.row_page_off[row], npages = p.row_npages[row], page_start = p.row_page_start[row];
      const int32_t *selrow = p.sel + static_cast<int64_t>(row) * p.K + unit.k0;
      // eight entries per thread at a time: all selection loads, then all
      // page-table loads, are in flight together
      constexpr int kB = 8;
      for (int base = 0; base < ntiles * C::TILE; base += kProdThreads * kB) {
        int j[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int e = base + u * kProdThreads + pt;
          j[u] = e < nent ? selrow[e] : -1;
        }
        int pg[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          pg[u] = -1;
          if (j[u] >= 0 && j[u] <= pos) {
            const int64_t pi = (static_cast<int64_t>(page_start) + j[u]) / p.P;
            if (pi < npages) pg[u] = p.pages[page_off + pi];
          }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int e = base + u * kProdThreads + pt;
          if (e >= ntiles * C::TILE) continue;
          int32_t r = -1;
          if (j[u] < -1 || j[u] > pos) {
            atomicOr(p.err, kErrBounds);            // a position this row cannot see
          } else if (j[u] >= 0) {
            const int64_t slot = static_cast<int64_t>(page_start) + j[u];
            if (pg[u] < 0 || pg[u] >= p.num_pages || slot / p.P >= npages) atomicOr(p.err, kErrBounds);
            else r = static_cast<int32_t>(static_cast<int64_t>(pg[u]) * p.P + slot % p.P);
          }
          rows_sm[e] = r;
        }
      }
    }
    named_bar_sync(1, kProdThreads + 128);   // the row table is complete (producers + softmax)
    const int col0 = static_cast<int>(crank) * C::HALF;
    const int rcol0 = L + static_cast<int>(crank) * 32;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % C::STAGES;
      if (!mbar_wait(kempty(st), ((t / C::STAGES) & 1) ^ 1, abort_flag, p.err)) break;
      const uint32_t kst = sbase + C::OFF_K + st * C::STAGE;
      for (int idx = pt; idx < C::TILE * C::PIECES; idx += kProdThreads) {
        const int key = idx / C::PIECES;
        const int piece = idx - key * C::PIECES;
        const int32_t prow = rows_sm[t * C::TILE + key];
        uint32_t dst;
        int col;
        if (piece < C::NPV * 8) {
          dst = kst + (piece >> 3) * C::CHUNK + sw128_offset(key, piece & 7);
          col = col0 + piece * 8;
        } else {
          dst = kst + C::NPV * C::CHUNK + sw64_offset(key, piece - C::NPV * 8);
          col = rcol0 + (piece - C::NPV * 8) * 8;
        }
        const uint8_t *src = p.latent + (prow >= 0 ? static_cast<int64_t>(prow) * ROWB + col * 2 : 0);
        cp_async_16_zfill(dst, src, prow >= 0 ? 16u : 0u);
      }
      cp_async_mbar_arrive(kfull(st));
    }
    cp_async_wait<0>();   // nothing in flight when the CTA leaves
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int h = quad * 32 + lane;                      // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t x_own = sbase + C::OFF_X + h * 256;
    const uint32_t x_peer = map_to_cta(x_own, peer);
    const uint32_t peer_xfull = map_to_cta(b_xfull, peer), peer_xfree = map_to_cta(b_xfree, peer);
    float m_ref = kNegBig, l = 0.f;
    named_bar_sync(1, kProdThreads + 128);   // the row table is complete
    bool ok = true;
    // The partial logits of tile t+1 are sent to the partner before the softmax
    // of tile t runs, so the transfer overlaps the math.  The partner reads its
    // copy of tile t before this CTA sends tile t+1 into the same buffer
    // (xfree), which both CTAs reach without waiting on each other.
    float s[C::TILE];
    auto load_s = [&](int t, float (&dst)[C::TILE]) -> bool {
      if (!mbar_wait(sfull(t & 1), (t >> 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < C::TILE; c0 += 16)
        tmem_ld16(tmem_base + lane_base + C::S_COL + (t & 1) * C::TILE + c0,
                  *reinterpret_cast<float(*)[16]>(dst + c0));
      tmem_ld_wait();
      return true;
    };
    auto send_s = [&](const float (&src)[C::TILE]) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_async_v4(x_peer + ((c ^ (h & 15)) << 4), src[4 * c], src[4 * c + 1], src[4 * c + 2], src[4 * c + 3],
                    peer_xfull);
    };
    if (ntiles > 0) {
      ok = load_s(0, s);
      if (ok) send_s(s);
    }
    for (int t = 0; t < ntiles && ok; ++t) {
      const uint32_t vlo = __ballot_sync(0xffffffffu, rows_sm[t * C::TILE + lane] >= 0);
      const uint32_t vhi = __ballot_sync(0xffffffffu, rows_sm[t * C::TILE + 32 + lane] >= 0);
      const int sb = t & 1;

      // 1. the partner's partial logits of tile t (asynchronous remote stores
      //    that land on this CTA's mbarrier as transaction bytes)
      if (h == 0) mbar_arrive_expect_tx(b_xfull, C::XBYTES);
      if (!mbar_wait<true>(b_xfull, t & 1, abort_flag, p.err)) { ok = false; break; }
      const float4 *xr = reinterpret_cast<const float4 *>(smem + C::OFF_X + h * 256);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 v = xr[c ^ (h & 15)];
        s[4 * c] += v.x;
        s[4 * c + 1] += v.y;
        s[4 * c + 2] += v.z;
        s[4 * c + 3] += v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(peer_xfree);

      // 2. this CTA's partial logits of tile t+1 go out now
      float s_next[C::TILE];
      if (t + 1 < ntiles) {
        if (!load_s(t + 1, s_next)) { ok = false; break; }
        if (!mbar_wait<true>(b_xfree, t & 1, abort_flag, p.err)) { ok = false; break; }
        send_s(s_next);
      }

      // online softmax in base 2 with a lazily moved reference max
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < C::TILE; ++i) {
        const bool v = ((i < 32 ? vlo >> i : vhi >> (i - 32)) & 1u) != 0;
        s[i] = v ? s[i] * p.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, s[i]);
      }
      float alpha = 1.f;
      const bool rescale = tmax > m_ref + kRescaleThreshold;
      if (rescale) {
        alpha = exp2f(m_ref - tmax);
        m_ref = tmax;
      }
      float sum = 0.f;
      uint32_t packed[C::TILE / 2];
#pragma unroll
      for (int i = 0; i < C::TILE; i += 2) {
        const __nv_bfloat162 pb = __floats2bfloat162_rn(exp2f(s[i] - m_ref), exp2f(s[i + 1] - m_ref));
        const float2 pf = __bfloat1622float2(pb);
        sum += pf.x + pf.y;
        packed[i / 2] = *reinterpret_cast<const uint32_t *>(&pb);
      }
      l = l * alpha + sum;

      // O must hold every earlier tile before it is rescaled
      if (rescale && t > 0) {
        if (!mbar_wait(b_pvdone, (t - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < C::HALF; c0 += 16) {
          float o[16];
          tmem_ld16(tmem_base + lane_base + C::O_COL + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha;
          tmem_st16(tmem_base + lane_base + C::O_COL + c0, o);
        }
      }
      // P (bf16 pairs, lower key in the low half) over the first 32 columns of this S tile
      tmem_st32(tmem_base + lane_base + C::S_COL + sb * C::TILE, packed);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_pfull);
#pragma unroll
      for (int i = 0; i < C::TILE; ++i) s[i] = s_next[i];
    }
    if (ok && ntiles > 0) ok = mbar_wait(b_pvdone, (ntiles - 1) & 1, abort_flag, p.err);
    tc_fence_after();
    if (ok && h < p.H) {
      const int col0 = static_cast<int>(crank) * C::HALF;
      if (unit.slot < 0) {
        float f = 0.f;
        if (p.sink) {
          const float xs = p.sink[h] * kLog2e;
          const float mf = fmaxf(m_ref, xs);
          const float a = exp2f(m_ref - mf);
          const float lf = l * a + exp2f(xs - mf);
          f = lf > 0.f ? a / lf : 0.f;
        } else {
          f = l > 0.f ? 1.f / l : 0.f;
        }
        __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(row) * p.H + h) * L + col0;
#pragma unroll 1
        for (int c0 = 0; c0 < C::HALF; c0 += 16) {
          float o[16];
          if (ntiles > 0) {
            tmem_ld16(tmem_base + lane_base + C::O_COL + c0, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = 0.f;
          }
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i] * f, o[2 * i + 1] * f);
            w[i] = *reinterpret_cast<const uint32_t *>(&b);
          }
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      } else {
        float *dst = p.opart + (static_cast<int64_t>(unit.slot) * p.H + h) * L + col0;
#pragma unroll 1
        for (int c0 = 0; c0 < C::HALF; c0 += 16) {
          float o[16];
          if (ntiles > 0) {
            tmem_ld16(tmem_base + lane_base + C::O_COL + c0, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = 0.f;
          }
          float4 *d4 = reinterpret_cast<float4 *>(dst + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
        if (crank == 0) {
          float *ml = p.mlpart + (static_cast<int64_t>(unit.slot) * p.H + h) * 2;
          ml[0] = m_ref;
          ml[1] = l;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its partner may still touch its shared memory
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Merge of split rows: o = sum_s 2^(m_s - m) O_s / (sum_s 2^(m_s - m) l_s [+ 2^(sink - m)]).
// One block per (row, head); threads over the latent columns.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) attend_combine_kernel(const AttCombine *__restrict__ combine,
                                                             const float *__restrict__ opart,
                                                             const float *__restrict__ mlpart,
                                                             const float *__restrict__ sink, __nv_bfloat16 *out,
                                                             int H, int L) {
  const AttCombine cb = combine[blockIdx.x / H];
  const int h = blockIdx.x % H;
  float m = sink ? sink[h] * kLog2e : -INFINITY;
  for (int s = 0; s < cb.nsplit; ++s) m = fmaxf(m, mlpart[((cb.first_slot + s) * static_cast<int64_t>(H) + h) * 2]);
  float lsum = sink ? exp2f(sink[h] * kLog2e - m) : 0.f;
  for (int s = 0; s < cb.nsplit; ++s) {
    const float *ml = mlpart + ((cb.first_slot + s) * static_cast<int64_t>(H) + h) * 2;
    lsum += exp2f(ml[0] - m) * ml[1];
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  for (int d = threadIdx.x; d < L; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < cb.nsplit; ++s) {
      const int64_t base = (cb.first_slot + s) * static_cast<int64_t>(H) + h;
      acc += exp2f(mlpart[base * 2] - m) * opart[base * L + d];
    }
    out[(static_cast<int64_t>(cb.row) * H + h) * L + d] = __float2bfloat16_rn(acc * inv);
  }
}

// ---------------------------------------------------------------------------
// CUDA-core fallback: one block per (row, head), fp32 throughout.  Handles any
// width and both latent formats (fp8 656-byte rows: code * per-128 scale).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float latent_value(const uint8_t *rowp, int i, int L, int fp8) {
  if (!fp8) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(rowp)[i]);
  if (i < L) {
    __nv_fp8_e4m3 c;
    c.__x = rowp[i];
    return static_cast<float>(c) * reinterpret_cast<const float *>(rowp + L)[i / 128];
  }
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(rowp + L + 4 * (L / 128))[i - L]);
}

__global__ void __launch_bounds__(128) attend_simt_kernel(
    const int32_t *__restrict__ sel, const __nv_bfloat16 *__restrict__ q_nope, const __nv_bfloat16 *__restrict__ q_pe,
    const uint8_t *__restrict__ latent, const float *__restrict__ sink, const int32_t *__restrict__ row_pos,
    const int32_t *__restrict__ row_page_off, const int32_t *__restrict__ row_npages,
    const int32_t *__restrict__ row_page_start, const int32_t *__restrict__ pages, __nv_bfloat16 *out, int *err,
    int H, int L, int R, int K, int P, int num_pages, int fp8, int64_t row_bytes, float scale_log2) {
  extern __shared__ float sm[];  // q [L+R], logits [K], reduce [32]
  float *qs = sm;
  float *lg = sm + L + R;
  float *red = lg + K;
  const int row = blockIdx.x / H, h = blockIdx.x % H;
  const int pos = row_pos[row];
  for (int i = threadIdx.x; i < L + R; i += blockDim.x)
    qs[i] = i < L ? __bfloat162float(q_nope[(static_cast<int64_t>(row) * H + h) * L + i])
                  : __bfloat162float(q_pe[(static_cast<int64_t>(row) * H + h) * R + (i - L)]);
  __syncthreads();
  const int32_t *sr = sel + static_cast<int64_t>(row) * K;
  float mloc = -INFINITY;
  for (int e = threadIdx.x; e < K; e += blockDim.x) {
    const int64_t pr = latent_row(sr[e], pos, row_page_off[row], row_npages[row], row_page_start[row], pages, P,
                                  num_pages, err);
    float x = -INFINITY;
    if (pr >= 0) {
      const uint8_t *rp = latent + pr * row_bytes;
      float d = 0.f;
      for (int i = 0; i < L + R; ++i) d = fmaf(qs[i], latent_value(rp, i, L, fp8), d);
      x = d * scale_log2;
    }
    lg[e] = x;
    mloc = fmaxf(mloc, x);
  }
  for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = mloc;
  __syncthreads();
  float m = -INFINITY;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) m = fmaxf(m, red[w]);
  if (sink) m = fmaxf(m, sink[h] * kLog2e);
  __syncthreads();
  float lloc = 0.f;
  for (int e = threadIdx.x; e < K; e += blockDim.x) {
    const float pe = lg[e] == -INFINITY ? 0.f : exp2f(lg[e] - m);
    lg[e] = pe;
    lloc += pe;
  }
  for (int o = 16; o; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = lloc;
  __syncthreads();
  float lsum = sink ? exp2f(sink[h] * kLog2e - m) : 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) lsum += red[w];
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  for (int d = threadIdx.x; d < L; d += blockDim.x) {
    float acc = 0.f;
    for (int e = 0; e < K; ++e) {
      if (lg[e] == 0.f) continue;
      const int j = sr[e];
      const int64_t slot = static_cast<int64_t>(row_page_start[row]) + j;
      const int64_t pr = static_cast<int64_t>(pages[row_page_off[row] + slot / P]) * P + slot % P;
      acc = fmaf(lg[e], latent_value(latent + pr * row_bytes, d, L, fp8), acc);
    }
    out[(static_cast<int64_t>(row) * H + h) * L + d] = __float2bfloat16_rn(acc * inv);
  }
}

template <int L>
cudaError_t run_tc(const dsa_ctx *ctx, const dsa_plan_t *plan, const int32_t *sel, const void *q_nope,
                   const void *q_pe, const void *latent, const float *sink, float sm_scale, void *out,
                   cudaStream_t s) {
  const dsa_config_t &c = ctx->cfg;
  AttParams prm{};
  if (!encode_tiled_2d(&prm.tm_qn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q_nope), L,
                       static_cast<uint64_t>(plan->T) * c.heads, L * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled_2d(&prm.tm_qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q_pe), 64,
                       static_cast<uint64_t>(plan->T) * c.heads, 64 * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  prm.sel = sel;
  prm.latent = static_cast<const uint8_t *>(latent);
  prm.sink = sink;
  prm.units = plan->units;
  prm.row_pos = plan->row_pos;
  prm.row_page_off = plan->row_page_off;
  prm.row_npages = plan->row_npages;
  prm.row_page_start = plan->row_page_start;
  prm.pages = plan->pages;
  prm.out = static_cast<__nv_bfloat16 *>(out);
  prm.opart = ctx->opart;
  prm.mlpart = ctx->mlpart;
  prm.err = ctx->err;
  prm.H = c.heads;
  prm.K = c.topk;
  prm.P = c.page_size;
  prm.num_pages = plan->cache_pages;
  prm.scale_log2 = sm_scale * kLog2e;
  const int smem = att_smem_bytes<L>(c.topk);
  auto kern = attend_tc_kernel<L>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<2 * plan->n_units, kAttThreads, smem, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool attend_tc_supported(const dsa_config_t &c) {
  if (c.latent_fmt != DSA_LATENT_BF16 || c.heads > 128 || c.rope_dim != 64) return false;
  if (c.kv_lora_rank != 512 && c.kv_lora_rank != 256 && c.kv_lora_rank != 128) return false;
  // the per-unit row table (topk int32) must fit beside the tiles
  return att_smem_bytes<512>(c.topk) <= 227 * 1024;
}

cudaError_t launch_attend(const dsa_ctx *ctx, const dsa_plan_t *plan, const int32_t *sel, const void *q_nope,
                          const void *q_pe, const void *latent, const float *sink, float sm_scale, void *out,
                          cudaStream_t s, int32_t *launches) {
  const dsa_config_t &c = ctx->cfg;
  cudaError_t e;
  if (attend_tc_supported(c)) {
    if (c.kv_lora_rank == 512) e = run_tc<512>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    else if (c.kv_lora_rank == 256) e = run_tc<256>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    else e = run_tc<128>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    if (plan->n_combine > 0) {
      attend_combine_kernel<<<plan->n_combine * c.heads, 128, 0, s>>>(plan->combine, ctx->opart, ctx->mlpart, sink,
                                                                      static_cast<__nv_bfloat16 *>(out), c.heads,
                                                                      c.kv_lora_rank);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      *launches += 1;
    }
    return cudaSuccess;
  }
  const int fp8 = c.latent_fmt == DSA_LATENT_FP8_656;
  const int64_t row_bytes = fp8 ? c.kv_lora_rank + 4 * (c.kv_lora_rank / 128) + 2 * c.rope_dim
                                : 2 * static_cast<int64_t>(c.kv_lora_rank + c.rope_dim);
  const size_t sm = (static_cast<size_t>(c.kv_lora_rank) + c.rope_dim + c.topk + 32) * sizeof(float);
  if (sm > 48 * 1024) {
    e = cudaFuncSetAttribute(attend_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
    if (e != cudaSuccess) return e;
  }
  attend_simt_kernel<<<plan->T * c.heads, 128, sm, s>>>(
      sel, static_cast<const __nv_bfloat16 *>(q_nope), static_cast<const __nv_bfloat16 *>(q_pe),
      static_cast<const uint8_t *>(latent), sink, plan->row_pos, plan->row_page_off, plan->row_npages,
      plan->row_page_start, plan->pages, static_cast<__nv_bfloat16 *>(out), ctx->err, c.heads, c.kv_lora_rank,
      c.rope_dim, c.topk, c.page_size, plan->cache_pages, fp8, row_bytes, sm_scale * kLog2e);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches += 1;
  return cudaSuccess;
}

}  // namespace dsa
