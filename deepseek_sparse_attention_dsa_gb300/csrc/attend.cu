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
// 512}, rope 64).  One CTA per (row, key range, output half c): it computes
// the full logits of all 128 heads and accumulates O for latent columns
// [c*L/2, (c+1)*L/2), so the two halves of a row share nothing but their
// inputs (the QK contraction is done by both; in exchange no CTA ever waits on
// another).  Per tile of 32 selected keys (four tiles in flight):
//   * 7 producer warps gather the tile's latent rows through the page table
//     (cp.async into 128-byte swizzled tiles; completion lands on an mbarrier;
//     the page-table lookups of the next tiles are already in flight);
//   * one thread issues S = Q . C^T (M = 128 heads, N = 32 keys, K = L + R,
//     fp32 in TMEM); the first columns of Q live in TMEM (the MMA's A operand
//     from tensor memory), the rest in shared memory;
//   * 4 softmax warps (thread = head) run a base-2 online softmax whose
//     reference max moves only when it grows by more than 2^8 (so O is rarely
//     rescaled) and write P as bf16 over the S tile in TMEM;
//   * one thread issues O += P . C[:, half] (A = P from TMEM, B = the gathered
//     tile read MN-major; M = 128, N = L/2, fp32 in TMEM).
// S is double-buffered in TMEM so QK of tile t+1 overlaps the softmax of tile t.
// Rows split over several key ranges write fp32 partials (O, max, sum) that
// attend_combine_kernel merges.
//
// fp8 latents (656-byte rows) take the same kernel: the producers load the
// codes, scales and rope into registers, dequantise (code x the scale of its
// 128-column group, rounded to bf16) and store the bf16 tile the MMAs read.
// Other shapes run attend_simt_kernel.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kNegBig = -1.0e30f;

// warp roles (12 warps; registers are handed out per group of four warps)
constexpr int kMmaWarp = 0;
constexpr int kProdWarp0 = 1;               // warps 1-7: producers (224 threads)
constexpr int kSoftWarp0 = 8;               // warps 8-11: softmax, thread = head
constexpr int kProdThreads = 224;
constexpr int kAttThreads = 12 * 32;

template <int L>
struct AttTraits {
  static constexpr int R = 64;
  static constexpr int HALF = L / 2;                     // output columns per CTA
  static constexpr int NPV = HALF / 64;                  // 64-column chunks of the output half
  static constexpr int NCH = (L + R) / 64;               // 64-column chunks of a latent row
  static constexpr int TILE = 32;                        // keys per tile (UMMA N of QK)
  static constexpr int CHUNK = TILE * 128;               // [32 keys x 64 cols] bf16, 128-byte swizzle
  static constexpr int STAGE = NCH * CHUNK;
  static constexpr int STAGES = 4;
  // tensor memory: [Q columns held in TMEM | S tile 0 | S tile 1 | O half]
  static constexpr int S_COLS = 2 * TILE;
  static constexpr int QT_CH_MAX = (512 - HALF - S_COLS) / 32;  // 64-column Q chunks that fit
  static constexpr int QT_CH = QT_CH_MAX < L / 64 ? QT_CH_MAX : L / 64;  // q_nope chunks only
  static constexpr uint32_t S_COL = QT_CH * 32;
  static constexpr uint32_t O_COL = S_COL + S_COLS;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int QS_CH = NCH - QT_CH;              // Q chunks in shared memory
  static constexpr int QCHUNK = 128 * 128;               // [128 heads x 64 cols]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QS_CH * QCHUNK;
  static constexpr int OFF_ROWS = OFF_K + STAGES * STAGE;  // int32 [STAGES][TILE]
  static constexpr int OFF_BAR = OFF_ROWS + STAGES * TILE * 4;
  static constexpr int NBAR = 20;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t IDESC_QK = mma_idesc(128, TILE, 1u, false, false);
  static constexpr uint32_t IDESC_PV = mma_idesc(128, HALF, 1u, false, true);
  static_assert(HALF % 64 == 0 && HALF <= 256, "latent width");
  static_assert(O_COL + HALF <= TMEM_COLS, "tensor memory");
  static_assert(QT_CH * QCHUNK <= STAGES * STAGE, "Q staging");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct AttParams {
  CUtensorMap tm_qn;       // q_nope as [T*H, L] bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tm_qp;       // q_pe as [T*H, R] bf16, box {64, 128}, 128-byte swizzle
  const int32_t *sel;
  const uint8_t *latent;   // [pages*P][L+R] bf16
  const __nv_bfloat16 *q_nope;
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

// 16 e4m3 codes (one 16-byte piece, lowest address first) times `scale`,
// rounded to 16 bf16 (two 16-byte pieces).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 raw, float scale, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hlf)) & 0xFFFFu),
                                                       __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
      o[2 * i + hlf] = *reinterpret_cast<const uint32_t *>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

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

template <int L, bool FP8>
__global__ void __launch_bounds__(kAttThreads, 1) attend_tc_kernel(const __grid_constant__ AttParams p) {
  using C = AttTraits<L>;
  constexpr int R = C::R;
  constexpr int ROWB = (L + R) * 2;        // bytes per latent row
  constexpr int T = C::TILE;
  constexpr int NS = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t b_qsfull = bar0 + 0, b_qtfull = bar0 + 8, b_qtdone = bar0 + 16;
  auto kfull = [&](int s) { return bar0 + 8u * (3 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (3 + NS + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (3 + 2 * NS + b); };
  auto sempty = [&](int b) { return bar0 + 8u * (5 + 2 * NS + b); };
  auto pfull = [&](int b) { return bar0 + 8u * (7 + 2 * NS + b); };
  const uint32_t b_pvdone = bar0 + 8u * (9 + 2 * NS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int32_t *rows_sm = reinterpret_cast<int32_t *>(smem + C::OFF_ROWS);

  const int warp = threadIdx.x / 32, lane = lane_id();
  const int half = blockIdx.x & 1;
  const AttUnit unit = p.units[blockIdx.x >> 1];
  const int row = unit.row;
  const int pos = p.row_pos[row];
  const int nent = unit.k1 - unit.k0;
  const int ntiles = (nent + T - 1) / T;
  const int32_t *selrow = p.sel + static_cast<int64_t>(row) * p.K + unit.k0;

  if (threadIdx.x == 0) {
    mbar_init(b_qsfull, 1);
    mbar_init(b_qtfull, 1);
    mbar_init(b_qtdone, 128);
    for (int s = 0; s < NS; ++s) {
      mbar_init(kfull(s), kProdThreads);
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull(b), 1);
      mbar_init(sempty(b), 1);
      mbar_init(pfull(b), 128);
    }
    mbar_init(b_pvdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Q columns kept in shared memory, and (through the still idle stage
      // buffers) the columns the softmax warps move into tensor memory
      mbar_arrive_expect_tx(b_qsfull, C::QS_CH * C::QCHUNK);
      for (int ch = C::QT_CH; ch < C::NCH; ++ch) {
        const uint32_t dst = sbase + C::OFF_Q + (ch - C::QT_CH) * C::QCHUNK;
        if (ch * 64 < L) tma_load_2d(dst, &p.tm_qn, ch * 64, row * p.H, b_qsfull);
        else tma_load_2d(dst, &p.tm_qp, ch * 64 - L, row * p.H, b_qsfull);
      }
      mbar_arrive_expect_tx(b_qtfull, C::QT_CH * C::QCHUNK);
      for (int ch = 0; ch < C::QT_CH; ++ch)
        tma_load_2d(sbase + C::OFF_K + ch * C::QCHUNK, &p.tm_qn, ch * 64, row * p.H, b_qtfull);
      bool ok = mbar_wait(b_qsfull, 0, abort_flag, p.err) && mbar_wait(b_qtdone, 0, abort_flag, p.err);
      const uint32_t o_tmem = tmem_base + C::O_COL;
      // descriptors are built once; a K step of 16 columns (32 bytes) adds 2 to
      // the encoded start address, a chunk adds chunk_bytes / 16
      const uint64_t qdesc = smem_desc(sbase + C::OFF_Q, 16, 1024, kSwizzle128);
      const uint64_t kdesc0 = smem_desc(sbase + C::OFF_K, 16, 1024, kSwizzle128);
      const uint64_t vdesc0 = smem_desc(sbase + C::OFF_K + half * C::NPV * C::CHUNK, C::CHUNK, 1024, kSwizzle128);
      constexpr uint64_t kStageStep = C::STAGE >> 4;
      // issue QK of the next tile or PV of the oldest softmaxed tile, whichever is ready
      int nq = 0, np = 0;
      uint64_t idle_since = 0;
      uint32_t idle = 0;
      while (ok && np < ntiles) {
        bool progressed = false;
        if (nq < ntiles && nq < np + 2) {
          const int st = nq % NS, sb = nq & 1;
          if (mbar_test(kfull(st), (nq / NS) & 1) && mbar_test(sempty(sb), ((nq >> 1) & 1) ^ 1)) {
            fence_proxy_async_smem();   // the gathered tile (cp.async writes) feeds the tensor core
            tc_fence_after();
            const uint32_t s_tmem = tmem_base + C::S_COL + sb * T;
            const uint64_t kd = kdesc0 + st * kStageStep;
#pragma unroll
            for (int ch = 0; ch < C::QT_CH; ++ch)       // Q columns in tensor memory
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_ts(s_tmem, tmem_base + ch * 32 + k * 8, kd + (ch * C::CHUNK >> 4) + 2 * k, C::IDESC_QK,
                           (ch | k) ? 1u : 0u);
#pragma unroll
            for (int ch = C::QT_CH; ch < C::NCH; ++ch)   // Q columns in shared memory
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_ss(s_tmem, qdesc + ((ch - C::QT_CH) * C::QCHUNK >> 4) + 2 * k,
                           kd + (ch * C::CHUNK >> 4) + 2 * k, C::IDESC_QK, (ch | k) ? 1u : 0u);
            mma_commit(sfull(sb));
            ++nq;
            progressed = true;
          }
        }
        if (np < nq && mbar_test(pfull(np & 1), (np >> 1) & 1)) {
          tc_fence_after();
          const int st = np % NS, sb = np & 1;
          const uint32_t p_tmem = tmem_base + C::S_COL + sb * T;
#pragma unroll
          for (int k = 0; k < T / 16; ++k)
            mma_f16_ts(o_tmem, p_tmem + k * 8, vdesc0 + st * kStageStep + (k * 16 * 128 >> 4), C::IDESC_PV,
                       (np > 0 || k > 0) ? 1u : 0u);
          mma_commit(b_pvdone);
          mma_commit(kempty(st));
          mma_commit(sempty(sb));
          ++np;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
          idle_since = 0;
        } else if ((++idle & 255) == 0) {
          if (*abort_flag) break;
          if (idle_since == 0) idle_since = globaltimer();
          else if (globaltimer() - idle_since > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.err, kErrTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < kSoftWarp0) {
    // ------------------------------------------------------------ producers
    // Three warps copy each tile with cp.async: eight lanes per 128-byte chunk
    // of a latent row, 128-byte swizzled into the tile; the arrival on the
    // stage's mbarrier fires when this thread's copies have landed.  Warp 1
    // resolves the tile's rows (lane l: key l); the selection entries of tile
    // t+2 and the page ids of tile t+1 are loaded while tile t is issued.
    const int pt = threadIdx.x - 32 * kProdWarp0;  // 0..223
    const int page_off = p.row_page_off[row], npages = p.row_npages[row], page_start = p.row_page_start[row];
    const bool resolver = warp == kProdWarp0;
    auto sel_at = [&](int t) -> int {
      const int e = t * T + lane;
      return (resolver && t < ntiles && e < nent) ? selrow[e] : -1;
    };
    auto page_of = [&](int j) -> int {
      if (j < 0 || j > pos) return -1;
      const int64_t pi = (static_cast<int64_t>(page_start) + j) / p.P;
      return pi < npages ? p.pages[page_off + pi] : -1;
    };
    auto phys = [&](int j, int pg) -> int32_t {   // -1: masked (zero-filled, its P is 0)
      if (j == -1) return -1;
      if (j < -1 || j > pos || pg < 0 || pg >= p.num_pages) {
        atomicOr(p.err, kErrBounds);
        return -1;
      }
      const int64_t slot = static_cast<int64_t>(page_start) + j;
      return static_cast<int32_t>(static_cast<int64_t>(pg) * p.P + slot % p.P);
    };
    int j0 = sel_at(0), j1 = sel_at(1);
    int pg0 = page_of(j0);
    const int piece = lane & 7, sub = pt >> 3;        // sub: one 128-byte chunk per 8 lanes
    // the stage buffers hold the tensor-memory part of Q until it has been moved
    bool ok = mbar_wait(b_qtdone, 0, abort_flag, p.err);
    for (int t = 0; ok && t < ntiles; ++t) {
      const int st = t % NS;
      const int pg1 = page_of(j1);
      const int j2 = sel_at(t + 2);
      if (!FP8 && !mbar_wait(kempty(st), ((t / NS) & 1) ^ 1, abort_flag, p.err)) break;
      int32_t *rows = rows_sm + st * T;
      if (resolver) rows[lane] = phys(j0, pg0);
      named_bar_sync(2, kProdThreads);
      const uint32_t kst = sbase + C::OFF_K + st * C::STAGE;
      if constexpr (!FP8) {
        // chunk q = key * NCH + ch: consecutive q are consecutive chunks of one row
#pragma unroll 4
        for (int q = sub; q < T * C::NCH; q += kProdThreads / 8) {
          const int key = q / C::NCH, ch = q - key * C::NCH;
          const int32_t prow = rows[key];
          const uint32_t dst = kst + ch * C::CHUNK + sw128_offset(key, piece);
          const uint8_t *src =
              p.latent + (prow >= 0 ? static_cast<int64_t>(prow) * ROWB + ch * 128 + piece * 16 : 0);
          cp_async_16_zfill(dst, src, prow >= 0 ? 16u : 0u);
        }
        cp_async_mbar_arrive(kfull(st));
      } else {
        // 656-byte rows [L e4m3 | L/128 fp32 scales | R bf16]: 16-byte pieces are
        // loaded into registers, dequantised (code x scale, rounded to bf16) and
        // stored into the same swizzled bf16 tile the bf16 path gathers.  The
        // loads are issued before the stage is known to be free.
        constexpr int CP = L / 16, RP = R * 2 / 16, PPK = CP + RP;
        constexpr int RB8 = L + 4 * (L / 128) + 2 * R;
        constexpr int PER = (T * PPK + kProdThreads - 1) / kProdThreads;
        uint4 raw[PER];
        float scl[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int i = pt + u * kProdThreads;
          raw[u] = make_uint4(0, 0, 0, 0);
          scl[u] = 0.f;
          if (i < T * PPK) {
            const int key = i / PPK, k = i - key * PPK;
            const int32_t prow = rows[key];
            if (prow >= 0) {
              const uint8_t *base = p.latent + static_cast<int64_t>(prow) * RB8;
              if (k < CP) {
                raw[u] = __ldg(reinterpret_cast<const uint4 *>(base + 16 * k));
                scl[u] = __ldg(reinterpret_cast<const float *>(base + L) + k / 8);
              } else {
                raw[u] = __ldg(reinterpret_cast<const uint4 *>(base + L + 4 * (L / 128) + 16 * (k - CP)));
              }
            }
          }
        }
        if (!mbar_wait(kempty(st), ((t / NS) & 1) ^ 1, abort_flag, p.err)) break;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int i = pt + u * kProdThreads;
          if (i >= T * PPK) continue;
          const int key = i / PPK, k = i - key * PPK;
          if (k < CP) {
            uint4 lo, hi;
            e4m3x16_to_bf16(raw[u], scl[u], lo, hi);
            const uint32_t chunk = kst + (k / 4) * C::CHUNK;
            st_shared_v4(chunk + sw128_offset(key, (k % 4) * 2), lo);
            st_shared_v4(chunk + sw128_offset(key, (k % 4) * 2 + 1), hi);
          } else {
            st_shared_v4(kst + (C::NCH - 1) * C::CHUNK + sw128_offset(key, k - CP), raw[u]);
          }
        }
        mbar_arrive(kfull(st));
      }
      j0 = j1;
      j1 = j2;
      pg0 = pg1;
    }
    cp_async_wait<0>();   // nothing in flight when the CTA leaves
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int h = quad * 32 + lane;                      // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = mbar_wait(b_qtfull, 0, abort_flag, p.err);
    if (ok) {
      // this head's row of the tensor-memory part of Q: from the staged
      // swizzled chunks into TMEM (bf16 pairs, lower column in the low half)
#pragma unroll 1
      for (int ch = 0; ch < C::QT_CH; ++ch) {
        const uint8_t *src = smem + C::OFF_K + ch * C::QCHUNK + h * 128;
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = *reinterpret_cast<const uint4 *>(src + ((i ^ (h & 7)) << 4));
          v[4 * i] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st32(tmem_base + lane_base + ch * 32, v);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(b_qtdone);
    float m_ref = kNegBig, l = 0.f;
    int jn = lane < nent ? selrow[lane] : -1;
    for (int t = 0; t < ntiles && ok; ++t) {
      const uint32_t valid = __ballot_sync(0xffffffffu, jn >= 0 && jn <= pos);
      if (t + 1 < ntiles) {
        const int e = (t + 1) * T + lane;
        jn = e < nent ? selrow[e] : -1;
      }
      const int sb = t & 1;
      if (!mbar_wait(sfull(sb), (t >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float s[T];
#pragma unroll
      for (int c0 = 0; c0 < T; c0 += 16)
        tmem_ld16(tmem_base + lane_base + C::S_COL + sb * T + c0, *reinterpret_cast<float(*)[16]>(s + c0));
      tmem_ld_wait();

      // online softmax in base 2 with a lazily moved reference max
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < T; ++i) {
        s[i] = ((valid >> i) & 1u) ? s[i] * p.scale_log2 : -INFINITY;
        mx[i & 3] = fmaxf(mx[i & 3], s[i]);
      }
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      float alpha = 1.f;
      const bool rescale = tmax > m_ref + kRescaleThreshold;
      if (rescale) {
        alpha = exp2f(m_ref - tmax);
        m_ref = tmax;
      }
      float sm[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t packed[T / 2];
#pragma unroll
      for (int i = 0; i < T; i += 2) {
        const __nv_bfloat162 pb = __floats2bfloat162_rn(exp2f(s[i] - m_ref), exp2f(s[i + 1] - m_ref));
        const float2 pf = __bfloat1622float2(pb);
        sm[(i >> 1) & 3] += pf.x + pf.y;
        packed[i / 2] = *reinterpret_cast<const uint32_t *>(&pb);
      }
      l = l * alpha + ((sm[0] + sm[1]) + (sm[2] + sm[3]));

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
      // P (bf16 pairs, lower key in the low half) over the first T/2 columns of this S tile
      tmem_st16(tmem_base + lane_base + C::S_COL + sb * T, *reinterpret_cast<const float(*)[16]>(packed));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pfull(sb));
    }
    if (ok && ntiles > 0) ok = mbar_wait(b_pvdone, (ntiles - 1) & 1, abort_flag, p.err);
    tc_fence_after();
    if (ok && h < p.H) {
      const int col0 = half * C::HALF;
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
        if (half == 0) {
          float *ml = p.mlpart + (static_cast<int64_t>(unit.slot) * p.H + h) * 2;
          ml[0] = m_ref;
          ml[1] = l;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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

template <int L, bool FP8>
cudaError_t run_tc(const dsa_ctx *ctx, const dsa_plan_t *plan, const int32_t *sel, const void *q_nope,
                   const void *q_pe, const void *latent, const float *sink, float sm_scale, void *out,
                   cudaStream_t s) {
  using Cfg = AttTraits<L>;
  const dsa_config_t &c = ctx->cfg;
  AttParams prm{};
  if (!encode_tiled_2d(&prm.tm_qn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q_nope), L,
                       static_cast<uint64_t>(plan->T) * c.heads, L * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled_2d(&prm.tm_qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q_pe), 64,
                       static_cast<uint64_t>(plan->T) * c.heads, 64 * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  prm.sel = sel;
  prm.latent = static_cast<const uint8_t *>(latent);
  prm.q_nope = static_cast<const __nv_bfloat16 *>(q_nope);
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
  auto kern = attend_tc_kernel<L, FP8>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<2 * plan->n_units, kAttThreads, Cfg::SMEM, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool attend_tc_supported(const dsa_config_t &c) {
  if (c.heads > 128 || c.rope_dim != 64) return false;
  if (c.latent_fmt == DSA_LATENT_FP8_656) return c.kv_lora_rank == 512;
  return c.kv_lora_rank == 512 || c.kv_lora_rank == 256 || c.kv_lora_rank == 128;
}

cudaError_t launch_attend(const dsa_ctx *ctx, const dsa_plan_t *plan, const int32_t *sel, const void *q_nope,
                          const void *q_pe, const void *latent, const float *sink, float sm_scale, void *out,
                          cudaStream_t s, int32_t *launches) {
  const dsa_config_t &c = ctx->cfg;
  cudaError_t e;
  if (attend_tc_supported(c)) {
    if (c.latent_fmt == DSA_LATENT_FP8_656)
      e = run_tc<512, true>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    else if (c.kv_lora_rank == 512)
      e = run_tc<512, false>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    else if (c.kv_lora_rank == 256)
      e = run_tc<256, false>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
    else
      e = run_tc<128, false>(ctx, plan, sel, q_nope, q_pe, latent, sink, sm_scale, out, s);
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
