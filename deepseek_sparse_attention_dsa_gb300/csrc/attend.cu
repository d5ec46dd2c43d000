// attend.cu -- sparse absorbed-MLA attention over the selected latents.
//
//   out[r, h] = sum_j softmax_j(l_j) c_j,   l_j = (q_nope[r,h] . c_j + q_pe[r,h] . kpe_j) * sm_scale
//
// over the positions j that row r selected (mstar DSAManager.attend: absorbed
// MLA over just the picked latents, (T, H, kv_lora_rank); ttnn sparse_sdpa: V
// is the leading kv_lora_rank columns of the same latent row, and an optional
// per-head sink joins only the softmax denominator).
//
// Tensor-core kernel (H <= 128, kv_lora_rank in {128, 256, 512}, rope 64): a
// cluster of two CTAs handles one (row, key range).  CTA c owns latent
// columns [c*L/2, (c+1)*L/2) and rope columns [32c, 32c+32), so every latent
// byte is gathered once and every MMA is issued once.  Per tile of 64 selected
// keys, four tiles in flight:
//   * 7 producer warps gather the CTA's 576 bytes of each latent row through
//     the page table (cp.async into 128- and 64-byte swizzled tiles;
//     completion lands on an mbarrier; the selection entries and page ids of
//     the next tiles are already in flight).  For fp8 latents (656-byte
//     rows) the codes and scales are loaded into registers, dequantised (code
//     x the scale of its 128-column group, rounded to bf16) and stored as the
//     same bf16 tiles, and the rope columns (bf16 already) come by cp.async;
//   * one thread issues the partial logits S_c = Q[:, cols_c] . C[:, cols_c]^T
//     (M = 128 heads, N = 64 keys, fp32 in TMEM; the q_nope columns of this
//     CTA live in tensor memory as the A operand, the rope columns in shared
//     memory).  A K = 16 tcgen05.mma costs about the same for N = 32 as for
//     N = 64 on sm_103a, so splitting the contraction between the pair halves
//     the instruction count per key where duplicating it would double it;
//   * 4 sender warps (thread = head) take each S tile out of TMEM as soon as
//     its QK is done, stage it in shared memory and bulk-copy it into the
//     partner's receive buffer (the copy lands on the partner's mbarrier).
//     The receive buffer is two halves of 32 keys with their own barriers,
//     so the first half of tile t+1 travels while tile t's second half is
//     being merged;
//   * 8 softmax warps, two per TMEM lane quadrant (thread = head, 32 keys of
//     the tile each), add the partner's partial to their own (a + b == b + a,
//     so both CTAs hold the identical full S) and run the same base-2 online
//     softmax (the pair shares each tile's max through shared memory; the
//     reference max moves only when it grows by more than 2^8, so O is rarely
//     rescaled); P goes to TMEM as bf16 in its own columns;
//   * one thread issues O_c += P . C[:, cols_c] (A = P from TMEM, B = the
//     gathered tile read MN-major; M = 128, N = L/2, fp32 in TMEM).
// S is double-buffered in TMEM so QK of tile t+1 overlaps the softmax of tile
// t; an S tile is free once the softmax and sender warps have read it.  Rows
// split over several key ranges write fp32 partials (O, max, sum) that
// attend_combine_kernel merges.
//
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

// warp roles (20 warps; every warp of a TMEM lane quadrant q sits on sub-partition q = warp % 4)
constexpr int kMmaWarp = 0;
constexpr int kProdWarp0 = 1;               // warps 1-7: producers (224 threads)
constexpr int kSoftWarp0 = 8;               // warps 8-15: softmax, thread = head; warps 8-11 keys 0-31, 12-15 keys 32-63
constexpr int kSendWarp0 = 16;              // warps 16-19: partial-logit senders, thread = head
constexpr int kProdThreads = 224;
constexpr int kAttThreads = 20 * 32;

template <int L>
struct AttTraits {
  static constexpr int R = 64;
  static constexpr int HALF = L / 2;                     // latent (and output) columns per CTA
  static constexpr int NPV = HALF / 64;                  // 64-column chunks of those
  static constexpr int RH = R / 2;                       // rope columns per CTA
  static constexpr int TILE = kAttTile;                  // keys per tile (UMMA N of QK)
  static constexpr int CHUNK = TILE * 128;               // [64 keys x 64 cols] bf16, 128-byte swizzle
  static constexpr int RCHUNK = TILE * 64;               // [64 keys x 32 rope cols], 64-byte swizzle
  static constexpr int STAGE = NPV * CHUNK + RCHUNK;
  static constexpr int STAGES = 4;
  static constexpr int PIECES = NPV * 8 + 4;             // 16-byte pieces of a key's part
  static constexpr int QCHUNK = 128 * 128;               // [128 heads x 64 cols]
  static constexpr int QRBYTES = 128 * 64;               // [128 heads x 32 rope cols]
  static constexpr int XBYTES = 128 * TILE * 4;          // partial logits of a tile, fp32
  // The receive buffer x_in is two halves, one per 32 keys of the tile, each
  // with its own full/free barriers: the partner sends the first half of tile
  // t+1 as soon as the first half of tile t has been merged.
  static constexpr int XHALF = XBYTES / 2;               // [128 heads x 32 keys] fp32, 128-byte rows
  static constexpr int XOUT = XHALF;                     // send staging: one half-row block (4 KB) per sender warp
  static_assert(XOUT / 4 == 32 * 128 && TILE == 64, "send staging slot");
  // q_nope chunks of this CTA: the first QT_CH in tensor memory (A operand),
  // the rest in shared memory
  static constexpr int QT_CH = NPV < 3 ? NPV : 3;
  static constexpr int QS_CH = NPV - QT_CH;
  // tensor memory: [q_nope chunks | P | S tile 0 | S tile 1 | O].  P has its
  // own columns, so an S tile is free for the next QK as soon as it has been
  // read, not only after PV.
  static constexpr uint32_t P_COL = 96;
  static constexpr uint32_t S_COL = 128;
  static constexpr uint32_t O_COL = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int OFF_QR = 0;
  static constexpr int OFF_QS = 8192;                    // q_nope chunks in shared memory
  static constexpr int OFF_K = OFF_QS + QS_CH * QCHUNK;
  static constexpr int OFF_X = OFF_K + STAGES * STAGE;   // x_in (two halves) then x_out (XOUT bytes)
  static constexpr int OFF_ROWS = OFF_X + XBYTES + XOUT;   // int32 [STAGES][TILE]
  // fp32 [2 tiles][2 halves][128] maxima, then [2 units][2 halves][128] sums
  static constexpr int OFF_RED = OFF_ROWS + STAGES * TILE * 4;
  static constexpr int OFF_BAR = OFF_RED + (4 + 4) * 128 * 4;
  static constexpr int NBAR = 24;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t IDESC_QK = mma_idesc(128, TILE, 1u, false, false);
  static constexpr uint32_t IDESC_PV = mma_idesc(128, HALF, 1u, false, true);
  static_assert(HALF % 64 == 0 && HALF <= 256, "latent width");
  static_assert(QT_CH * 32 <= static_cast<int>(P_COL) && P_COL + TILE / 2 <= S_COL, "tensor memory: Q, P");
  static_assert(O_COL + HALF <= TMEM_COLS, "tensor memory: O");
  static_assert(QRBYTES <= OFF_K && STAGE % 1024 == 0, "alignment");
  static_assert(NBAR >= 16 + 2 * STAGES, "barriers");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct AttParams {
  CUtensorMap tm_qn;       // q_nope as [T*H, L] bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tm_qp;       // q_pe as [T*H, R] bf16, box {32, 128}, 64-byte swizzle
  const __nv_bfloat16 *qn; // q_nope [T][H][L] (the chunks that go to tensor memory are read directly)
  const int32_t *sel;
  const uint8_t *latent;   // bf16 rows [L+R] or fp8 656-byte rows, [pages*P]
  const float *sink;
  const AttUnit *units;
  const AttCluster *clusters;   // [grid / 2]
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

// 2^x with the MUFU approximation (relative error ~2^-22; tiny results flush
// to zero, which the bf16 probabilities would round to anyway).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttThreads, 1)
    attend_tc_kernel(const __grid_constant__ AttParams p) {
  using C = AttTraits<L>;
  constexpr int R = C::R;
  constexpr int T = C::TILE;
  constexpr int NS = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  // qsfull: a unit's rope and shared-memory q_nope columns landed (TMA);
  // qkdone: a unit's last QK completed (its Q may be replaced); qtdone: the
  // softmax warps wrote a unit's tensor-memory q_nope columns; pvdone: a PV
  // completed; ofree: the softmax warps have read a unit's O out
  const uint32_t b_qsfull = bar0, b_qkdone = bar0 + 8, b_qtdone = bar0 + 16, b_pvdone = bar0 + 24;
  auto kfull = [&](int s) { return bar0 + 8u * (4 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (4 + NS + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (4 + 2 * NS + b); };
  auto sempty = [&](int b) { return bar0 + 8u * (6 + 2 * NS + b); };
  auto pfull = [&](int b) { return bar0 + 8u * (8 + 2 * NS + b); };
  auto xfull = [&](int b) { return bar0 + 8u * (10 + 2 * NS + b); };   // the partner's partial landed in x_in[b]
  auto xfree = [&](int b) { return bar0 + 8u * (12 + 2 * NS + b); };   // the partner has read our x_in[b] copy
  const uint32_t b_ofree = bar0 + 8u * (14 + 2 * NS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  int32_t *rows_sm = reinterpret_cast<int32_t *>(smem + C::OFF_ROWS);

  const int warp = threadIdx.x / 32, lane = lane_id();
  const uint32_t crank = cluster_rank();
  const uint32_t peer = crank ^ 1u;
  // this cluster's units: contiguous pieces of rows, `ntotal` key tiles in all
  const AttCluster cl = p.clusters[blockIdx.x >> 1];
  if (cl.u0 >= cl.u1) return;   // an idle cluster: both CTAs of the pair leave before any cluster step
  const int ntotal = cl.tiles;
  auto unit_tiles = [&](const AttUnit &u) { return (u.k1 - u.k0 + T - 1) / T; };

  if (threadIdx.x == 0) {
    mbar_init(b_qsfull, 1);
    mbar_init(b_qkdone, 1);
    mbar_init(b_qtdone, 8);   // softmax arrivals are one elected lane per warp (after __syncwarp)
    mbar_init(b_pvdone, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(kfull(s), FP8 ? 2 * kProdThreads : kProdThreads);   // fp8: stores and rope copies
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull(b), 1);
      mbar_init(sempty(b), 12);   // S tile b read by the 8 softmax and the 4 sender warps
      mbar_init(pfull(b), 8);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(xfull(b), 1);   // armed locally with the tile's bytes, filled by the partner's bulk copy
      mbar_init(xfree(b), 4);   // one arrival per partner softmax warp of half b
    }
    mbar_init(b_ofree, 8);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // One polling loop over the cluster's tiles: PV of the oldest softmaxed
    // tile or QK of the next, whichever is ready (PV first: it releases the
    // stage and the P columns; QK only runs ahead).  A unit's first QK waits
    // for its Q (rope and shared-memory columns by TMA, issued once the
    // previous unit's QKs completed; tensor-memory columns from the softmax
    // warps); its first PV waits until the previous unit's O has been read out.
    if (lane == 0) {
      auto load_q = [&](int row) {
        mbar_arrive_expect_tx(b_qsfull, C::QRBYTES + C::QS_CH * C::QCHUNK);
        tma_load_2d(sbase + C::OFF_QR, &p.tm_qp, static_cast<int>(crank) * C::RH, row * p.H, b_qsfull);
        for (int ch = C::QT_CH; ch < C::NPV; ++ch)
          tma_load_2d(sbase + C::OFF_QS + (ch - C::QT_CH) * C::QCHUNK, &p.tm_qn,
                      static_cast<int>(crank) * C::HALF + ch * 64, row * p.H, b_qsfull);
      };
      load_q(p.units[cl.u0].row);
      const uint32_t o_tmem = tmem_base + C::O_COL;
      // descriptors are built once; a K step of 16 columns adds 32 bytes (2
      // encoded), a stage adds STAGE / 16
      const uint64_t qrdesc = smem_desc(sbase + C::OFF_QR, 16, 512, kSwizzle64);
      const uint64_t qsdesc = smem_desc(sbase + C::OFF_QS, 16, 1024, kSwizzle128);
      const uint64_t kdesc0 = smem_desc(sbase + C::OFF_K, 16, 1024, kSwizzle128);
      const uint64_t krdesc0 = smem_desc(sbase + C::OFF_K + C::NPV * C::CHUNK, 16, 512, kSwizzle64);
      const uint64_t vdesc0 = smem_desc(sbase + C::OFF_K, C::CHUNK, 1024, kSwizzle128);
      constexpr uint64_t kStageStep = C::STAGE >> 4;
      int nq = 0, np = 0;                                 // QKs / PVs issued, over the cluster's tiles
      int uq = cl.u0, lq = 0, q_end = unit_tiles(p.units[cl.u0]);   // unit of the next QK, its index, its end
      int lp = 0, p_start = 0, p_end = q_end;                       // the same for the next PV
      int up = cl.u0;
      bool q_ready = false, q_pending = false;   // Q of unit lq in place; a Q load waits for unit lq-1's QKs
      bool ok = true;
      uint64_t idle_since = 0;
      uint32_t idle = 0;
      while (ok && np < ntotal) {
        bool progressed = false;
        if (np < nq && mbar_test(pfull(np & 1), (np >> 1) & 1) &&
            (np != p_start || lp == 0 || mbar_test(b_ofree, (lp - 1) & 1))) {
          tc_fence_after();
          const int st = np % NS;
          const uint32_t p_tmem = tmem_base + C::P_COL;
#pragma unroll
          for (int k = 0; k < T / 16; ++k)
            mma_f16_ts(o_tmem, p_tmem + k * 8, vdesc0 + st * kStageStep + (k * 16 * 128 >> 4), C::IDESC_PV,
                       (np > p_start || k > 0) ? 1u : 0u);
          mma_commit(b_pvdone);
          mma_commit(kempty(st));
          ++np;
          if (np == p_end && np < ntotal) {
            ++up;
            ++lp;
            p_start = np;
            p_end = np + unit_tiles(p.units[up]);
          }
          progressed = true;
        }
        if (q_pending && mbar_test(b_qkdone, (lq - 1) & 1)) {
          load_q(p.units[uq].row);   // the previous unit's QKs have read the old Q
          q_pending = false;
          progressed = true;
        }
        if (nq < ntotal) {
          if (!q_ready && !q_pending) q_ready = mbar_test(b_qsfull, lq & 1) && mbar_test(b_qtdone, lq & 1);
          const int st = nq % NS, sb = nq & 1;
          if (q_ready && mbar_test(kfull(st), (nq / NS) & 1) && mbar_test(sempty(sb), ((nq >> 1) & 1) ^ 1)) {
            fence_proxy_async_smem();   // the gathered tile feeds the tensor core
            tc_fence_after();
            const uint32_t s_tmem = tmem_base + C::S_COL + sb * T;
            const uint64_t kd = kdesc0 + st * kStageStep, krd = krdesc0 + st * kStageStep;
#pragma unroll
            for (int ch = 0; ch < C::QT_CH; ++ch)        // q_nope chunks in tensor memory
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_ts(s_tmem, tmem_base + ch * 32 + k * 8, kd + (ch * C::CHUNK >> 4) + 2 * k, C::IDESC_QK,
                           (ch | k) ? 1u : 0u);
#pragma unroll
            for (int ch = C::QT_CH; ch < C::NPV; ++ch)   // q_nope chunks in shared memory
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_ss(s_tmem, qsdesc + ((ch - C::QT_CH) * C::QCHUNK >> 4) + 2 * k,
                           kd + (ch * C::CHUNK >> 4) + 2 * k, C::IDESC_QK, 1u);
#pragma unroll
            for (int k = 0; k < 2; ++k)                  // rope columns in shared memory
              mma_f16_ss(s_tmem, qrdesc + 2 * k, krd + 2 * k, C::IDESC_QK, 1u);
            mma_commit(sfull(sb));
            ++nq;
            if (nq == q_end) {
              mma_commit(b_qkdone);   // the unit's QKs are issued: its Q may be replaced once they complete
              if (nq < ntotal) {
                ++uq;
                ++lq;
                q_end = nq + unit_tiles(p.units[uq]);
                q_ready = false;
                q_pending = true;
              }
            }
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
          idle_since = 0;
        } else {
          ++idle;
          __nanosleep(32);   // leave the issue slots to the other warps on this sub-partition
        }
        if (!progressed && (idle & 255) == 0) {
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
    // Warps 1-2 resolve a tile's rows (key = 32 * (warp - 1) + lane); the
    // selection entries of tile t+2 and the page ids of tile t+1 of the unit
    // are loaded while tile t is issued.  The stage ring runs on over the
    // cluster's tiles, so the next unit's gathers start while the current
    // unit finishes.
    const int pt = threadIdx.x - 32 * kProdWarp0;  // 0..223
    const bool resolver = warp < kProdWarp0 + 2;
    const int rkey = (warp - kProdWarp0) * 32 + lane;
    // Every exit from the tile loop is decided at the named barrier (an OR
    // over the producers), so no producer is left waiting there alone.
    // (`ok` is this thread's; `stop` is decided at the barrier, the same in
    // every producer, and alone ends the unit loop)
    bool ok = true, stop = false;
    int g = 0;   // the cluster's tile counter
    for (int ui = cl.u0; ui < cl.u1 && !stop; ++ui) {
      const AttUnit unit = p.units[ui];
      const int row = unit.row;
      const int pos = p.row_pos[row];
      const int nent = unit.k1 - unit.k0;
      const int ntiles = (nent + T - 1) / T;
      const int32_t *selrow = p.sel + static_cast<int64_t>(row) * p.K + unit.k0;
      const int page_off = p.row_page_off[row], npages = p.row_npages[row], page_start = p.row_page_start[row];
      auto sel_at = [&](int t) -> int {
        const int e = t * T + rkey;
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
      for (int t = 0; t < ntiles; ++t, ++g) {
        const int st = g % NS;
        const int pg1 = page_of(j1);
        const int j2 = sel_at(t + 2);
        if (!FP8 && ok) ok = mbar_wait(kempty(st), ((g / NS) & 1) ^ 1, abort_flag, p.err);
        int32_t *rows = rows_sm + st * T;
        if (resolver && ok) rows[rkey] = phys(j0, pg0);
        if (named_bar_any(2, kProdThreads, !ok)) {
          stop = true;
          break;
        }
        const uint32_t kst = sbase + C::OFF_K + st * C::STAGE;
        if constexpr (!FP8) {
          constexpr int ROWB = (L + R) * 2;
          // piece q of a key: this CTA's q_nope columns, then its rope columns.
          // Producer thread pt takes pieces pt, pt + 224, ...; the (key, piece)
          // pair advances by (224 / PIECES, 224 % PIECES) with a carry.
          constexpr int NIT = (T * C::PIECES + kProdThreads - 1) / kProdThreads;
          constexpr int DK = kProdThreads / C::PIECES, DP = kProdThreads % C::PIECES;
          int key = pt / C::PIECES, piece = pt - key * C::PIECES;
          const int off_nope = static_cast<int>(crank) * C::HALF * 2;
          const int off_rope = L * 2 + static_cast<int>(crank) * C::RH * 2 - C::NPV * 8 * 16;
#pragma unroll
          for (int u = 0; u < NIT; ++u) {
            if (u + 1 < NIT || key < T) {
              const int32_t prow = rows[key];
              const bool rope = piece >= C::NPV * 8;
              const uint32_t dst = rope ? kst + C::NPV * C::CHUNK + sw64_offset(key, piece - C::NPV * 8)
                                        : kst + (piece >> 3) * C::CHUNK + sw128_offset(key, piece & 7);
              const int off = (rope ? off_rope : off_nope) + piece * 16;
              const uint8_t *src = p.latent + (prow >= 0 ? static_cast<int64_t>(prow) * ROWB + off : 0);
              cp_async_16_zfill(dst, src, prow >= 0 ? 16u : 0u);
            }
            piece += DP;
            key += DK;
            if (piece >= C::PIECES) {
              piece -= C::PIECES;
              ++key;
            }
          }
          cp_async_mbar_arrive(kfull(st));
        } else {
          // 656-byte rows [L e4m3 | L/128 fp32 scales | R bf16]: this CTA's
          // codes (CPH 16-byte pieces a key) and their scales are loaded into
          // registers before the stage is known to be free, dequantised (code
          // x scale, rounded to bf16) and stored as the bf16 tile.  The rope
          // half (RP pieces, already bf16) is copied straight into the stage
          // by cp.async once it is free: the full barrier then counts each
          // producer twice (its stores, its copies).  Register loads are what
          // holds a producer up (every barrier, fence and release arrive
          // waits for them), so only the pieces that need arithmetic take
          // that path.
          constexpr int CPH = C::HALF / 16, RP = 4;
          constexpr int RB8 = L + 4 * (L / 128) + 2 * R;
          constexpr int PER = (T * CPH + kProdThreads - 1) / kProdThreads;
          uint4 raw[PER];
          float scl[PER];
#pragma unroll
          for (int u = 0; u < PER; ++u) {
            const int i = pt + u * kProdThreads;
            raw[u] = make_uint4(0, 0, 0, 0);
            scl[u] = 0.f;
            if (i < T * CPH) {
              const int key = i / CPH, k = i - key * CPH;
              const int32_t prow = rows[key];
              if (prow >= 0) {
                const uint8_t *base = p.latent + static_cast<int64_t>(prow) * RB8;
                raw[u] = __ldg(reinterpret_cast<const uint4 *>(base + static_cast<int>(crank) * C::HALF + 16 * k));
                scl[u] = __ldg(reinterpret_cast<const float *>(base + L) + (static_cast<int>(crank) * C::HALF) / 128 +
                               k / 8);
              }
            }
          }
          ok = mbar_wait(kempty(st), ((g / NS) & 1) ^ 1, abort_flag, p.err);
          if (ok) {
            for (int idx = pt; idx < T * RP; idx += kProdThreads) {
              const int key = idx / RP, piece = idx - key * RP;
              const int32_t prow = rows[key];
              const uint8_t *src = p.latent + (prow >= 0 ? static_cast<int64_t>(prow) * RB8 + L + 4 * (L / 128) +
                                                               static_cast<int>(crank) * C::RH * 2 + 16 * piece
                                                         : 0);
              cp_async_16_zfill(kst + C::NPV * C::CHUNK + sw64_offset(key, piece), src, prow >= 0 ? 16u : 0u);
            }
            cp_async_mbar_arrive(kfull(st));
          }
#pragma unroll
          for (int u = 0; u < PER; ++u) {
            const int i = pt + u * kProdThreads;
            if (!ok || i >= T * CPH) continue;
            const int key = i / CPH, k = i - key * CPH;
            // a piece is two 16-byte bf16 units of its key's 128-byte row;
            // pieces in odd chunks store their upper unit first, so that
            // the eight pieces of a store phase cover eight different units
            const int par = (k >> 2) & 1;
            uint4 r = raw[u];
            if (par) r = make_uint4(r.z, r.w, r.x, r.y);
            uint4 first, second;
            e4m3x16_to_bf16(r, scl[u], first, second);
            const uint32_t chunk = kst + (k / 4) * C::CHUNK;
            st_shared_v4(chunk + sw128_offset(key, (k % 4) * 2 + par), first);
            st_shared_v4(chunk + sw128_offset(key, (k % 4) * 2 + (par ^ 1)), second);
          }
          fence_proxy_async_smem();
          if (ok) mbar_arrive(kfull(st));
        }
        j0 = j1;
        j1 = j2;
        pg0 = pg1;
      }
    }
    cp_async_wait<0>();   // nothing in flight when the CTA leaves
  } else if (warp >= kSendWarp0) {
    // ------------------------------------------------------------ senders
    // Warp q (heads 32q..32q+31) sends its rows of this CTA's partial logits
    // of every tile, as soon as its QK is done, in two halves of 32 keys: a
    // half is staged in the warp's 4 KB x_out slot (row h's 16-byte chunks
    // swizzled by h) and bulk-copied into the same half of the partner's x_in
    // once all four partner softmax warps have merged that half of tile u-1
    // (a bulk copy lands ~1 us sooner than the same bytes sent by st.async
    // from registers).  The S tile is released (sempty) once its values are
    // in registers.  Tiles are counted over the cluster's units.
    const int quad = warp & 3;
    const int h = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t slot = sbase + C::OFF_X + C::XBYTES + quad * (C::XOUT / 4);
    const uint32_t dst0 = map_to_cta(sbase + C::OFF_X, peer) + static_cast<uint32_t>(quad * 32) * 128;
    bool ok = true;
    for (int u = 0; u < ntotal && ok; ++u) {
      const int b = u & 1;
      const uint32_t use = static_cast<uint32_t>(u >> 1);
      // warp-uniform, as the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(sfull(b), use & 1, abort_flag, p.err))) break;
      tc_fence_after();
      float v[T];
#pragma unroll
      for (int c0 = 0; c0 < T; c0 += 16)
        tmem_ld16(tmem_base + lane_base + C::S_COL + b * T + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty(b));
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (lane == 0) bulk_wait_read_all();   // the slot's previous copy has been read
        __syncwarp();
        const uint32_t r = slot + lane * 128;
#pragma unroll
        for (int c = 0; c < T / 8; ++c) {
          const int k = hh * (T / 2) + 4 * c;
          st_shared_v4(r + ((c ^ (h & 7)) << 4), make_uint4(__float_as_uint(v[k]), __float_as_uint(v[k + 1]),
                                                           __float_as_uint(v[k + 2]), __float_as_uint(v[k + 3])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        int sent_ok = 1;
        if (lane == 0) {
          sent_ok = mbar_wait<true>(xfree(hh), (static_cast<uint32_t>(u) & 1) ^ 1, abort_flag, p.err) ? 1 : 0;
          if (sent_ok) {
            bulk_copy_to_cta(dst0 + hh * C::XHALF, slot, C::XOUT / 4, map_to_cta(xfull(hh), peer));   // 32 rows of 128 bytes
            bulk_commit();
          }
        }
        if (__shfl_sync(0xffffffffu, sent_ok, 0) == 0) {
          ok = false;
          break;
        }
      }
    }
    if (lane == 0) bulk_wait_read_all();   // x_out stays valid until every copy has read it
  } else {
    // ------------------------------------------------------------ softmax
    // Two warps per TMEM lane quadrant: warp half hf takes keys 32hf..32hf+31
    // of every tile (the half of x_in the partner sends for them) and output
    // columns [hf, hf+1) * HALF/2.  The pair shares each tile's maximum
    // through shared memory, so both take the same reference max, and adds
    // its row sums at the end of each unit; every exit from the tile loop is
    // decided at the pair's barrier (an OR of their failures).  Per unit: the
    // unit's tiles, then (once its last S has been read, so every QK of the
    // unit has completed) the next unit's q_nope columns from global memory
    // into tensor memory, then this unit's O read out and written.
    const int quad = warp & 3;
    const int hf = (warp - kSoftWarp0) >> 2;
    const int h = quad * 32 + lane;                      // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t pair_bar = 3 + quad;
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);   // [t&1][hf][h] maxima, then [unit&1][hf][h] sums
    // this head's row of the tensor-memory q_nope columns (bf16 pairs, lower
    // column in the low half); the pair's warps take alternate chunks
    auto move_q = [&](int row) {
      const bool in = h < p.H;
#pragma unroll 1
      for (int ch = hf; ch < C::QT_CH; ch += 2) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            p.qn + (static_cast<int64_t>(row) * p.H + (in ? h : 0)) * L + static_cast<int>(crank) * C::HALF + ch * 64);
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = in ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * i] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st32(tmem_base + lane_base + ch * 32, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qtdone);
    };
    constexpr int TH = T / 2;                            // keys of a tile per warp
    move_q(p.units[cl.u0].row);
    bool ok = true;
    int g = 0;   // the cluster's tile counter
    for (int ui = cl.u0, lu = 0; ui < cl.u1 && ok; ++ui, ++lu) {
      const AttUnit unit = p.units[ui];
      const int row = unit.row;
      const int pos = p.row_pos[row];
      const int nent = unit.k1 - unit.k0;
      const int ntiles = (nent + T - 1) / T;
      const int32_t *selrow = p.sel + static_cast<int64_t>(row) * p.K + unit.k0;
      float m_ref = kNegBig, l = 0.f;
      int jn = hf * TH + lane < nent ? selrow[hf * TH + lane] : -1;
      for (int t = 0; t < ntiles; ++t, ++g) {
        const uint32_t vmask = __ballot_sync(0xffffffffu, jn >= 0 && jn <= pos);
        if (t + 1 < ntiles) {
          const int e = (t + 1) * T + hf * TH + lane;
          jn = e < nent ? selrow[e] : -1;
        }
        const int sb = g & 1;
        const uint32_t use = static_cast<uint32_t>(g >> 1);
        if (h == 0) mbar_arrive_expect_tx(xfull(hf), C::XHALF);
        bool good = ok && __all_sync(0xffffffffu, mbar_wait(sfull(sb), use & 1, abort_flag, p.err));
        tc_fence_after();
        float s[TH];
        if (good) {
#pragma unroll
          for (int c0 = 0; c0 < TH; c0 += 16)
            tmem_ld16(tmem_base + lane_base + C::S_COL + sb * T + hf * TH + c0,
                      *reinterpret_cast<float(*)[16]>(s + c0));
          tmem_ld_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (good && lane == 0) mbar_arrive(sempty(sb));   // our partial is in registers: the S tile can take QK of tile g+2
        // full logits of this warp's keys: our partial + the partner's (x_in half hf)
        good = good && __all_sync(0xffffffffu,
                                  mbar_wait<true>(xfull(hf), static_cast<uint32_t>(g) & 1, abort_flag, p.err));
        float lmax = -INFINITY;
        if (good) {
          const float4 *xr = reinterpret_cast<const float4 *>(smem + C::OFF_X + hf * C::XHALF + h * 128);
#pragma unroll
          for (int c = 0; c < TH / 4; ++c) {
            const float4 v = xr[c ^ (h & 7)];
            // a + b == b + a in IEEE arithmetic: both CTAs get the same S
            f2_unpack(f2_add(f2_pack(s[4 * c], s[4 * c + 1]), f2_pack(v.x, v.y)), s[4 * c], s[4 * c + 1]);
            f2_unpack(f2_add(f2_pack(s[4 * c + 2], s[4 * c + 3]), f2_pack(v.z, v.w)), s[4 * c + 2], s[4 * c + 3]);
          }
          // (scale_log2 > 0, so the max of the raw logits picks the same key)
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < TH; ++i) {
            s[i] = ((vmask >> i) & 1u) ? s[i] : -INFINITY;
            mx[i & 3] = fmaxf(mx[i & 3], s[i]);
          }
          lmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        }
        // this warp's rows of its x_in half have been read (a release arrive
        // here costs more than it saves)
        __syncwarp();
        if (good && lane == 0) mbar_arrive_remote_relaxed(map_to_cta(xfree(hf), peer));
        red[(sb * 2 + hf) * 128 + h] = lmax;
        if (named_bar_any(pair_bar, 64, !good)) {   // both halves' maxima are in place
          ok = false;
          break;
        }
        // online softmax in base 2 with a lazily moved reference max
        const float tmax = fmaxf(red[(sb * 2) * 128 + h], red[(sb * 2 + 1) * 128 + h]) * p.scale_log2;
        float alpha = 1.f;
        const bool rescale = tmax > m_ref + kRescaleThreshold;
        if (rescale) {
          alpha = fast_exp2(m_ref - tmax);
          m_ref = tmax;
        }
        // P (bf16 pairs, lower key in the low half) for this warp's keys; the
        // row sum takes the fp32 probabilities before their bf16 rounding (no
        // conversion back per key), in four partial sums (key pair k into
        // sum k mod 4) held as two pairs for the packed adds
        uint64_t sm01 = 0, sm23 = 0;
        uint32_t packed[TH / 2];
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_ref, -m_ref);
#pragma unroll
        for (int i = 0; i < TH; i += 8) {
          float x[8];
#pragma unroll
          for (int j = 0; j < 8; j += 2) f2_unpack(f2_fma(f2_pack(s[i + j], s[i + j + 1]), sc2, nm2), x[j], x[j + 1]);
          float2 pf[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            pf[j] = make_float2(fast_exp2(x[2 * j]), fast_exp2(x[2 * j + 1]));
            const __nv_bfloat162 pb = __floats2bfloat162_rn(pf[j].x, pf[j].y);
            packed[i / 2 + j] = *reinterpret_cast<const uint32_t *>(&pb);
          }
          sm01 = f2_add(sm01, f2_add(f2_pack(pf[0].x, pf[1].x), f2_pack(pf[0].y, pf[1].y)));
          sm23 = f2_add(sm23, f2_add(f2_pack(pf[2].x, pf[3].x), f2_pack(pf[2].y, pf[3].y)));
        }
        float sm[4];
        f2_unpack(sm01, sm[0], sm[1]);
        f2_unpack(sm23, sm[2], sm[3]);
        l = l * alpha + ((sm[0] + sm[1]) + (sm[2] + sm[3]));
        // PV of tile g-1 (of this unit or the one before) must be done before
        // P is overwritten, and before O is rescaled (PV of g-2 finished
        // before PV of g-1 was issued); a failure here is seen at the next
        // pair barrier
        if (g > 0) {
          good = __all_sync(0xffffffffu, mbar_wait(b_pvdone, (g - 1) & 1, abort_flag, p.err));
          tc_fence_after();
        }
        // the O loads and stores are warp-collective: the warp rescales when
        // any of its heads needs it (alpha is exactly 1 for the others); the
        // unit's first tile has no O yet
        if (good && t > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c0 = 0; c0 < C::HALF / 2; c0 += 16) {
            float o[16];
            tmem_ld16(tmem_base + lane_base + C::O_COL + hf * (C::HALF / 2) + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 2)
              f2_unpack(f2_mul(f2_pack(o[i], o[i + 1]), f2_pack(alpha, alpha)), o[i], o[i + 1]);
            tmem_st16(tmem_base + lane_base + C::O_COL + hf * (C::HALF / 2) + c0, o);
          }
        }
        if (good) {
          tmem_st16(tmem_base + lane_base + C::P_COL + hf * (TH / 2), *reinterpret_cast<const float(*)[16]>(packed));
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (good && lane == 0) mbar_arrive(pfull(sb));
        ok = good;
      }
      if (!ok) break;
      // every QK of this unit has completed (its last S was read): the next
      // unit's q_nope columns can replace this unit's in tensor memory
      if (ui + 1 < cl.u1) move_q(p.units[ui + 1].row);
      ok = __all_sync(0xffffffffu, mbar_wait(b_pvdone, (g - 1) & 1, abort_flag, p.err));   // this unit's last PV
      tc_fence_after();
      // the row sum is the two halves' sums (in a fixed order, the same in
      // both CTAs); the sums alternate between two slots by unit.  The pair's
      // barrier also makes `ok` the same in both warps, so they leave the
      // unit loop together.
      float *rsum = red + (4 + 2 * (lu & 1)) * 128;
      rsum[hf * 128 + h] = l;
      ok = !named_bar_any(pair_bar, 64, !ok);
      l = rsum[h] + rsum[128 + h];
      // (ok is warp-uniform and every lane takes its row out of TMEM, since the
      // loads are warp-collective; only heads below H are stored)
      const bool store = h < p.H;
      if (ok) {
        const int col0 = static_cast<int>(crank) * C::HALF + hf * (C::HALF / 2);
        const uint32_t ocol = C::O_COL + hf * (C::HALF / 2);
        if (unit.slot < 0) {
          float f = 0.f;
          if (p.sink && store) {
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
          for (int c0 = 0; c0 < C::HALF / 2; c0 += 16) {
            float o[16];
            __syncwarp();   // converged for the warp-collective load
            tmem_ld16(tmem_base + lane_base + ocol + c0, o);
            tmem_ld_wait();
            if (!store) continue;
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
          for (int c0 = 0; c0 < C::HALF / 2; c0 += 16) {
            float o[16];
            __syncwarp();   // converged for the warp-collective load
            tmem_ld16(tmem_base + lane_base + ocol + c0, o);
            tmem_ld_wait();
            if (!store) continue;
            float4 *d4 = reinterpret_cast<float4 *>(dst + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
          if (crank == 0 && hf == 0 && store) {
            float *ml = p.mlpart + (static_cast<int64_t>(unit.slot) * p.H + h) * 2;
            ml[0] = m_ref;
            ml[1] = l;
          }
        }
      }
      // O is free for the next unit's first PV
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the partner sends nothing more into this CTA's shared memory
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Merge of split rows: o = sum_s 2^(m_s - m) O_s / (sum_s 2^(m_s - m) l_s [+ 2^(sink - m)]).
// A block takes kCombHeads heads of one merged row: one thread per head turns
// the pieces' (m, l) into per-piece weights in shared memory, then the block
// streams those heads' columns, four at a time (a float4 of each piece's
// partial, then four bf16 out).
// ---------------------------------------------------------------------------
constexpr int kCombHeads = 8;
constexpr int kCombThreads = 256;

__global__ void __launch_bounds__(kCombThreads, 4) attend_combine_kernel(const AttCombine *__restrict__ combine,
                                                                     const float *__restrict__ opart,
                                                                     const float *__restrict__ mlpart,
                                                                     const float *__restrict__ sink,
                                                                     __nv_bfloat16 *out, int H, int L, int n_merge,
                                                                     const int32_t *__restrict__ n_merge_dev) {
  __shared__ float wsm[kCombHeads][kAttMaxPieces];
  __shared__ float invl[kCombHeads];
  // (merge, group of kCombHeads heads) pairs; a capturable plan's merge count is on the device
  const int hb = (H + kCombHeads - 1) / kCombHeads;
  const int n_work = (n_merge_dev ? *n_merge_dev : n_merge) * hb;
  for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
    const AttCombine cb = combine[w / hb];
    const int h0 = (w % hb) * kCombHeads;
    if (cb.row < 0) continue;   // padding of a capturable plan (uniform over the block)
    const int ns = cb.nsplit < kAttMaxPieces ? cb.nsplit : kAttMaxPieces;
    if (ns == 2) {
      // a row split in two (the usual case): every thread derives its heads'
      // weights itself, and its loads (both pieces' O and (max, sum) of two
      // float4 groups at a time) go out together
      const int L4 = L / 4, total = kCombHeads * L4;
      const float *o0 = opart + static_cast<int64_t>(cb.first_slot) * H * L;
      const float *o1 = o0 + static_cast<int64_t>(H) * L;
      const float2 *ml0 = reinterpret_cast<const float2 *>(mlpart) + static_cast<int64_t>(cb.first_slot) * H;
      const float2 *ml1 = ml0 + H;
      for (int e0 = threadIdx.x; e0 < total; e0 += 2 * kCombThreads) {
        float4 a[2], b[2];
        float2 ma[2], mb[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int e = e0 + k * kCombThreads;
          const int hh = e / L4, d = (e - hh * L4) * 4, h = h0 + hh;
          if (e < total && h < H) {
            a[k] = *reinterpret_cast<const float4 *>(o0 + static_cast<int64_t>(h) * L + d);
            b[k] = *reinterpret_cast<const float4 *>(o1 + static_cast<int64_t>(h) * L + d);
            ma[k] = ml0[h];
            mb[k] = ml1[h];
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int e = e0 + k * kCombThreads;
          const int hh = e / L4, d = (e - hh * L4) * 4, h = h0 + hh;
          if (e >= total || h >= H) continue;
          float m = sink ? sink[h] * kLog2e : -INFINITY;
          m = fmaxf(m, ma[k].x);
          m = fmaxf(m, mb[k].x);
          const float wa = exp2f(ma[k].x - m), wb = exp2f(mb[k].x - m);
          float lsum = sink ? exp2f(sink[h] * kLog2e - m) : 0.f;
          lsum = fmaf(wa, ma[k].y, lsum);
          lsum = fmaf(wb, mb[k].y, lsum);
          const float f = lsum > 0.f ? 1.f / lsum : 0.f;
          float4 acc;
          acc.x = fmaf(wb, b[k].x, wa * a[k].x);
          acc.y = fmaf(wb, b[k].y, wa * a[k].y);
          acc.z = fmaf(wb, b[k].z, wa * a[k].z);
          acc.w = fmaf(wb, b[k].w, wa * a[k].w);
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f),
                               hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
          *reinterpret_cast<uint2 *>(out + (static_cast<int64_t>(cb.row) * H + h) * L + d) =
              make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
        }
      }
      continue;
    }
    __syncthreads();   // the previous item's weights have been used
    if (threadIdx.x < kCombHeads && h0 + static_cast<int>(threadIdx.x) < H) {
      const int h = h0 + threadIdx.x;
      float m = sink ? sink[h] * kLog2e : -INFINITY;
      for (int s = 0; s < ns; ++s) m = fmaxf(m, mlpart[((cb.first_slot + s) * static_cast<int64_t>(H) + h) * 2]);
      float lsum = sink ? exp2f(sink[h] * kLog2e - m) : 0.f;
      for (int s = 0; s < ns; ++s) {
        const float *ml = mlpart + ((cb.first_slot + s) * static_cast<int64_t>(H) + h) * 2;
        const float ws = exp2f(ml[0] - m);
        wsm[threadIdx.x][s] = ws;
        lsum += ws * ml[1];
      }
      invl[threadIdx.x] = lsum > 0.f ? 1.f / lsum : 0.f;
    }
    __syncthreads();
    const int ngroups = kCombHeads * (L / 4);
    for (int e = threadIdx.x; e < ngroups; e += kCombThreads) {
      const int hh = e / (L / 4), d = (e - hh * (L / 4)) * 4;
      const int h = h0 + hh;
      if (h >= H) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < ns; ++s) {
        const float4 v = *reinterpret_cast<const float4 *>(opart + ((cb.first_slot + s) * static_cast<int64_t>(H) + h) * L + d);
        const float ws = wsm[hh][s];
        acc.x = fmaf(ws, v.x, acc.x);
        acc.y = fmaf(ws, v.y, acc.y);
        acc.z = fmaf(ws, v.z, acc.z);
        acc.w = fmaf(ws, v.w, acc.w);
      }
      const float f = invl[hh];
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f), hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
      *reinterpret_cast<uint2 *>(out + (static_cast<int64_t>(cb.row) * H + h) * L + d) =
          make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
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
  if (pos < 0) return;   // padding row of a capturable plan
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
                       static_cast<uint64_t>(plan->T) * c.heads, 64 * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  prm.qn = static_cast<const __nv_bfloat16 *>(q_nope);
  prm.sel = sel;
  prm.latent = static_cast<const uint8_t *>(latent);
  prm.sink = sink;
  prm.units = plan->units;
  prm.clusters = plan->clusters;
  prm.row_pos = plan->row_pos;
  prm.row_page_off = plan->row_page_off;
  prm.row_npages = plan->row_npages;
  prm.row_page_start = plan->row_page_start;
  prm.pages = plan->pages;
  prm.out = static_cast<__nv_bfloat16 *>(out);
  prm.opart = plan_opart(ctx, plan);
  prm.mlpart = plan_mlpart(ctx, plan);
  prm.err = ctx->err;
  prm.H = c.heads;
  prm.K = c.topk;
  prm.P = c.page_size;
  prm.num_pages = plan->cache_pages;
  prm.scale_log2 = sm_scale * kLog2e;
  auto kern = attend_tc_kernel<L, FP8>;
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(kern, Cfg::SMEM, ctx->device, smem_limit_set); e != cudaSuccess) return e;
  if (plan->n_clusters <= 0) return cudaSuccess;
  kern<<<2 * plan->n_clusters, kAttThreads, Cfg::SMEM, s>>>(prm);
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
      // a capturable plan's merge count is known only on the device: a grid
      // that strides over its (merge, head) pairs
      const int hb = (c.heads + kCombHeads - 1) / kCombHeads;
      const int grid = plan->capturable ? std::min(plan->n_combine * hb, ctx->num_sms * 8) : plan->n_combine * hb;
      attend_combine_kernel<<<grid, kCombThreads, 0, s>>>(plan->combine, plan_opart(ctx, plan), plan_mlpart(ctx, plan),
                                                          sink, static_cast<__nv_bfloat16 *>(out), c.heads,
                                                          c.kv_lora_rank, plan->n_combine,
                                                          plan->capturable ? plan->counts + 3 : nullptr);
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
