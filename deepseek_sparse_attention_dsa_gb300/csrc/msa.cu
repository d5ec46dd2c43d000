// msa.cu -- block-sparse MSA on sm_103a: block selection and GQA attention
// over the selected blocks.
//
// LLMServingSim, "Sparse attention (DSA and block-sparse MSA)", table "Two
// shapes, three checkpoints", MiniMax-M3 column: every row keeps the top 16
// blocks of 128 tokens and attends over them with plain GQA; the index cache
// holds one bf16 vector per token.  The pages give no block-scoring formula;
// the reading built here: a token's score is the DSA indexer score over its
// index vector (index_tc_kernel, unchanged), a block's score is the largest
// score among the positions the row sees, the selection is the causal top-k
// over blocks with ties to the lower block, and attention covers the
// positions <= the row's own in the kept blocks.
//
// msa_select_kernel: one CTA per row; warps take blocks and reduce their
// scores to order-preserving 32-bit keys (redux.sync max), or read the block
// maxima the indexer's block-maximum epilogue left.  Rows of up to 256
// blocks rank each block by counting the blocks that beat it; longer rows
// take four 8-bit radix passes to find the topk_blocks-th largest key tau,
// and two block scans over contiguous runs of blocks write every block above
// tau and the lowest blocks equal to it (ties to the lower block), in
// ascending order either way.
//
// msa_attend_tc_kernel (block_size 128, head_dim 128): a persistent grid, one
// CTA per SM walking its rows (every grid-th row) as a run of (tile, kv head)
// steps.  A tile is 128 positions, one UMMA M:
//     S^T[token, head] = K[token, :] . Q_g[head, :]      (M = 128 tokens, N = group heads padded to 16)
//     O^T_g[dim, head] += V[:, dim]^T . P^T[:, head]     (M = 128 dims, A = V read MN-major, B = P^T)
// Warp 10 builds each row's tile list (kept blocks in ascending order) up to
// two rows ahead, warp 0 issues the TMA loads of a step's K and V boxes (the
// paged cache as a 2-D tensor, 128-byte swizzle) into a ring of stages that
// runs on across rows, warp 1 issues the MMAs (QK of step t+1 before PV of
// step t waits for its P; the next row's QKs start while the current row
// drains), and eight
// softmax warps, two per TMEM lane quadrant (thread = TMEM lane = token of S,
// dim of O; each warp of a pair takes half of the heads), reduce each head's
// maximum and sum with halving shuffle exchanges (one transposing pass per
// reduction, not one butterfly per head), keep a per-head
// reference max that moves only when it grows by more than 2^8 (O is then
// rescaled in TMEM), write P^T as bf16 in the 128-byte-swizzled K-major
// layout, and normalise a row's output at the start of their next row.  Tiles start on the box boundary below
// the span's page_start (as the indexer's key tiles do): with page_start a
// multiple of the box height a tile is exactly one block, otherwise a block
// spans two tiles and rows outside the kept blocks are masked (their V rows
// are zeroed before PV so no stale value meets a zero probability).
//
// msa_attend_simt_kernel covers other shapes: one CTA per (row, query head),
// fp32 on CUDA cores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr float kMsaLog2e = 1.4426950408889634f;
constexpr float kMsaRescale = 8.0f;         // log2 units the reference max may lag the true max
constexpr float kMsaNegBig = -1.0e30f;

constexpr int kSelThreads = 512;
constexpr int kSelMaxBlocks = 16384;          // blocks per row held in shared memory
constexpr int kSelRankBlocks = 256;           // rows with at most this many blocks rank by counting
static_assert(kSelRankBlocks <= kSelThreads, "one block per thread when ranking by counting");
constexpr int kMsaMaxK = 64;                  // topk_blocks
constexpr int kMsaTile = 128;                 // positions per tile (UMMA M)
constexpr int kMsaMaxTiles = 2 * kMsaMaxK;
constexpr int kMsaThreads = 352;              // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two per lane quadrant), warp 10 tile lists
constexpr int kMsaListWarp = 10;
constexpr int kMsaSoftThreads = 256;
constexpr int kMsaMaxKvHeads = 8;

__device__ __forceinline__ uint32_t score_key(float f) { return score_order_key(f); }
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---------------------------------------------------------------------------
// block selection
// ---------------------------------------------------------------------------
// Exclusive prefix sum of one int per thread over the kSelThreads threads of
// the block (ws: kSelThreads / 32 + 1 words; ends with a barrier, so ws is
// free again on return).
__device__ __forceinline__ int sel_block_scan(int v, int *ws, int warp, int lane) {
  constexpr int kWarps = kSelThreads / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kWarps ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) ws[lane] = t - ws[lane];   // exclusive per-warp offsets
  }
  __syncthreads();
  const int r = ws[warp] + x - v;
  __syncthreads();
  return r;
}

// `block_keys` non-null: the block maxima come ready from the indexer's
// block-maximum epilogue (row r's at block_key_base), and `scores` is unused.
__global__ void __launch_bounds__(kSelThreads) msa_select_kernel(const float *__restrict__ scores,
                                                                 const uint32_t *__restrict__ block_keys,
                                                                 const int64_t *__restrict__ row_score_off,
                                                                 const int32_t *__restrict__ row_pos, int T, int bs,
                                                                 int K, int32_t *__restrict__ sel) {
  extern __shared__ uint32_t bkey[];   // [kSelMaxBlocks] block keys (every score's key is above 0)
  __shared__ int hist[256];
  __shared__ int scan_ws[kSelThreads / 32 + 1];
  __shared__ uint32_t sel_prefix;
  __shared__ int sel_kleft;
  constexpr int kWarps = kSelThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    const int pos = row_pos[row];
    if (pos < 0) continue;   // padding row (uniform over the CTA)
    const int nblk = pos / bs + 1;
    if (nblk <= K) {   // every block is kept: nothing to rank
      int32_t *out = sel + static_cast<int64_t>(row) * K;
      for (int i = threadIdx.x; i < K; i += kSelThreads) out[i] = i < nblk ? i : -1;
      continue;
    }
    if (block_keys) {
      const uint32_t *bk = block_keys + block_key_base(row_score_off[row], row, bs);
      for (int b = threadIdx.x; b < nblk; b += kSelThreads) bkey[b] = bk[b];
    }
    const float *s = block_keys ? nullptr : scores + row_score_off[row];
    // block maxima: warp w takes blocks w, w + kWarps, ...; four blocks per
    // pass keep their loads in flight together
    for (int b0 = block_keys ? nblk : warp; b0 < nblk; b0 += 4 * kWarps) {
      uint32_t m[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b = b0 + u * kWarps;
        m[u] = 0u;
        if (b < nblk) {
          const int j0 = b * bs, j1 = min(j0 + bs - 1, pos);
          for (int j = j0 + lane; j <= j1; j += 32) m[u] = max(m[u], score_key(__ldg(s + j)));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b = b0 + u * kWarps;
        const uint32_t mu = __reduce_max_sync(0xffffffffu, m[u]);
        if (lane == 0 && b < nblk) bkey[b] = mu;
      }
    }
    __syncthreads();
    int32_t *out = sel + static_cast<int64_t>(row) * K;
    if (nblk <= kSelRankBlocks) {
      // few blocks: thread i ranks block i by counting the blocks that beat
      // it (a larger key, or the same key at a lower block), and one block
      // scan gives the kept blocks their slots in block order
      bool take = false;
      if (static_cast<int>(threadIdx.x) < nblk) {
        const uint32_t ki = bkey[threadIdx.x];
        int rank = 0;
        for (int j = 0; j < nblk; ++j) {
          const uint32_t kj = bkey[j];
          rank += (kj > ki || (kj == ki && j < static_cast<int>(threadIdx.x))) ? 1 : 0;
        }
        take = rank < K;
      }
      const int slot = sel_block_scan(take ? 1 : 0, scan_ws, warp, lane);
      if (take && slot < K) out[slot] = static_cast<int>(threadIdx.x);
      continue;   // (the scan ended on a barrier: bkey is free for the next row)
    }
    // tau = the K-th largest key: four 8-bit radix passes from the top, each
    // over the keys that share the digits found so far
    uint32_t prefix = 0u, pmask = 0u;
    int kleft = K;   // keys still to take among those matching prefix
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      // (block maxima of one row share their leading digits: the lanes of a
      // warp with the same digit add once, by their lowest lane)
      for (int i0 = 0; i0 < nblk; i0 += kSelThreads) {
        const int i = i0 + static_cast<int>(threadIdx.x);
        const uint32_t k = i < nblk ? bkey[i] : 0u;
        const bool act = i < nblk && (k & pmask) == prefix;
        const uint32_t d = act ? (k >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (act && __ffs(peers) - 1 == lane) atomicAdd(&hist[d], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds digits 8l..8l+7; above[l] = keys with a digit of a higher lane
        int c[8], tot = 0;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          c[d] = hist[8 * lane + d];
          tot += c[d];
        }
        // suffix sum over the lanes: incl = keys with a digit in this lane or above
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, incl, o);
          if (lane + o < 32) incl += y;
        }
        int acc = incl - tot;
        if (acc < kleft && kleft <= incl) {
#pragma unroll
          for (int d = 7; d >= 0; --d) {
            if (acc + c[d] >= kleft) {
              sel_prefix = prefix | (static_cast<uint32_t>(8 * lane + d) << shift);
              sel_kleft = kleft - acc;
              break;
            }
            acc += c[d];
          }
        }
      }
      __syncthreads();
      prefix = sel_prefix;
      kleft = sel_kleft;
      pmask |= 255u << shift;
    }
    // the chosen blocks: every key above tau, and the kleft lowest blocks
    // whose key equals tau; each thread takes a contiguous run of blocks so
    // two block scans give the tie ranks and the output slots in block order
    const uint32_t tau = prefix;
    const int per = (nblk + kSelThreads - 1) / kSelThreads;
    const int c0 = min(nblk, threadIdx.x * per), c1 = min(nblk, c0 + per);
    int n_eq = 0;
    for (int i = c0; i < c1; ++i) n_eq += bkey[i] == tau;
    int eq_before = sel_block_scan(n_eq, scan_ws, warp, lane);
    int n_take = 0;
    {
      int e = eq_before;
      for (int i = c0; i < c1; ++i) {
        const uint32_t k = bkey[i];
        if (k > tau) ++n_take;
        else if (k == tau) n_take += (e++ < kleft);
      }
    }
    const int slot0 = sel_block_scan(n_take, scan_ws, warp, lane);
    {
      int e = eq_before, o = slot0;
      for (int i = c0; i < c1; ++i) {
        const uint32_t k = bkey[i];
        const bool take = k > tau || (k == tau && e++ < kleft);
        if (take && o < K) out[o++] = i;
      }
    }
    __syncthreads();   // bkey, hist and the scan words are reused by the next row
  }
}

// ---------------------------------------------------------------------------
// GQA attention over the selected blocks, tensor cores
// ---------------------------------------------------------------------------
// 2^x with the MUFU approximation (relative error ~2^-22; the results feed
// bf16 probabilities and a lazily moved reference max).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Reduces over the warp N per-lane values (N = 8, 16 or 32) by halving
// exchanges: at each step a lane keeps half of its values and combines them
// with the partner's copy, so N - 1 + (5 - log2 N) shuffles replace 5 N.  The
// lane ends with the result for value (lane >> (5 - log2 N)): N = 8, lanes
// 4h..4h+3 hold value h; N = 16, lanes 2h and 2h+1; N = 32, lane h.
struct SumOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};
struct MaxOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
template <int N, class Op>
__device__ __forceinline__ float warp_reduce_transpose(const float (&in)[N], Op op) {
  static_assert(N == 8 || N == 16 || N == 32, "values per lane");
  float v[N];
#pragma unroll
  for (int k = 0; k < N; ++k) v[k] = in[k];
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = N, j = 4; c > 1; c >>= 1, --j) {
    const bool up = (lane >> j) & 1;
#pragma unroll
    for (int k = 0; k < c / 2; ++k) {
      const float send = up ? v[k] : v[k + c / 2];
      const float keep = up ? v[k + c / 2] : v[k];
      v[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 1 << j));
    }
  }
#pragma unroll
  for (int j = (N == 8 ? 1 : N == 16 ? 0 : -1); j >= 0; --j) v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1 << j));
  return v[0];
}
template <int N>
__device__ __forceinline__ float warp_sum_transpose(const float (&in)[N]) {
  return warp_reduce_transpose<N>(in, SumOp{});
}

struct MsaParams {
  CUtensorMap tm_kv;   // kv cache as [pages*P, 2*Hkv*128] bf16, box {64, BH}, 128-byte swizzle
  CUtensorMap tm_q;    // q as [T*Hq, 128] bf16, box {64, NG}, 128-byte swizzle
  const int32_t *sel;  // [T][K] block ids, -1 padded
  const int32_t *row_pos, *row_page_off, *row_npages, *row_page_start, *pages;
  __nv_bfloat16 *out;  // [T][Hq][128]
  int *err;
  int T, Hq, Hkv, group, K, P, BH, num_pages, stages;
  float scale_log2;    // sm_scale * log2(e)
};

constexpr int kMsaBars = 28;

// Shared-memory layout of one CTA (bytes from a 1024-aligned base).
struct MsaLayout {
  uint32_t off_q, off_p, off_red, off_ml, off_tiles, off_bar, off_misc, bytes;
  __host__ __device__ MsaLayout(int NG, int stages, int Hkv) {
    const uint32_t ch = kMsaTile * 128, stage = 4 * ch;   // K and V, two 64-column chunks each
    off_q = stages * stage;
    off_p = off_q + Hkv * 2 * NG * 128;
    off_red = off_p + 2 * 2 * NG * 128;
    off_ml = off_red + 4 * 8 * NG * 4;          // [group][step parity][max keys | sums][NG][4 quads]
    off_tiles = off_ml + 4 * Hkv * NG * 4;      // m [tile parity][Hkv][NG], l [row parity][Hkv][NG]
    off_bar = (off_tiles + 2 * 2 * kMsaMaxTiles * 4 + 7) / 8 * 8;   // [row parity][tile | flags][kMsaMaxTiles]
    off_misc = off_bar + kMsaBars * 8;
    bytes = off_misc + 16 + 1024;   // + alignment slack
  }
};

// The tile list of one row, built by a warp (every lane returns its length):
// the kept blocks in ascending order (rank placement: the selection may come
// in any order), each block's tile and, when the span's token 0 is off the
// box boundary, the tile holding the block's last `lead` positions.  tu and
// tf hold kMsaMaxTiles entries; the sorted blocks pass through tf's upper
// half (list entry n <= 2 i + 1 is written after sorted block i is read).
__device__ __forceinline__ int msa_row_tiles(const int32_t *sr, int K, int pos, int lead, int32_t *tu, int32_t *tf,
                                             int *err) {
  const int lane = threadIdx.x & 31;
  const int last = pos / kMsaTile;
  int b[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    int v = e < K ? sr[e] : -1;
    if (v < -1 || v > last) {
      atomicOr(err, kErrBounds);
      v = -1;
    }
    b[h] = v;
  }
  int rank[2] = {0, 0};
  for (int e = 0; e < 64; ++e) {
    const int v = __shfl_sync(0xffffffffu, b[e >> 5], e & 31);
    if (v < 0) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (b[h] >= 0 && (v < b[h] || (v == b[h] && e < lane + 32 * h))) ++rank[h];
  }
  int32_t *sorted = tf + kMsaMaxK;
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (b[h] >= 0) sorted[rank[h]] = b[h];
  const int nvalid = __reduce_add_sync(0xffffffffu, (b[0] >= 0 ? 1 : 0) + (b[1] >= 0 ? 1 : 0));
  __syncwarp();
  int n = 0;
  if (lane == 0) {
    for (int i = 0; i < nvalid; ++i) {
      const int blk = sorted[i];
      // tile blk holds the block's positions from row `lead` on (bit 1)
      if (n > 0 && tu[n - 1] == blk) tf[n - 1] |= 2;
      else { tu[n] = blk; tf[n] = 2; ++n; }
      // tile blk+1 holds its last `lead` positions in rows 0..lead-1 (bit 0)
      if (lead > 0 && kMsaTile * (blk + 1) - lead <= pos) {
        tu[n] = blk + 1;
        tf[n] = 1;
        ++n;
      }
    }
  }
  n = __shfl_sync(0xffffffffu, n, 0);
  __syncwarp();
  return n;
}

// O / l of one row into its output, by one softmax warp (thread = dim i):
// for the kv heads g = grp, grp + NGRP, ... the warp's NH heads from h0 on.
// ocol is this lane quadrant's tensor-memory address of the row's O for kv
// head 0, head h0; l_row the row's sums [Hkv][NG].
template <int NG, int NGRP, int NH>
__device__ __forceinline__ void msa_write_out(uint32_t ocol, const float *l_row, int Hkv, int grp, int h0, int group,
                                              __nv_bfloat16 *out_row, int i) {
  constexpr int CW = NH < 16 ? NH : 16;   // heads per tensor-memory load
  for (int g = grp; g < Hkv; g += NGRP) {
#pragma unroll
    for (int c0 = 0; c0 < NH; c0 += CW) {
      float o[CW];
      if constexpr (CW == 8) tmem_ld8(ocol + g * NG + c0, o);
      else tmem_ld16(ocol + g * NG + c0, o);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < CW; ++k) {
        const int h = h0 + c0 + k;
        if (h >= group) continue;
        const float l = l_row[g * NG + h];
        out_row[(g * group + h) * 128 + i] = __float2bfloat16_rn(l > 0.f ? o[k] / l : 0.f);
      }
    }
  }
}

// A persistent grid: CTA b takes rows b, b + grid, b + 2 grid, ... (padding
// rows of a capturable plan, pos < 0, are skipped by every role alike).  The
// stage ring, the S and P buffers and their barriers run on across rows
// (barrier parities follow the CTA's global step count), so the next row's
// loads and QKs start while the current row drains.  Each row's tile list is
// built by the producer into one of two buffers (row parity) and released by
// the MMA thread and the softmax warps once they are past the row; the row's
// Q is reloaded once the previous row's last QK has completed.  A row's
// output is written by its softmax warps at the start of their next row,
// while that row's first QK is on its way (its sums l are double-buffered by
// row parity; O has one buffer: a row's first PV into a kv head's columns
// needs a P that the warps owning that head write only after reading the
// previous row's O out).
template <int NG, int NGRP>
__global__ void __launch_bounds__(kMsaThreads, 1) msa_attend_tc_kernel(const __grid_constant__ MsaParams p) {
  constexpr int CH = kMsaTile * 128;        // [128 rows][64 columns] bf16
  constexpr int KVB = 2 * CH;               // K (or V) of one kv head
  constexpr int STAGE = 2 * KVB;
  constexpr int QG = 2 * NG * 128;          // Q of one kv head: 2 chunks [NG heads][64 dims]
  constexpr int PB = 2 * NG * 128;          // P^T: 2 chunks [NG heads][64 tokens]
  constexpr uint32_t IDESC_QK = mma_idesc(128, NG, 1u, false, false);
  constexpr uint32_t IDESC_PV = mma_idesc(128, NG, 1u, true, false);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int S = p.stages, Hkv = p.Hkv;
  const MsaLayout lay(NG, S, Hkv);
  const uint32_t bar0 = sbase + lay.off_bar;
  auto kfull = [&](int s) { return bar0 + 8u * s; };
  auto vfull = [&](int s) { return bar0 + 8u * (3 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (6 + s); };   // the stage's K half is free (its QK completed)
  auto vempty = [&](int s) { return bar0 + 8u * (9 + s); };   // the stage's V half is free (its PV completed)
  auto sfull = [&](int b) { return bar0 + 8u * (12 + b); };
  auto sempty = [&](int b) { return bar0 + 8u * (14 + b); };
  auto pfull = [&](int b) { return bar0 + 8u * (16 + b); };
  auto pempty = [&](int b) { return bar0 + 8u * (18 + b); };
  const uint32_t b_pvdone = bar0 + 8u * 20, b_qfull = bar0 + 8u * 21, b_qempty = bar0 + 8u * 22;
  auto tfull = [&](int b) { return bar0 + 8u * (23 + b); };    // tile list b written
  auto tempty = [&](int b) { return bar0 + 8u * (25 + b); };   // tile list b read by every consumer
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + lay.off_misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + lay.off_misc + 4);
  int *ntiles_sm = reinterpret_cast<int *>(smem + lay.off_misc + 8);   // [row parity]
  int32_t *tiles_sm = reinterpret_cast<int32_t *>(smem + lay.off_tiles);
  auto tile_u = [&](int b) { return tiles_sm + b * 2 * kMsaMaxTiles; };
  auto tile_fl = [&](int b) { return tiles_sm + b * 2 * kMsaMaxTiles + kMsaMaxTiles; };
  float *m_sm = reinterpret_cast<float *>(smem + lay.off_ml);   // [tile parity][Hkv][NG]
  float *l_sm = m_sm + 2 * Hkv * NG;                            // [row parity][Hkv][NG]
  uint32_t *redmax = reinterpret_cast<uint32_t *>(smem + lay.off_red);       // [step parity] at stride 8*NG: [NG][4]
  float *redsum = reinterpret_cast<float *>(smem + lay.off_red) + 4 * NG;    // the same, after the maxima

  const int warp = threadIdx.x / 32, lane = lane_id();
  const int row0 = blockIdx.x, rstride = gridDim.x;

  // the first row's tile list is built while the barriers and tensor memory
  // are set up (published on its barrier by thread 0 after the setup)
  int first = row0;
  while (first < p.T && p.row_pos[first] < 0) first += rstride;
  if (warp == kMsaListWarp && first < p.T) {
    const int n = msa_row_tiles(p.sel + static_cast<int64_t>(first) * p.K, p.K, p.row_pos[first],
                                p.row_page_start[first] % p.BH, tile_u(0), tile_fl(0), p.err);
    if (lane == 0) ntiles_sm[0] = n;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(kfull(s), 1);
      mbar_init(vfull(s), 1);
      mbar_init(kempty(s), 1);
      mbar_init(vempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull(b), 1);
      mbar_init(sempty(b), 8 / NGRP);   // one arrival per softmax warp that takes the buffer's steps
      mbar_init(pfull(b), 8 / NGRP);
      mbar_init(pempty(b), 1);
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 2 + 8);      // the producer, the MMA thread and one lane per softmax warp
    }
    mbar_init(b_pvdone, 1);
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (first < p.T) mbar_arrive(tfull(0));
    tma_prefetch_desc(&p.tm_kv);
    tma_prefetch_desc(&p.tm_q);
  }
  const int tiles_cols = 2 * NG + Hkv * NG;
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tiles_cols <= 32 ? 32 : tiles_cols <= 64 ? 64 : tiles_cols <= 128 ? 128
                                    : tiles_cols <= 256 ? 256 : 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const int nbox = kMsaTile / p.BH;
    int issued_k = 0, issued_v = 0;   // global steps whose K / V loads went out
    int gbase = 0;                    // global step of the row's first step
    int j = 0;                        // rows taken so far
    int nq = 0;                       // rows whose Q was loaded
    bool ok = true;
    for (int row = row0; row < p.T && ok; row += rstride) {
      const int pos = p.row_pos[row];
      if (pos < 0) continue;
      const int page_start = p.row_page_start[row], page_off = p.row_page_off[row], npages = p.row_npages[row];
      const int lead = page_start % p.BH;
      const int buf = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(tfull(buf), (j >> 1) & 1, abort_flag, p.err));
      ++j;
      if (!ok) break;
      const int32_t *tu = tile_u(buf);
      const int nsteps = ntiles_sm[buf] * Hkv;
      bool qdone = false;
      if (nsteps > 0 && nq == 0) {   // the first row's Q goes out ahead of its keys
        if (lane == 0) {
          mbar_arrive_expect_tx(b_qfull, static_cast<uint32_t>(Hkv * QG));
          for (int gg = 0; gg < Hkv; ++gg)
            for (int c = 0; c < 2; ++c)
              tma_load_2d(sbase + lay.off_q + gg * QG + c * NG * 128, &p.tm_q, c * 64, row * p.Hq + gg * p.group,
                          b_qfull);
        }
        ++nq;
        qdone = true;
      }
      for (int ls = 0; ls < nsteps && ok; ++ls) {
        const int t = gbase + ls;
        const int ti = ls / Hkv, g = ls - ti * Hkv;
        const int u = tu[ti];
        const int st = t % S;
        // lane b: box b of the tile (positions q0 .. q0+BH-1), loaded when it
        // holds a position 0 .. pos and its page exists
        int crow = -1;
        if (lane < nbox) {
          const int q0 = kMsaTile * u - lead + lane * p.BH;
          if (q0 + p.BH - 1 >= 0 && q0 <= pos) {
            const uint32_t slot = static_cast<uint32_t>(page_start - lead + kMsaTile * u + lane * p.BH);
            const uint32_t pi = slot / static_cast<uint32_t>(p.P);
            const int page = pi < static_cast<uint32_t>(npages) ? __ldg(p.pages + page_off + pi) : -1;
            if (page < 0 || page >= p.num_pages) atomicOr(p.err, kErrBounds);
            else crow = page * p.P + static_cast<int>(slot % static_cast<uint32_t>(p.P));
          }
        }
        const uint32_t valid = __ballot_sync(0xffffffffu, crow >= 0);
        const uint32_t bytes = __popc(valid) * p.BH * 128 * 2;
        const uint32_t kst = sbase + st * STAGE, vst = kst + KVB;
        // K once the stage's previous K has been read by its QK, V once its
        // previous PV completed: the keys of a step run ahead of its values
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          const uint32_t full = half ? vfull(st) : kfull(st);
          if (lane == 0) ok = mbar_wait(half ? vempty(st) : kempty(st), ((t / S) & 1) ^ 1, abort_flag, p.err);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(full, bytes);
            else mbar_arrive(full);
          }
          __syncwarp();
          if (crow >= 0) {
            const uint32_t dst = (half ? vst : kst) + lane * p.BH * 128;
            const int x0 = (half * Hkv + g) * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) tma_load_2d(dst + c * CH, &p.tm_kv, x0 + c * 64, crow, full);
          }
          if (half) {
            issued_v = t + 1;
          } else {
            issued_k = t + 1;
            if (ls == 0 && !qdone) {
              // the row's Q, once the previous row's last QK has completed
              if (lane == 0) {
                if (nq > 0) ok = mbar_wait(b_qempty, (nq - 1) & 1, abort_flag, p.err);
                if (ok) {
                  mbar_arrive_expect_tx(b_qfull, static_cast<uint32_t>(Hkv * QG));
                  for (int gg = 0; gg < Hkv; ++gg)
                    for (int c = 0; c < 2; ++c)
                      tma_load_2d(sbase + lay.off_q + gg * QG + c * NG * 128, &p.tm_q, c * 64,
                                  row * p.Hq + gg * p.group, b_qfull);
                }
              }
              ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
              ++nq;
              if (!ok) break;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(buf));   // the row's list is no longer read here
      gbase += nsteps;
    }
    // nothing of ours may still be landing when the CTA leaves: wait (bounded,
    // whatever the abort flag says) for the loads of the last stages issued
    if (lane == 0) {
      volatile int no_abort = 0;
      for (int t = max(0, issued_k - S); t < issued_k; ++t) mbar_wait(kfull(t % S), (t / S) & 1, &no_abort, p.err);
      for (int t = max(0, issued_v - S); t < issued_v; ++t) mbar_wait(vfull(t % S), (t / S) & 1, &no_abort, p.err);
      if (nq > 0) mbar_wait(b_qfull, (nq - 1) & 1, &no_abort, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      auto issue_pv = [&](int t, int g, bool accumulate) {
        const int st = t % S;
        const uint32_t vaddr = sbase + st * STAGE + KVB;
        const uint32_t paddr = sbase + lay.off_p + (t & 1) * PB;
#pragma unroll
        for (int k = 0; k < kMsaTile / 16; ++k) {
          // A = V^T (dims x tokens), read MN-major: 64-dim chunks CH apart,
          // 8-token groups 1024 bytes apart; B = P^T, K-major
          const uint64_t ad = smem_desc(vaddr + k * 16 * 128, CH, 1024, kSwizzle128);
          const uint64_t bd = smem_desc(paddr + (k >> 2) * NG * 128 + (k & 3) * 32, 16, 1024, kSwizzle128);
          mma_f16_ss(tmem_base + 2 * NG + g * NG, ad, bd, IDESC_PV, (accumulate || k > 0) ? 1u : 0u);
        }
        mma_commit(vempty(st));
        mma_commit(pempty(t & 1));
        mma_commit(b_pvdone);
      };
      auto issue_qk = [&](int t, int g) {
        const int st = t % S;
        const uint32_t kaddr = sbase + st * STAGE;
        const uint32_t qaddr = sbase + lay.off_q + g * QG;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ss(tmem_base + (t & 1) * NG, smem_desc(kaddr + c * CH + k * 32, 16, 1024, kSwizzle128),
                       smem_desc(qaddr + c * NG * 128 + k * 32, 16, 1024, kSwizzle128), IDESC_QK, (c | k) ? 1u : 0u);
        mma_commit(sfull(t & 1));
        mma_commit(kempty(st));
      };
      auto next_row = [&](int r) {
        while (r < p.T && p.row_pos[r] < 0) r += rstride;
        return r;
      };
      // Two cursors over the CTA's global steps, QK ahead and PV behind it.
      // A cursor's row ends at a global step (q_end, p_end) known once the
      // row's step count has been read from its tile list (the QK cursor
      // waits for the list's barrier; `seen` lists so far; the PV cursor reads
      // the count after that, and the list stays put until this thread has
      // released it).  The ready tests compare steps only; row changes are
      // taken when a cursor stands at its row's end.
      int rq = next_row(row0), jq = 0, qrows = 0;
      int rp = rq, jp = 0;
      int seen = 0, nq = 0, np = 0;
      int q_end = 0, p_end = 0, p_row0 = 0;   // (q_end, p_end: 0 until a row is known)
      int gq = 0, gp = 0;                     // kv head of the next QK / PV
      bool q_known = false, p_known = false, qready = false;
      bool ok = true;
      uint32_t idle = 0;
      uint64_t idle_since = 0;
      // a polling issuer: PV of the oldest softmaxed step or QK of the next
      // step, whichever is ready, PV first (it frees a V half and a P buffer)
      while (ok && rp < p.T) {
        bool progressed = false;
        if (np < p_end && np < nq && mbar_test(pfull(np & 1), (np >> 1) & 1) && mbar_test(vfull(np % S), (np / S) & 1)) {
          tc_fence_after();
          issue_pv(np, gp, np - p_row0 >= Hkv);
          ++np;
          gp = gp + 1 == Hkv ? 0 : gp + 1;
          progressed = true;
        }
        if (nq < q_end && qready && mbar_test(kfull(nq % S), (nq / S) & 1) &&
            mbar_test(sempty(nq & 1), ((nq >> 1) & 1) ^ 1)) {
          tc_fence_after();
          issue_qk(nq, gq);
          ++nq;
          gq = gq + 1 == Hkv ? 0 : gq + 1;
          if (nq == q_end) {
            mma_commit(b_qempty);   // the row's Q may be replaced once its last QK completes
            ++qrows;
          }
          progressed = true;
        }
        if (!(q_known && nq < q_end) || !qready || !p_known || np == p_end) {
          // row changes
          if (q_known && nq == q_end) {
            rq = next_row(rq + rstride);
            ++jq;
            q_known = false;
            qready = false;
          }
          if (!q_known && rq < p.T && mbar_test(tfull(jq & 1), (jq >> 1) & 1)) {
            q_end = nq + ntiles_sm[jq & 1] * Hkv;
            gq = 0;
            ++seen;
            q_known = true;
            progressed = true;
          }
          if (q_known && !qready && nq < q_end) qready = mbar_test(b_qfull, qrows & 1);
          if (!p_known && jp < seen) {
            p_row0 = np;
            p_end = np + ntiles_sm[jp & 1] * Hkv;
            gp = 0;
            p_known = true;
          }
          if (p_known && np == p_end) {
            mbar_arrive(tempty(jp & 1));
            rp = next_row(rp + rstride);
            ++jp;
            p_known = false;
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
          idle_since = 0;
        } else {
          ++idle;
          __nanosleep(32);
          if ((idle & 255) == 0) {
            if (*abort_flag) break;
            if (idle_since == 0) {
              idle_since = globaltimer();
            } else if (globaltimer() - idle_since > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(p.err, kErrTimeout);
              break;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMsaListWarp) {
    // ------------------------------------------------------------ tile lists
    // The lists of the CTA's rows after the first, each into its row-parity
    // buffer once every consumer has released that buffer's previous row:
    // built up to two rows ahead, off the producer's path.
    int j = 1;
    for (int row = first + rstride; row < p.T; row += rstride) {
      const int pos = p.row_pos[row];
      if (pos < 0) continue;
      const int buf = j & 1;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(tempty(buf), ((j >> 1) & 1) ^ 1, abort_flag, p.err))) break;
      ++j;
      const int n = msa_row_tiles(p.sel + static_cast<int64_t>(row) * p.K, p.K, pos, p.row_page_start[row] % p.BH,
                                  tile_u(buf), tile_fl(buf), p.err);
      if (lane == 0) {
        ntiles_sm[buf] = n;
        mbar_arrive(tfull(buf));
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Eight warps, two per TMEM lane quadrant.  NGRP = 1: warp half hf takes
    // heads [hf * NG/2, (hf+1) * NG/2) of every step.  NGRP = 2 (an even
    // number of kv heads): warp half x takes every head of the steps
    // t = x, x+2, ..., i.e. of the kv heads of parity x, so the two halves
    // keep disjoint softmax state and their per-step latency chains overlap.
    // One named barrier per step and group: the per-quad maxima and sums are
    // double-buffered by the group's step parity, the reference maxima by
    // tile parity, and each step's sums are folded into l at the group's next
    // step; every exit from the loop is decided at that barrier (an OR of the
    // group's failures), so no softmax warp waits there alone.
    constexpr int NH = NG / (3 - NGRP);   // heads per warp: NG/2, or NG
    constexpr int GTHREADS = kMsaSoftThreads / NGRP;
    const int quad = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int grp = NGRP == 2 ? hf : 0;
    const int h0 = NGRP == 2 ? 0 : hf * NH;
    const int i = quad * 32 + lane;       // TMEM lane: token of S, dim of O
    const int et = threadIdx.x - 64;      // 0 .. 255
    const int gt = et - grp * GTHREADS;   // thread within the group
    const uint32_t gbar = 1 + grp;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    int j = 0, gbase = 0;
    // the row whose output is still to be written (at the next row's start,
    // overlapping that row's first QK): its row, its l buffer and the
    // group's last step in it
    const uint32_t ocol = tmem_base + lane_base + 2 * NG + h0;   // O of kv head 0, this warp's heads
    int pend_row = -1, pend_buf = 0, pend_tlast = -1;
    auto flush = [&](bool wait_pv) {   // writes the pending row's output
      bool pg = true;
      if (wait_pv && pend_tlast >= 0) pg = __all_sync(0xffffffffu, mbar_wait(pempty(pend_tlast & 1), (pend_tlast >> 1) & 1, abort_flag, p.err));
      tc_fence_after();
      if (pg)
        msa_write_out<NG, NGRP, NH>(ocol, l_sm + pend_buf * Hkv * NG, Hkv, grp, h0, p.group,
                                    p.out + static_cast<int64_t>(pend_row) * p.Hq * 128, i);
      tc_fence_before();
      pend_row = -1;
      return pg;
    };
    // the next row's position and first slot are loaded a row ahead
    int pos_n = row0 < p.T ? p.row_pos[row0] : -1, ps_n = row0 < p.T ? p.row_page_start[row0] : 0;
    auto prefetch = [&](int r) {
      if (r < p.T) {
        pos_n = p.row_pos[r];
        ps_n = p.row_page_start[r];
      }
    };
    for (int row = row0; row < p.T && ok; row += rstride) {
      const int pos = pos_n, lead = ps_n % p.BH;
      if (pos < 0) {
        prefetch(row + rstride);
        continue;
      }
      const int buf = j & 1;
      bool good = __all_sync(0xffffffffu, mbar_wait(tfull(buf), (j >> 1) & 1, abort_flag, p.err));
      ++j;
      const int nsteps = (good ? ntiles_sm[buf] : 0) * Hkv;
      const int32_t *tu = tile_u(buf), *tf = tile_fl(buf);
      float *l_row = l_sm + buf * Hkv * NG;
      // the group's softmax state starts afresh (every reader of the previous
      // row's passed the barrier that ended that row)
      for (int k = gt; k < Hkv * NG; k += GTHREADS) {
        if ((k / NG) % NGRP != grp) continue;
        m_sm[k] = kMsaNegBig;            // reference maxima, tile parity 0
        m_sm[Hkv * NG + k] = kMsaNegBig; // tile parity 1
        l_row[k] = 0.f;
      }
      if (named_bar_any(gbar, GTHREADS, !good)) {
        ok = false;
        break;
      }
      // (loaded after the barrier: a load still in flight holds its thread
      // at the next one)
      prefetch(row + rstride);
      // the previous row's output, while this row's first QK is on its way:
      // its last PV first (no P of this row is written yet, so the wait on
      // that PV's P buffer names it exactly)
      if (pend_row >= 0) ok = flush(true);
      bool carry = true;        // this warp's result of the previous step's last wait
      float alpha_prev = 1.f;   // (gt < NG) alpha of head gt at the group's previous step of the row
      int g_prev = 0;
      int t_last = -1;          // the group's last step of the row
      for (int ls = grp, lr = 0; ls < nsteps && ok; ls += NGRP, ++lr) {
        const int t = gbase + ls;           // global step (gbase is even when NGRP = 2)
        const int lt = t / NGRP;            // the group's own step count
        const int ti = ls / Hkv, g = ls - ti * Hkv;
        const int u = tu[ti], fl = tf[ti];
        const int q = kMsaTile * u - lead + i;
        const bool valid = q >= 0 && q <= pos && ((i < lead) ? (fl & 1) : (fl & 2));
        uint32_t *rmax = redmax + (grp * 2 + (lt & 1)) * 8 * NG;
        float *rsum = redsum + (grp * 2 + (lt & 1)) * 8 * NG;
        good = carry && __all_sync(0xffffffffu, mbar_wait(sfull(t & 1), (t >> 1) & 1, abort_flag, p.err));
        tc_fence_after();
        float s[NH];
        if (good) {
          if constexpr (NH == 8) {
            tmem_ld8(tmem_base + lane_base + (t & 1) * NG + h0, s);
          } else {
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 16)
              tmem_ld16(tmem_base + lane_base + (t & 1) * NG + h0 + c0, *reinterpret_cast<float(*)[16]>(s + c0));
          }
          tmem_ld_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (good && lane == 0) mbar_arrive(sempty(t & 1));
        // each head's largest logit over this warp's 32 rows of the tile (as an
        // order key; masked rows count as -inf), by the transposing reduction
        {
          float mx[NH];
#pragma unroll
          for (int h = 0; h < NH; ++h) mx[h] = valid ? s[h] : -INFINITY;
          if constexpr (NH <= 16) {
            const float m = warp_reduce_transpose<NH>(mx, MaxOp{});   // lane l holds head (l >> (5 - log2 NH))
            constexpr int SHIFT = NH == 8 ? 2 : 1;
            if ((lane & ((1 << SHIFT) - 1)) == 0) rmax[(h0 + (lane >> SHIFT)) * 4 + quad] = score_key(m);
          } else {
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 32) {
              const float m = warp_reduce_transpose<32>(*reinterpret_cast<float(*)[32]>(mx + c0), MaxOp{});
              rmax[(h0 + c0 + lane) * 4 + quad] = score_key(m);
            }
          }
        }
        if (named_bar_any(gbar, GTHREADS, !good)) {
          ok = false;
          break;
        }
        // the group's previous step's sums (its barrier has passed in every warp of the group)
        if (lr > 0 && gt < NG) {
          const float4 ps = reinterpret_cast<const float4 *>(redsum + (grp * 2 + ((lt - 1) & 1)) * 8 * NG)[gt];
          l_row[g_prev * NG + gt] = l_row[g_prev * NG + gt] * alpha_prev + ((ps.x + ps.y) + (ps.z + ps.w));
        }
        const float *mold_sm = m_sm + ((ti & 1) ^ 1) * Hkv * NG + g * NG;   // written at the group's previous tile
        float *mnew_sm = m_sm + (ti & 1) * Hkv * NG + g * NG;
        // reference max of head h for this step (every thread that needs a
        // head derives the same value from the same shared data)
        auto head_max = [&](int h, float &alpha) -> float {
          const uint4 k4 = reinterpret_cast<const uint4 *>(rmax)[h];
          const uint32_t k = max(max(k4.x, k4.y), max(k4.z, k4.w));
          const float mold = mold_sm[h];
          // (a tile always holds a kept position, so k is a real score: a
          // quadrant with none gives the key of -inf, below every score)
          const float tmax = key_score(k) * p.scale_log2;
          alpha = 1.f;
          if (tmax > mold + kMsaRescale) {
            alpha = fast_exp2(mold - tmax);
            return tmax;
          }
          return mold;
        };
        float alpha[NH], mnew[NH];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          mnew[h] = head_max(h0 + h, alpha[h]);
          rescale = rescale || alpha[h] != 1.f;
        }
        if (gt < NG) {
          float a;
          mnew_sm[gt] = head_max(gt, a);
          alpha_prev = a;
          g_prev = g;
        }
        t_last = t;
        // P (bf16) and the tile's per-head sums of what PV will add
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float e = valid ? fast_exp2(fmaf(s[h], p.scale_log2, -mnew[h])) : 0.f;
          s[h] = __bfloat162float(__float2bfloat16_rn(e));
        }
        if constexpr (NH <= 16) {
          const float sum = warp_sum_transpose<NH>(s);   // lane l holds head (l >> (5 - log2 NH))
          constexpr int SHIFT = NH == 8 ? 2 : 1;
          if ((lane & ((1 << SHIFT) - 1)) == 0) rsum[(h0 + (lane >> SHIFT)) * 4 + quad] = sum;
        } else {
#pragma unroll
          for (int c0 = 0; c0 < NH; c0 += 32) {
            const float sum = warp_sum_transpose<32>(*reinterpret_cast<float(*)[32]>(s + c0));   // lane h: head h
            rsum[(h0 + c0 + lane) * 4 + quad] = sum;
          }
        }
        // P^T buffer (t & 1) is free once PV(t-2) completed (with NGRP = 2 that
        // wait also orders the O rescale below after every earlier PV into O)
        good = __all_sync(0xffffffffu, mbar_wait(pempty(t & 1), ((t >> 1) & 1) ^ 1, abort_flag, p.err));
        tc_fence_after();
        if (good) {
          const uint32_t pbase = sbase + lay.off_p + (t & 1) * PB + (i >> 6) * NG * 128 + ((i & 7) << 1);
          const uint32_t c8 = (i & 63) >> 3;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int hh = h0 + h;
            const uint32_t a = pbase + hh * 128 + ((c8 ^ (hh & 7)) << 4);
            const __nv_bfloat16 pb = __float2bfloat16_rn(s[h]);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<const uint16_t *>(&pb)) : "memory");
          }
        }
        // V rows of positions outside the kept blocks are zeroed once the tile
        // has landed (a zero probability must not meet a stale value); with
        // NGRP = 1, warp half hf zeroes 64-column chunk hf
        if (good && __any_sync(0xffffffffu, !valid)) {
          const int st = t % S;
          good = __all_sync(0xffffffffu, mbar_wait(vfull(st), (t / S) & 1, abort_flag, p.err));
          if (good && !valid) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if (NGRP == 1 && c != hf) continue;
              const uint32_t vrow = sbase + st * STAGE + KVB + c * CH + i * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k) st_shared_v4(vrow + k * 16, make_uint4(0u, 0u, 0u, 0u));
            }
          }
        }
        fence_proxy_async_smem();
        // O of this kv head (this warp's head columns) is rescaled once every
        // earlier PV into it has completed (its first tile has no O yet).  With
        // NGRP = 2 that is PV(t-2), already waited for above (PV(t-1) belongs
        // to another kv head); with NGRP = 1 it is PV(t-1) (the wait above has
        // PV(t-2) complete, so the parity wait cannot pass two phases short).
        if (good && __any_sync(0xffffffffu, rescale) && ti > 0) {
          if (NGRP == 1) {
            good = __all_sync(0xffffffffu, mbar_wait(b_pvdone, (t - 1) & 1, abort_flag, p.err));
            tc_fence_after();
          }
          if (good) {
            const uint32_t oaddr = ocol + g * NG;
            if constexpr (NH == 8) {
              float o[8];
              tmem_ld8(oaddr, o);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 8; ++k) o[k] *= alpha[k];
              tmem_st8(oaddr, o);
            } else {
#pragma unroll
              for (int c0 = 0; c0 < NH; c0 += 16) {
                float o[16];
                tmem_ld16(oaddr + c0, o);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) o[k] *= alpha[c0 + k];
                tmem_st16(oaddr + c0, o);
              }
            }
            tmem_st_wait();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (good && lane == 0) mbar_arrive(pfull(t & 1));
        carry = good;
      }
      // the row's last sums into l; its output is written at the start of the
      // next row (or after the last one)
      ok = !named_bar_any(gbar, GTHREADS, !(ok && carry));   // the group's last sums are in place
      if (ok && t_last >= 0 && gt < NG) {
        const float4 ps = reinterpret_cast<const float4 *>(redsum + (grp * 2 + ((t_last / NGRP) & 1)) * 8 * NG)[gt];
        l_row[g_prev * NG + gt] = l_row[g_prev * NG + gt] * alpha_prev + ((ps.x + ps.y) + (ps.z + ps.w));
      }
      pend_row = row;
      pend_buf = buf;
      pend_tlast = t_last;
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(buf));
      gbase += nsteps;
    }
    // the CTA's last row (its sums were folded before the group's last barrier)
    ok = !named_bar_any(gbar, GTHREADS, !ok);
    if (ok && pend_row >= 0) flush(true);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    tmem_dealloc(tmem_base, tiles_cols <= 32 ? 32 : tiles_cols <= 64 ? 64 : tiles_cols <= 128 ? 128
                                                 : tiles_cols <= 256 ? 256 : 512);
}

// ---------------------------------------------------------------------------
// GQA attention over the selected blocks, CUDA cores (any shape)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) msa_attend_simt_kernel(
    const int32_t *__restrict__ sel, const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kv,
    const int32_t *__restrict__ row_pos, const int32_t *__restrict__ row_page_off,
    const int32_t *__restrict__ row_npages, const int32_t *__restrict__ row_page_start,
    const int32_t *__restrict__ pages, __nv_bfloat16 *__restrict__ out, int *err, int Hq, int Hkv, int D, int bs,
    int K, int P, int num_pages, float scale_log2) {
  extern __shared__ float sm[];   // q [D], logits [K*bs], reduce [32]
  float *qs = sm;
  float *lg = sm + D;
  float *red = lg + static_cast<int64_t>(K) * bs;
  const int row = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const int g = h / (Hq / Hkv);
  const int pos = row_pos[row];
  if (pos < 0) return;
  const int64_t row_elems = 2 * static_cast<int64_t>(Hkv) * D;
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    qs[d] = __bfloat162float(q[(static_cast<int64_t>(row) * Hq + h) * D + d]);
  __syncthreads();
  const int32_t *sr = sel + static_cast<int64_t>(row) * K;
  const int n = K * bs;
  auto cache_row = [&](int e) -> int64_t {   // physical row of entry e, or -1
    const int blk = sr[e / bs];
    if (blk == -1) return -1;
    if (blk < -1 || blk > pos / bs) {
      atomicOr(err, kErrBounds);
      return -1;
    }
    const int j = blk * bs + e % bs;
    if (j > pos) return -1;
    const int64_t slot = static_cast<int64_t>(row_page_start[row]) + j;
    const int64_t pi = slot / P;
    const int page = pi < row_npages[row] ? pages[row_page_off[row] + pi] : -1;
    if (page < 0 || page >= num_pages) {
      atomicOr(err, kErrBounds);
      return -1;
    }
    return static_cast<int64_t>(page) * P + slot % P;
  };
  float mloc = -INFINITY;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int64_t r = cache_row(e);
    float x = -INFINITY;
    if (r >= 0) {
      const __nv_bfloat16 *k = kv + r * row_elems + static_cast<int64_t>(g) * D;
      float a = 0.f;
      for (int d = 0; d < D; ++d) a = fmaf(qs[d], __bfloat162float(k[d]), a);
      x = a * scale_log2;
    }
    lg[e] = x;
    mloc = fmaxf(mloc, x);
  }
  for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = mloc;
  __syncthreads();
  float m = -INFINITY;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float lloc = 0.f;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const float pe = lg[e] == -INFINITY ? 0.f : exp2f(lg[e] - m);
    lg[e] = pe;
    lloc += pe;
  }
  for (int o = 16; o; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = lloc;
  __syncthreads();
  float lsum = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) lsum += red[w];
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int e = 0; e < n; ++e) {
      if (lg[e] == 0.f) continue;
      const int64_t r = cache_row(e);
      acc = fmaf(lg[e], __bfloat162float(kv[r * row_elems + static_cast<int64_t>(Hkv + g) * D + d]), acc);
    }
    out[(static_cast<int64_t>(row) * Hq + h) * D + d] = __float2bfloat16_rn(acc * inv);
  }
}

template <int NG, int NGRP>
cudaError_t run_msa_tc(const dsa_ctx *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t &ms, const int32_t *sel,
                       const void *q, const void *kv, float sm_scale, void *out, cudaStream_t s) {
  MsaParams prm{};
  const int BH = plan->box_rows;
  const int P = ctx->cfg.page_size;
  if (!encode_tiled_2d(&prm.tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(kv),
                       2 * static_cast<uint64_t>(ms.kv_heads) * 128, static_cast<uint64_t>(plan->cache_pages) * P,
                       2 * static_cast<uint64_t>(ms.kv_heads) * 128 * 2, 64, BH, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled_2d(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(q), 128,
                       static_cast<uint64_t>(plan->T) * ms.q_heads, 256, 64, NG, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  prm.sel = sel;
  prm.row_pos = plan->row_pos;
  prm.row_page_off = plan->row_page_off;
  prm.row_npages = plan->row_npages;
  prm.row_page_start = plan->row_page_start;
  prm.pages = plan->pages;
  prm.out = static_cast<__nv_bfloat16 *>(out);
  prm.err = ctx->err;
  prm.T = plan->T;
  prm.Hq = ms.q_heads;
  prm.Hkv = ms.kv_heads;
  prm.group = ms.q_heads / ms.kv_heads;
  prm.K = ms.topk_blocks;
  prm.P = P;
  prm.BH = BH;
  prm.num_pages = plan->cache_pages;
  prm.scale_log2 = sm_scale * kMsaLog2e;
  prm.stages = MsaLayout(NG, 3, ms.kv_heads).bytes <= 227 * 1024 ? 3 : 2;
  const int bytes = static_cast<int>(MsaLayout(NG, prm.stages, ms.kv_heads).bytes);
  auto kern = msa_attend_tc_kernel<NG, NGRP>;
  // the limit is set to the largest layout this instance can have
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(kern, 227 * 1024, ctx->device, smem_limit_set); e != cudaSuccess) return e;
  // persistent: one CTA per SM (the layout fills shared memory), rows strided over the grid
  kern<<<std::min(plan->T, std::max(1, ctx->num_sms)), kMsaThreads, bytes, s>>>(prm);
  return cudaGetLastError();
}

int msa_group_cols(int group) { return (group + 15) / 16 * 16; }

}  // namespace

bool msa_attend_tc_supported(const dsa_config_t &c, const dsa_msa_shape_t &ms, int box_rows) {
  if (ms.block_size != kMsaTile || ms.head_dim != 128 || ms.kv_heads > kMsaMaxKvHeads) return false;
  const int NG = msa_group_cols(ms.q_heads / ms.kv_heads);
  if (NG != 16 && NG != 32 && NG != 64) return false;
  if (2 * NG + ms.kv_heads * NG > 512) return false;
  if (box_rows < 8 || c.page_size % box_rows != 0) return false;
  return MsaLayout(NG, 2, ms.kv_heads).bytes <= 227 * 1024;
}

cudaError_t launch_msa_select(const dsa_ctx *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t &ms,
                              const float *scores, const uint32_t *block_keys, int32_t *sel, cudaStream_t s,
                              int32_t *launches) {
  // shared memory for the plan's longest row only, so short rows (prefill)
  // fit four CTAs per SM; the grid is what stays resident
  const int max_blocks = static_cast<int>(static_cast<int64_t>(plan->max_pos) / ms.block_size + 1);
  const int smem = std::min(kSelMaxBlocks, std::max(max_blocks, 32)) * 4;
  static std::atomic<uint64_t> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(msa_select_kernel, kSelMaxBlocks * 4, ctx->device, smem_limit_set);
      e != cudaSuccess)
    return e;
  int per_sm = 1;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, msa_select_kernel, kSelThreads, smem);
      e != cudaSuccess)
    return e;
  const int grid = std::min(plan->T, std::max(1, per_sm) * ctx->num_sms);
  msa_select_kernel<<<std::max(1, grid), kSelThreads, smem, s>>>(scores, block_keys, plan->row_score_off,
                                                                  plan->row_pos, plan->T, ms.block_size,
                                                                  ms.topk_blocks, sel);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_msa_attend(const dsa_ctx *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t &ms,
                              const int32_t *sel, const void *q, const void *kv, float sm_scale, void *out,
                              cudaStream_t s, int32_t *launches) {
  cudaError_t e;
  if (msa_attend_tc_supported(ctx->cfg, ms, plan->box_rows)) {
    const int NG = msa_group_cols(ms.q_heads / ms.kv_heads);
    // an even number of kv heads: two warp groups take alternate steps
    const bool two = ms.kv_heads % 2 == 0;
    if (NG == 16) e = two ? run_msa_tc<16, 2>(ctx, plan, ms, sel, q, kv, sm_scale, out, s)
                          : run_msa_tc<16, 1>(ctx, plan, ms, sel, q, kv, sm_scale, out, s);
    else if (NG == 32) e = two ? run_msa_tc<32, 2>(ctx, plan, ms, sel, q, kv, sm_scale, out, s)
                               : run_msa_tc<32, 1>(ctx, plan, ms, sel, q, kv, sm_scale, out, s);
    else e = run_msa_tc<64, 1>(ctx, plan, ms, sel, q, kv, sm_scale, out, s);
  } else {
    const size_t sm = (static_cast<size_t>(ms.head_dim) + static_cast<size_t>(ms.topk_blocks) * ms.block_size + 32) *
                      sizeof(float);
    if (sm > 227 * 1024) return cudaErrorInvalidValue;
    if (sm > 48 * 1024) {
      e = cudaFuncSetAttribute(msa_attend_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sm));
      if (e != cudaSuccess) return e;
    }
    msa_attend_simt_kernel<<<plan->T * ms.q_heads, 128, sm, s>>>(
        sel, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(kv), plan->row_pos,
        plan->row_page_off, plan->row_npages, plan->row_page_start, plan->pages, static_cast<__nv_bfloat16 *>(out),
        ctx->err, ms.q_heads, ms.kv_heads, ms.head_dim, ms.block_size, ms.topk_blocks, ctx->cfg.page_size,
        plan->cache_pages, sm_scale * kMsaLog2e);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) *launches += 1;
  return e;
}

bool msa_select_supported(const dsa_plan_t *plan, const dsa_msa_shape_t &ms) {
  return static_cast<int64_t>(plan->max_pos) / ms.block_size + 1 <= kSelMaxBlocks;
}

}  // namespace dsa

// ----------------------------------------------------------------------------
// C ABI
// ----------------------------------------------------------------------------
namespace {

dsa_status msa_check(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *ms) {
  if (!ctx || !plan || !ms || plan->ctx != ctx || ctx->device < 0) return DSA_ERR_INVALID_ARG;
  if (ms->block_size <= 0 || ms->topk_blocks <= 0 || ms->q_heads <= 0 || ms->kv_heads <= 0 || ms->head_dim <= 0 ||
      ms->reserved != 0 || ms->q_heads % ms->kv_heads != 0)
    return DSA_ERR_INVALID_ARG;
  if (ms->topk_blocks > dsa::kMsaMaxK || ms->head_dim % 8 != 0 || ms->head_dim > 1024) return DSA_ERR_UNSUPPORTED;
  if (plan->capturable) return DSA_ERR_UNSUPPORTED;   // host plans only
  if (cudaSetDevice(ctx->device) != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

dsa_status msa_status(dsa_ctx_t *ctx, cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  snprintf(ctx->last_cuda_error, sizeof(ctx->last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

}  // namespace

extern "C" {

dsa_status dsa_msa_select_blocks(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape,
                                 const float *scores, int32_t *block_sel, dsa_stream_t stream) {
  dsa_status st = msa_check(ctx, plan, shape);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (!dsa::msa_select_supported(plan, *shape)) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!scores || !block_sel) return DSA_ERR_INVALID_ARG;
  return msa_status(ctx, dsa::launch_msa_select(ctx, plan, *shape, scores, nullptr, block_sel,
                                                reinterpret_cast<cudaStream_t>(stream), &ctx->last_launches));
}

dsa_status dsa_msa_index_select(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape, const void *q,
                                const float *w, const void *index_cache, int32_t *block_sel, dsa_stream_t stream) {
  dsa_status st = msa_check(ctx, plan, shape);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (!dsa::msa_select_supported(plan, *shape)) return DSA_ERR_UNSUPPORTED;
  if (plan->T == 0) return DSA_OK;
  if (!q || !w || !index_cache || !block_sel) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t n = 0;
  cudaError_t e;
  if (dsa::index_block_keys_supported(ctx, plan)) {
    // block maxima straight from the indexer's epilogue: no token scores
    const size_t words = static_cast<size_t>(plan->num_scores / shape->block_size) + plan->T + 1;
    if (words > ctx->block_keys_cap) {
      cudaFree(ctx->block_keys);
      ctx->block_keys = nullptr;
      ctx->block_keys_cap = 0;
      if (cudaMalloc(&ctx->block_keys, words * sizeof(uint32_t)) != cudaSuccess) return DSA_ERR_OOM;
      ctx->block_keys_cap = words;
    }
    e = cudaMemsetAsync(ctx->block_keys, 0, words * sizeof(uint32_t), s);
    if (e == cudaSuccess)
      e = dsa::launch_index_block_keys(ctx, plan, q, w, index_cache, ctx->block_keys, shape->block_size, s, &n);
    if (e == cudaSuccess) e = dsa::launch_msa_select(ctx, plan, *shape, nullptr, ctx->block_keys, block_sel, s, &n);
  } else {
    if (static_cast<size_t>(plan->num_scores) > ctx->scores_cap) return DSA_ERR_INVALID_ARG;   // plan of another size
    e = dsa::launch_index_scores(ctx, plan, q, w, index_cache, ctx->scores, s, &n);
    if (e == cudaSuccess) e = dsa::launch_msa_select(ctx, plan, *shape, ctx->scores, nullptr, block_sel, s, &n);
  }
  ctx->last_launches = n;
  return msa_status(ctx, e);
}

dsa_status dsa_msa_attend(dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape,
                          const int32_t *block_sel, const void *q, const void *kv_cache, float sm_scale, void *out,
                          dsa_stream_t stream) {
  dsa_status st = msa_check(ctx, plan, shape);
  if (st != DSA_OK) return st;
  ctx->last_launches = 0;
  if (plan->T == 0) return DSA_OK;
  if (!block_sel || !q || !kv_cache || !out) return DSA_ERR_INVALID_ARG;
  if (!dsa::msa_attend_tc_supported(ctx->cfg, *shape, plan->box_rows) &&
      (static_cast<size_t>(shape->head_dim) + static_cast<size_t>(shape->topk_blocks) * shape->block_size + 32) *
              sizeof(float) >
          227 * 1024)
    return DSA_ERR_UNSUPPORTED;
  return msa_status(ctx, dsa::launch_msa_attend(ctx, plan, *shape, block_sel, q, kv_cache, sm_scale, out,
                                                reinterpret_cast<cudaStream_t>(stream), &ctx->last_launches));
}

int dsa_msa_attend_on_tensor_cores(const dsa_ctx_t *ctx, const dsa_plan_t *plan, const dsa_msa_shape_t *shape) {
  if (!ctx || !plan || !shape || shape->kv_heads <= 0 || shape->q_heads % shape->kv_heads != 0) return 0;
  return dsa::msa_attend_tc_supported(ctx->cfg, *shape, plan->box_rows) ? 1 : 0;
}

}  // extern "C"
