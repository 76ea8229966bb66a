// S1 / S3: indexer scores (the indexer side attention of recipes.vllm.ai
// "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention"; the formula
// score = sum_h w_h * ReLU(q_h . k) is the one this library fixes).
//
// Per query the scores are one skinny contraction: keys [rows x 128] times
// q_idx^T [128 x 16 heads], 4096 flop per key. Tiles of 128 key rows are the
// M side of a tcgen05.mma (M = 128, N = 16, fp32 accumulators in tensor
// memory), which keeps the key stream HBM-bound: CUDA-core FMA could not keep
// up with HBM at 31 flop per byte.
//
// A persistent CTA per SM runs a warp-specialised pipeline over its share of
// (query, tile) pairs, with four tiles in flight in tensor memory. Tiles
// alternate between two halves of the CTA (tile i belongs to half i % 2), and
// each half has its own producer warp and load ring: small gathered boxes
// stream at about twice the rate with two independent producers per SM. A
// ring stage holds TPS of its half's tiles behind one TMA barrier (1 for bf16
// keys, whose tiles are 32 KB; 2 for the narrower MXFP8 and MXFP4 tiles)
// because a TMA ring streams HBM fastest with about 32 KB per barrier.
//   warps 0-1  producers: TMA tiled loads (128-byte swizzle) of the tiles' key
//              rows: one box of 128 rows for block keys or a plain latent
//              range, one box of 8 rows per candidate block otherwise; MX
//              scales (4 bytes a row) come with the tiles: one bulk copy for a
//              contiguous tile, two 16-byte cp.async per gathered block;
//   warps 2, 11 MMA issuers, one per half: 8 MMAs (K = 128) per tile (a
//              barrier wait costs a single thread a few hundred cycles, so
//              two issuers overlap their waits);
//   warps 3-10 two math sets of four warps, set k for half k.
//              Thread = TMEM lane = key row of the tile.
// bf16 keys: the swizzled raw tile is the MMA's A operand as loaded.
// MXFP8 keys (e4m3 codes + one UE8M0 scale per 32 values) and MXFP4 keys
// (e2m1 codes two a byte + one UE8M0 scale per 32 values): each math thread
// converts its own row code by code to f16 (exact: every e4m3 and every e2m1
// value is an f16 normal or zero) and writes it into tensor memory, where the
// MMA reads A; each 32-wide group gets its own accumulator (4 x 16 TMEM
// columns), so the power-of-two scales are applied exactly in the epilogue.
// An MXFP4 row is 64 bytes: the TMA sees the key array as rows of 128 bytes
// (two keys each), so a 128-key tile is a box of 64 such rows and a gathered
// block of 8 keys a box of 4. The index query is taken to f16 with a
// power-of-two scale per head that puts its largest element in [2^14, 2^15),
// which keeps every bf16 element exact unless it is below 2^-31 of its head's
// largest.
// The epilogue of tile i - 4 runs before tile i is prepared and writes
// score = sum_h w_h * max(0, dot_h), summed in head order.
#include <type_traits>

#include "kernels.h"

namespace dsa {

namespace {

constexpr int kTile = 128;          // key rows per tile (MMA M)
constexpr int kThreads = 384;       // 2 producers, MMA, 2 x 4 math warps, MMA
constexpr int kMmaWarp = 2;         // issues the MMAs of even tiles
constexpr int kMmaWarp2 = 11;       // issues the MMAs of odd tiles
constexpr int kMathWarp0 = 3;
constexpr int kMathThreads = 128;   // per math set
constexpr int kSlots = 4;           // tiles in flight (TMEM slots)
constexpr int kQRing = 3;           // index-query slots per math set

template <int FMT>
struct Plan;
template <>
struct Plan<DSA_FMT_BF16> {
  static constexpr int kRowBytes = 256;
  static constexpr int kCodeBytes = kTile * 256;  // 2 K-atoms x 128 rows x 128 B
  static constexpr int kScaleBytes = 0;
  static constexpr int kAccCols = 16;
  static constexpr int kSlotCols = 16;             // accumulator only
  static constexpr int kTmemCols = 64;
};
template <>
struct Plan<DSA_FMT_MXFP8> {
  static constexpr int kRowBytes = 128;
  static constexpr int kCodeBytes = kTile * 128;  // codes, swizzled
  static constexpr int kScaleBytes = kTile * 4;
  static constexpr int kAccCols = 64;    // 4 groups x 16 heads
  static constexpr int kSlotCols = 128;  // A operand (64 columns of f16 pairs) + accumulator
  static constexpr int kTmemCols = 512;
};
template <>
struct Plan<DSA_FMT_MXFP4> {
  static constexpr int kRowBytes = 64;
  static constexpr int kCodeBytes = kTile * 64;   // 64 rows of two keys, swizzled
  static constexpr int kScaleBytes = kTile * 4;
  static constexpr int kAccCols = 64;
  static constexpr int kSlotCols = 128;
  static constexpr int kTmemCols = 512;
};

// Tiles per ring stage of a gathered (token-stage) scan over MX keys.
#ifndef DSA_SCAN_GATHER_TPS
#define DSA_SCAN_GATHER_TPS 2
#endif
// Tiles per ring stage of an MXFP4 scan, contiguous and gathered.
#ifndef DSA_SCAN_MXFP4_TPS
#define DSA_SCAN_MXFP4_TPS 2
#endif
#ifndef DSA_SCAN_MXFP4_GATHER_TPS
#define DSA_SCAN_MXFP4_GATHER_TPS 2
#endif

// A ring stage: TPS tiles' codes (each 1024-byte aligned, as the 128-byte
// swizzle wants), then their scales; stages per half as shared memory allows.
template <int FMT, int TPS>
struct Ring {
  using P = Plan<FMT>;
  static constexpr int kTPS = TPS;
  static constexpr int kStageBytes = TPS * (P::kCodeBytes + P::kScaleBytes);
  static constexpr int kRawStride = (kStageBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = FMT == DSA_FMT_BF16 ? 3 : (TPS == 1 ? 5 : (TPS == 2 ? 3 : 2));
  __device__ static uint32_t codes(uint32_t stage, int t) {
    return stage + static_cast<uint32_t>(t * P::kCodeBytes);
  }
  __device__ static uint32_t scales(uint32_t stage, int t) {
    return stage + static_cast<uint32_t>(TPS * P::kCodeBytes + t * P::kScaleBytes);
  }
};

constexpr int kMaxStages = 5;
constexpr int kMaxTPS = 4;

struct TileMeta {
  uint32_t valid[4];  // row r holds a key
};

struct QSlot {
  float w[kIdxHeads];
  float qinv[kIdxHeads];
};

struct Shared {
  uint64_t raw_full[2][kMaxStages], raw_empty[2][kMaxStages];
  uint64_t op_full[kSlots], acc_full[kSlots];
  uint32_t tmem_base;
  int abort;
  TileMeta meta[2][kMaxStages][kMaxTPS];
  QSlot qs[2][kQRing];
  int tile_slot[kSlots];  // index-query slot of the tile in each TMEM slot (set by its math set)
};

template <int FMT, int TPS>
struct Layout {
  using R = Ring<FMT, TPS>;
  static_assert(R::kStages <= kMaxStages && TPS <= kMaxTPS, "ring plan");
  static constexpr int kRaw = 0;                                    // [half][stage]
  static constexpr int kQ = kRaw + 2 * R::kStages * R::kRawStride;  // [set][ring] x 4 KB B operands
  static constexpr int kShared = kQ + 2 * kQRing * 4096;
  static constexpr int kBytes = kShared + static_cast<int>(sizeof(Shared));
  static_assert(kBytes + 1024 <= 232448, "shared memory");
};

struct Maps {
  // bf16: {128 elems, rows}, box {64, R}; MXFP8: {128 B, rows}, box {128, R};
  // MXFP4: {128 B, rows / 2} (two keys a row), box {128, R / 2}
  CUtensorMap keys;
};

__device__ __forceinline__ int visible_latents(const ScanArgs& a, int b) {
  int n = a.prefill ? static_cast<int>((query_pos(a.ctx, a.mq, a.n_tokens, b) + 1) / a.ratio)
                    : a.n_latents[b];
  if (n > a.max_latents) n = static_cast<int>(a.max_latents);
  return n < 0 ? 0 : n;
}

// Key rows of query b in the contiguous modes. Prefill block rows stop at the
// last complete block; a partially visible block is scored by its own kernel.
__device__ __forceinline__ int64_t contiguous_rows(const ScanArgs& a, int n_vis) {
  int64_t n;
  if (a.mode == ROWS_BLOCKS) {
    n = a.prefill ? n_vis / 8 : (n_vis + 7) / 8;
  } else {
    n = n_vis;
  }
  return n < a.n_rows ? n : a.n_rows;
}

// First key row of query b's sequence in a contiguous cache.
__device__ __forceinline__ int64_t seq_row0(const ScanArgs& a, int b) {
  return static_cast<int64_t>(a.mq > 0 ? b / a.mq : b) * a.key_stride;
}

// Position of a CTA's tile: query b and first row r0 of that query's rows.
// Tiles advance by a small fixed step (at most 2 x TPS tiles) without
// divisions.
struct TilePos {
  int b;
  int64_t r0;
  __device__ void init(int64_t tile, int64_t tpq) {
    b = static_cast<int>(tile / tpq);
    r0 = (tile % tpq) * kTile;
  }
  __device__ void advance(int step, int64_t q_rows) {
    r0 += static_cast<int64_t>(step) * kTile;
    while (r0 >= q_rows) {
      r0 -= q_rows;
      ++b;
    }
  }
};

template <int FMT, int TPS>
__device__ void producer(const ScanArgs& a, const Maps& maps, Shared& sh, uint32_t sbase,
                         int64_t t_begin, int64_t n_tiles, int64_t tpq, int half) {
  using P = Plan<FMT>;
  using R = Ring<FMT, TPS>;
  using Lo = Layout<FMT, TPS>;
  const int lane = threadIdx.x & 31;
  if (lane == 0) tma_prefetch_map(&maps.keys);
  const int64_t n_own = n_tiles > half ? (n_tiles - half + 1) / 2 : 0;  // tiles half, half + 2, ...
  if (n_own == 0) return;
  const int64_t q_rows = tpq * kTile;
  // Gathered blocks, and every row of a paged cache, come in groups of 8 rows
  // (one TMA box each: a page holds whole groups).
  const bool paged = a.pages.table != nullptr;
  const bool gather = a.mode == ROWS_GATHER || paged;
  // MX scales of 8 (gathered block) or 128 (contiguous tile) consecutive rows
  // are 32 or 512 contiguous bytes, copied whole when 16-byte aligned.
  const bool scale_vec =
      ((reinterpret_cast<uintptr_t>(a.key_scales) | static_cast<uintptr_t>(a.key_stride * 4)) &
       15u) == 0;
  // Grouped mode: in round k lane l serves 8-row group l % 16 of the stage's
  // tile 2k + l / 16 (16 groups of 8 rows per tile): the candidate block
  // (gathered) or the group's own place in the query's rows (paged). Block ids
  // are loaded two stages ahead and (paged) their page-table entries one stage
  // ahead, each from a value that has had a whole stage to arrive.
  constexpr int kRounds = (TPS * 16 + 31) / 32;
  auto fetch_blocks = [&](const TilePos& first, int64_t j0, int (&ids)[kRounds]) {
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      const int t = 2 * k + (lane >> 4);
      ids[k] = -1;
      if (!gather || t >= TPS || j0 + t >= n_own) continue;
      TilePos tp = first;
      tp.advance(2 * t, q_rows);
      const int64_t bi = (tp.r0 >> 3) + (lane & 15);
      if (a.mode != ROWS_GATHER) {
        ids[k] = static_cast<int>(bi);
      } else if (bi < a.k_blocks) {
        ids[k] = a.block_ids[static_cast<int64_t>(tp.b) * a.k_blocks + bi];
      }
    }
  };
  auto fetch_pages = [&](const TilePos& first, const int (&ids)[kRounds],
                         int64_t (&phys)[kRounds]) {
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      phys[k] = -1;
      if (!paged || ids[k] < 0) continue;
      TilePos tp = first;
      tp.advance(2 * (2 * k + (lane >> 4)), q_rows);
      phys[k] = paged_row(a.pages, tp.b, int64_t{ids[k]} * kBlock);
    }
  };
  TilePos first;  // the stage's first tile
  first.init(t_begin + half, tpq);
  int blk[kRounds], blk1[kRounds];  // groups of this stage and of the next
  int64_t phys[kRounds];            // (paged) their rows in the pool
  fetch_blocks(first, 0, blk);
  fetch_pages(first, blk, phys);
  TilePos next = first;
  next.advance(2 * TPS, q_rows);
  fetch_blocks(next, TPS, blk1);
  // Visible latents of a query, cached for the last query asked about: a
  // lane's tiles move through the queries in order.
  int nv_b = -1, nv = 0;
  auto n_vis_of = [&](int b) -> int {
    if (b != nv_b) {
      nv = visible_latents(a, b);
      nv_b = b;
    }
    return nv;
  };
  int s = 0;           // stage of this iteration
  bool waited = !a.defer_wait;  // the dependency wait has been taken
  const uint64_t pol = l2_evict_first_policy();  // keys are read once a launch
  uint32_t kpar = 0;   // parity of the stage's use count
  for (int64_t j0 = 0; j0 < n_own; j0 += TPS) {
    TilePos next2 = next;
    next2.advance(2 * TPS, q_rows);
    int blk2[kRounds];
    fetch_blocks(next2, j0 + 2 * TPS, blk2);
    int64_t phys1[kRounds];
    fetch_pages(next, blk1, phys1);
    if (j0 >= static_cast<int64_t>(TPS) * R::kStages &&
        !mbar_wait_abortable(&sh.raw_empty[half][s], kpar ^ 1u, &sh.abort, a.status, SITE_SCAN)) {
      return;
    }
    const uint32_t stage = sbase + Lo::kRaw + (half * R::kStages + s) * R::kRawStride;
    uint64_t* full = &sh.raw_full[half][s];
    if (gather) {
      int nrows[kRounds];
      int64_t y[kRounds];
      uint32_t vm[kRounds][4];
      uint32_t bytes = 0;
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
        const int t = 2 * k + (lane >> 4);
        nrows[k] = 0;
        y[k] = 0;
        if (blk[k] >= 0) {
          TilePos tp = first;
          tp.advance(2 * t, q_rows);
          // logical first row of the group and the rows the query has there
          const int64_t t0 = static_cast<int64_t>(blk[k]) * kBlock;
          const int n_vis = n_vis_of(tp.b);
          const int64_t v = (a.mode == ROWS_BLOCKS ? contiguous_rows(a, n_vis) : n_vis) - t0;
          if (v > 0) {
            nrows[k] = static_cast<int>(v < kBlock ? v : kBlock);
            y[k] = seq_row0(a, tp.b) + t0;
            if (paged) {
              y[k] = phys[k];
              if (y[k] < 0) {
                nrows[k] = 0;  // its scores stay -inf
                record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_SCAN, static_cast<uint32_t>(tp.b));
              }
            }
            if (nrows[k] > 0 &&
                !DSA_DCHECK(y[k] >= 0 && y[k] + nrows[k] <= a.key_rows, a.status, SITE_SCAN, y[k])) {
              nrows[k] = 0;
            }
          }
        }
        const int row0 = (lane & 15) * kBlock;
        bytes += nrows[k] > 0 ? kBlock * P::kRowBytes : 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) vm[k][w] = range_bits(w, row0, row0 + nrows[k]);
        // the tile's rows: OR over its 16 lanes
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
          for (int w = 0; w < 4; ++w) vm[k][w] |= __shfl_xor_sync(0xFFFFFFFFu, vm[k][w], o);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xFFFFFFFFu, bytes, o);
      // lane 0 records every tile's rows (tile 2k + 1's come from lane 16)
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t hi = __shfl_sync(0xFFFFFFFFu, vm[k][w], 16);
          if (lane == 0) {
            sh.meta[half][s][2 * k].valid[w] = vm[k][w];
            if (2 * k + 1 < TPS) sh.meta[half][s][2 * k + 1].valid[w] = hi;
          }
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(full, bytes);
      __syncwarp();
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
        if (nrows[k] <= 0) continue;
        const int t = 2 * k + (lane >> 4);
        const int row0 = (lane & 15) * kBlock;
        const uint32_t codes = R::codes(stage, t);
        if constexpr (FMT == DSA_FMT_BF16) {
          // two K halves (64 elements = 128 bytes each) into the two K-atoms
          tma_load_2d_hint(codes + row0 * 128, &maps.keys, 0, static_cast<int>(y[k]), full, pol);
          tma_load_2d_hint(codes + kTile * 128 + row0 * 128, &maps.keys, 64,
                           static_cast<int>(y[k]), full, pol);
        } else {
          if constexpr (FMT == DSA_FMT_MXFP8) {
            tma_load_2d_hint(codes + row0 * 128, &maps.keys, 0, static_cast<int>(y[k]), full,
                             pol);
          } else {
            tma_load_2d_hint(codes + row0 * 64, &maps.keys, 0, static_cast<int>(y[k] >> 1), full,
                             pol);
          }
          const uint32_t sc_dst = R::scales(stage, t) + row0 * 4;
          const uint8_t* sc_src = a.key_scales + y[k] * 4;
          if (scale_vec && nrows[k] == kBlock) {
            cp_async_16_hint(sc_dst, sc_src, pol);
            cp_async_16_hint(sc_dst + 16, sc_src + 16, pol);
          } else {
            for (int r = 0; r < nrows[k]; ++r) cp_async_4(sc_dst + r * 4, sc_src + r * 4);
          }
        }
      }
    } else {
      // Contiguous rows: the same values in every lane; lane 0 issues the boxes.
      int nrows[TPS];
      uint32_t bytes = 0;
      bool tail = false;  // a tile of the stage reaches its sequence's last row
#pragma unroll
      for (int t = 0; t < TPS; ++t) {
        nrows[t] = 0;
        if (j0 + t < n_own) {
          TilePos tp = first;
          tp.advance(2 * t, q_rows);
          int64_t v = contiguous_rows(a, n_vis_of(tp.b)) - tp.r0;
          tail = tail || (v > 0 && v <= kTile);
          v = v < 0 ? 0 : (v > kTile ? kTile : v);
          nrows[t] = static_cast<int>(v);
          const int64_t row = seq_row0(a, tp.b) + tp.r0;
          if (nrows[t] > 0 &&
              !DSA_DCHECK(row >= 0 && row + nrows[t] <= a.key_rows, a.status, SITE_SCAN, row)) {
            nrows[t] = 0;
          }
        }
        const bool bulk_sc = FMT != DSA_FMT_BF16 && scale_vec && nrows[t] == kTile;
        bytes += (nrows[t] > 0 ? P::kCodeBytes : 0) + (bulk_sc ? P::kScaleBytes : 0);
      }
      if (tail && !waited) {
        griddep_wait();  // the tail pool has written the last blocks (all lanes)
        waited = true;
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TPS; ++t) {
#pragma unroll
          for (int w = 0; w < 4; ++w) sh.meta[half][s][t].valid[w] = range_bits(w, 0, nrows[t]);
        }
        mbar_arrive_expect_tx(full, bytes);
      }
#pragma unroll
      for (int t = 0; t < TPS; ++t) {
        if (nrows[t] == 0) continue;
        TilePos tp = first;
        tp.advance(2 * t, q_rows);
        const int64_t row = seq_row0(a, tp.b) + tp.r0;
        const uint32_t codes = R::codes(stage, t);
        const bool bulk_sc = FMT != DSA_FMT_BF16 && scale_vec && nrows[t] == kTile;
        if (lane == 0) {
          if constexpr (FMT == DSA_FMT_BF16) {
            tma_load_2d_hint(codes, &maps.keys, 0, static_cast<int>(row), full, pol);
            tma_load_2d_hint(codes + kTile * 128, &maps.keys, 64, static_cast<int>(row), full,
                             pol);
          } else if constexpr (FMT == DSA_FMT_MXFP8) {
            tma_load_2d_hint(codes, &maps.keys, 0, static_cast<int>(row), full, pol);
          } else {
            tma_load_2d_hint(codes, &maps.keys, 0, static_cast<int>(row >> 1), full, pol);
          }
          if (bulk_sc) {
            bulk_g2s_hint(R::scales(stage, t), a.key_scales + row * 4, P::kScaleBytes, full,
                          pol);
          }
        }
        if constexpr (FMT != DSA_FMT_BF16) {
          if (!bulk_sc) {
            // lane l copies the scales of rows l, l + 32, l + 64, l + 96
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = lane + 32 * k;
              if (r < nrows[t]) {
                cp_async_4(R::scales(stage, t) + r * 4, a.key_scales + (row + r) * 4);
              }
            }
          }
        }
      }
    }
    cp_async_mbar_arrive_noinc(full);
    first = next;
    next = next2;
#pragma unroll
    for (int k = 0; k < kRounds; ++k) {
      blk[k] = blk1[k];
      phys[k] = phys1[k];
      blk1[k] = blk2[k];
    }
    if (++s == R::kStages) {
      s = 0;
      kpar ^= 1u;
    }
  }
}

template <int FMT, int TPS>
__device__ void mma_issuer(const ScanArgs& a, Shared& sh, uint32_t sbase, int n_tiles, int set) {
  using P = Plan<FMT>;
  using R = Ring<FMT, TPS>;
  using Lo = Layout<FMT, TPS>;
  static_assert(FMT != DSA_FMT_BF16 || TPS == 1, "bf16 tiles are read by the MMA, one a stage");
  constexpr uint32_t idesc = mma_idesc(kTile, kIdxHeads, FMT == DSA_FMT_BF16, false, false);
  const uint32_t tmem = sh.tmem_base;
  int stage = 0;  // bf16: raw stage of the half of tile i (advances per own tile)
  for (int i = set; i < n_tiles; i += 2) {
    const int q = i & (kSlots - 1);
    const uint32_t u = static_cast<uint32_t>(i >> 2);
    // op_full(i) also means the slot's accumulator is free: the set that
    // prepares tile i read tile i - 4's accumulator before (program order,
    // with the tcgen05 fence before its arrival).
    if (!mbar_wait_abortable(&sh.op_full[q], u & 1, &sh.abort, a.status, SITE_SCAN)) return;
    tc_fence_after();
    // the tile's index query: the slot its math set wrote before arriving
    const uint32_t qb = sbase + Lo::kQ + (set * kQRing + sh.tile_slot[q]) * 4096;
    const uint64_t bd0 = sw128_desc(qb, 16, 1024);
    const uint32_t slot = tmem + q * P::kSlotCols;
    if constexpr (FMT == DSA_FMT_BF16) {
      const uint32_t raw = sbase + Lo::kRaw + (set * R::kStages + stage) * R::kRawStride;
      const uint64_t ad0 = sw128_desc(raw, 16, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // K = 128 in steps of 16
        const uint64_t ad = ad0 + (((k >> 2) * (kTile * 128) + (k & 3) * 32) >> 4);
        const uint64_t bd = bd0 + (((k >> 2) * 2048 + (k & 3) * 32) >> 4);
        mma_f16(slot, ad, bd, idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(&sh.acc_full[q]);
      mma_commit(&sh.raw_empty[set][stage]);
    } else {
      // A in tensor memory: columns [slot, slot + 64) hold the row's 128 f16
      // values in pairs; group g = k / 2 accumulates into columns 64 + 16 g.
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t bd = bd0 + (((k >> 2) * 2048 + (k & 3) * 32) >> 4);
        mma_f16_tmem_a(slot + 64 + (k >> 1) * 16, slot + k * 8, bd, idesc, (k & 1) ? 1u : 0u);
      }
      mma_commit(&sh.acc_full[q]);
    }
    if (++stage == R::kStages) stage = 0;
  }
}

// Index query of query b -> ring slot [set][ring] (one math set, 128 threads).
// A query's index vectors and weight as one math thread of a set loads them
// (the loads go out when the fetch is made and are used when the query's ring
// slot is built, so a fetch made a tile ahead hides their latency).
struct QFetch {
  int b;  // the query (-1: none)
  uint4 v0, v1;
  float w;
};
__device__ __forceinline__ uint4 ld_global_v4_early(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
template <int FMT>
__device__ __forceinline__ QFetch fetch_query(const ScanArgs& a, int b, int mt) {
  QFetch f;
  f.b = b;
  const uint16_t* q = a.q_idx + static_cast<int64_t>(b) * kIdxHeads * kIdxDim;
  if constexpr (FMT == DSA_FMT_BF16) {
    // thread mt: 16-byte chunks c = mt and mt + 128 (head c / 16, chunk c % 16)
    f.v0 = ld_global_v4_early(q + (mt >> 4) * kIdxDim + (mt & 15) * 8);
    const int c1 = mt + kMathThreads;
    f.v1 = ld_global_v4_early(q + (c1 >> 4) * kIdxDim + (c1 & 15) * 8);
  } else {
    const int h = mt >> 3, part = mt & 7;  // 8 threads per head, 16 elements each
    f.v0 = ld_global_v4_early(q + h * kIdxDim + part * 16);
    f.v1 = ld_global_v4_early(q + h * kIdxDim + part * 16 + 8);
  }
  f.w = 0.f;
  if (mt < kIdxHeads) {
    asm volatile("ld.global.nc.f32 %0, [%1];\n"
                 : "=f"(f.w)
                 : "l"(a.w + static_cast<int64_t>(b) * kIdxHeads + mt));
  }
  return f;
}

// Query f.b's index vectors -> ring slot [set][ring] (one math set, 128 threads).
template <int FMT, int TPS>
__device__ void build_query(Shared& sh, uint32_t sbase, const QFetch& f, int mt, int set,
                            int ring) {
  using Lo = Layout<FMT, TPS>;
  const uint32_t qb = sbase + Lo::kQ + (set * kQRing + ring) * 4096;
  QSlot& slot = sh.qs[set][ring];
  if (mt < kIdxHeads) slot.w[mt] = f.w;
  if constexpr (FMT == DSA_FMT_BF16) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = mt + kMathThreads * j;
      const int h = c >> 4, cr = c & 15;
      st_shared_v4(qb + (cr >> 3) * 2048 + sw128_off(h, cr & 7), j == 0 ? f.v0 : f.v1);
    }
    if (mt < kIdxHeads) slot.qinv[mt] = 1.0f;
  } else {
    const int h = mt >> 3, part = mt & 7;  // 8 threads per head, 16 elements each
    const uint32_t wv[8] = {f.v0.x, f.v0.y, f.v0.z, f.v0.w, f.v1.x, f.v1.y, f.v1.z, f.v1.w};
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_bits_to_float(wv[i] & 0xFFFF);
      x[2 * i + 1] = bf16_bits_to_float(wv[i] >> 16);
      amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    int s = 0;
    if (amax > 0.f) {
      const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // floor(log2)
      s = min(126, max(-126, 14 - e));
    }
    const float up = __uint_as_float(static_cast<uint32_t>(127 + s) << 23);
    uint32_t hw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __half2 hv = __floats2half2_rn(x[2 * i] * up, x[2 * i + 1] * up);
      hw[i] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    const int c0 = 2 * part;  // f16 chunks c0, c0 + 1 of row h
    st_shared_v4(qb + (c0 >> 3) * 2048 + sw128_off(h, c0 & 7),
                 make_uint4(hw[0], hw[1], hw[2], hw[3]));
    st_shared_v4(qb + ((c0 + 1) >> 3) * 2048 + sw128_off(h, (c0 + 1) & 7),
                 make_uint4(hw[4], hw[5], hw[6], hw[7]));
    if (part == 0) slot.qinv[h] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  }
}

template <int FMT, int TPS>
__device__ void math(const ScanArgs& a, Shared& sh, uint32_t sbase, int64_t t_begin,
                     int n_tiles, int64_t tpq) {
  using P = Plan<FMT>;
  using R = Ring<FMT, TPS>;
  using Lo = Layout<FMT, TPS>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int set = (warp - kMathWarp0) >> 2;               // tiles i with i % 2 == set
  const int mt = threadIdx.x - 32 * kMathWarp0 - kMathThreads * set;  // 0..127 within the set
  const int row = 32 * (warp & 3) + lane;  // TMEM lane = key row of this thread
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const uint32_t tmem = sh.tmem_base;
  const int64_t q_rows = tpq * kTile;
  // per-thread state of this set's two tiles waiting for their epilogue
  uint32_t pend_sc0 = 0, pend_sc1 = 0;
  bool pend_valid0 = false, pend_valid1 = false;
  TilePos prep, epi;  // positions of this set's next prepared and next finished tile
  prep.init(t_begin + set, tpq);
  epi = prep;
  // Index-query slots follow the queries: a query's tiles share one slot,
  // and a tile of another query builds the next slot (last used by a tile at
  // least three own tiles back, whose epilogue is done).
  int cur_b = -1, cur_slot = kQRing - 1;
  int pend_slot0 = 0, pend_slot1 = 0;  // of the two tiles waiting for their epilogue
  int stage = 0;                 // ring stage of the tile being prepared (advances per TPS
  uint32_t spar = 0;             // own tiles) and the parity of that stage's use
  // The query of this set's next tile of another query, fetched one own tile
  // ahead.
  QFetch nq;
  nq.b = -1;
  if (set < n_tiles) nq = fetch_query<FMT>(a, prep.b, mt);

  auto epilogue = [&](int e) -> bool {
    const int q = e & (kSlots - 1);
    const int pe = (e >> 1) & 1;
    const int b = epi.b;
    const int64_t r = epi.r0 + row;
    if (!mbar_wait_abortable(&sh.acc_full[q], static_cast<uint32_t>((e >> 2) & 1), &sh.abort,
                             a.status, SITE_SCAN)) {
      return false;
    }
    tc_fence_after();
    const uint32_t acc = tmem + lane_base + q * P::kSlotCols + (P::kSlotCols - P::kAccCols);
    float dot[kIdxHeads];
    if constexpr (FMT == DSA_FMT_BF16) {
      tmem_ld16(acc, dot);
    } else {
      float v[64];
      tmem_ld64(acc, v);
#pragma unroll
      for (int h = 0; h < kIdxHeads; ++h) dot[h] = 0.f;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t sc = ((pe ? pend_sc1 : pend_sc0) >> (8 * g)) & 0xFF;
        const float f = __uint_as_float(sc == 0 ? 0x00400000u : sc << 23);
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) dot[h] = fmaf(v[16 * g + h], f, dot[h]);
      }
    }
    tc_fence_before();
    const QSlot& slot = sh.qs[set][pe ? pend_slot1 : pend_slot0];
    if (r < a.n_rows) {
      float s = -INFINITY;
      if (pe ? pend_valid1 : pend_valid0) {
        s = 0.f;
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) {
          s = fmaf(slot.w[h], fmaxf(dot[h] * slot.qinv[h], 0.f), s);
        }
      }
      a.scores[static_cast<int64_t>(b) * a.n_rows + r] = s;
    }
    epi.advance(2, q_rows);
    return true;
  };

  // Own tiles i = set, set + 2, ...: the epilogue of tile i - 4 (which shares
  // tile i's pending entry and TMEM slot), then the preparation of tile i.
  // The loop is unrolled by U = max(2, TPS) own tiles so that the two pending
  // entries (parity pi) are distinct registers (the MX scale load issued here
  // is first used two own tiles later and its latency stays hidden) and the
  // tile's place t in its ring stage is known at compile time.
  auto own_tile = [&](int i, auto pic, auto tc) -> bool {
    constexpr int pi = decltype(pic)::value;
    constexpr int t = decltype(tc)::value;
    if (i >= 4 && i - 4 < n_tiles) {
      if (!epilogue(i - 4)) return false;
    }
    if (i >= n_tiles) return true;
    const int q = i & (kSlots - 1);
    const int b = prep.b;
    if (b != cur_b) {
      // The next slot last served a tile at most i - 6 (each slot holds one
      // query, and the two slots since hold the queries of tiles i - 4 and
      // i - 2 at the latest), whose epilogue every thread of the set has
      // finished once all of them reach this barrier.
      const int ns = cur_slot + 1 == kQRing ? 0 : cur_slot + 1;
      if (nq.b != b) nq = fetch_query<FMT>(a, b, mt);
      named_sync(1 + set, kMathThreads);
      build_query<FMT, TPS>(sh, sbase, nq, mt, set, ns);
      fence_proxy_async_smem();
      named_sync(1 + set, kMathThreads);
      cur_b = b;
      cur_slot = ns;
    }
    if constexpr (pi) pend_slot1 = cur_slot; else pend_slot0 = cur_slot;
    if (mt == 0) sh.tile_slot[q] = cur_slot;  // read by the MMA issuer after op_full[q]
    if (t == 0 && !mbar_wait_abortable(&sh.raw_full[set][stage], spar, &sh.abort, a.status,
                                       SITE_SCAN)) {
      return false;
    }
    const TileMeta& m = sh.meta[set][stage][t];
    const bool valid_i = (m.valid[row >> 5] >> (row & 31)) & 1u;
    if constexpr (pi) pend_valid1 = valid_i; else pend_valid0 = valid_i;
    if constexpr (FMT != DSA_FMT_BF16) {
      const uint32_t st_base = sbase + Lo::kRaw + (set * R::kStages + stage) * R::kRawStride;
      const uint32_t raw = R::codes(st_base, t);
      // The A slot of tile i was last read by the MMA of tile i - 4, which the
      // epilogue above has already seen complete (its acc_full commit).
      // Own row to f16 pairs: word j holds elements 2j, 2j + 1.
      uint32_t f[64];
      if constexpr (FMT == DSA_FMT_MXFP8) {
        // 8 chunks of 16 codes at their swizzled positions
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = ld_shared_v4(raw + sw128_off(row, c));
          asm("{\n .reg .b16 a, b, c, d, e, f, g, h;\n"
              " mov.b32 {a, b}, %8;\n mov.b32 {c, d}, %9;\n"
              " mov.b32 {e, f}, %10;\n mov.b32 {g, h}, %11;\n"
              " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n"
              " cvt.rn.f16x2.e4m3x2 %2, c;\n cvt.rn.f16x2.e4m3x2 %3, d;\n"
              " cvt.rn.f16x2.e4m3x2 %4, e;\n cvt.rn.f16x2.e4m3x2 %5, f;\n"
              " cvt.rn.f16x2.e4m3x2 %6, g;\n cvt.rn.f16x2.e4m3x2 %7, h;\n}\n"
              : "=r"(f[8 * c + 0]), "=r"(f[8 * c + 1]), "=r"(f[8 * c + 2]), "=r"(f[8 * c + 3]),
                "=r"(f[8 * c + 4]), "=r"(f[8 * c + 5]), "=r"(f[8 * c + 6]), "=r"(f[8 * c + 7])
              : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
        }
      } else {
        // the row is half of 128-byte row row / 2: its 4 chunks of 32 codes
        // (two a byte, element 2j in the low nibble of byte j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = ld_shared_v4(raw + sw128_off(row >> 1, 4 * (row & 1) + c));
          const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %4;\n"
                " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n"
                " cvt.rn.f16x2.e2m1x2 %2, c;\n cvt.rn.f16x2.e2m1x2 %3, d;\n}\n"
                : "=r"(f[16 * c + 4 * k + 0]), "=r"(f[16 * c + 4 * k + 1]),
                  "=r"(f[16 * c + 4 * k + 2]), "=r"(f[16 * c + 4 * k + 3])
                : "r"(vw[k]));
          }
        }
      }
      // The row's four group scales (one 32-bit word): loaded now, used by the
      // epilogue two own tiles later, so the load's latency is hidden.
      uint32_t& sc_i = pi ? pend_sc1 : pend_sc0;
      asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(sc_i) : "r"(R::scales(st_base, t) + row * 4));
      tmem_st64(tmem + lane_base + q * P::kSlotCols, f);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the stage is free once its last tile is converted
        if (t == TPS - 1) mbar_arrive(&sh.raw_empty[set][stage]);
        mbar_arrive(&sh.op_full[q]);
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.op_full[q]);
    }
    prep.advance(2, q_rows);
    if (i + 2 < n_tiles && prep.b != b && nq.b != prep.b) nq = fetch_query<FMT>(a, prep.b, mt);
    if (t == TPS - 1 && ++stage == R::kStages) {
      stage = 0;
      spar ^= 1u;
    }
    return true;
  };
  using I0 = std::integral_constant<int, 0>;
  using I1 = std::integral_constant<int, 1>;
  using I2 = std::integral_constant<int, 2>;
  using I3 = std::integral_constant<int, 3>;
  if constexpr (TPS <= 2) {
    // Own tiles taken two at a time (parities 0, 1; stage places 0, TPS - 1).
    using T1 = std::integral_constant<int, TPS - 1>;
    for (int i = set; i < n_tiles + 4; i += 4) {
      if (!own_tile(i, I0{}, I0{})) return;
      if (!own_tile(i + 2, I1{}, T1{})) return;
    }
  } else {
    // Four at a time: one ring stage.
    for (int i = set; i < n_tiles + 4; i += 8) {
      if (!own_tile(i, I0{}, I0{})) return;
      if (!own_tile(i + 2, I1{}, I1{})) return;
      if (!own_tile(i + 4, I0{}, I2{})) return;
      if (!own_tile(i + 6, I1{}, I3{})) return;
    }
  }
}

template <int FMT, int TPS>
__global__ void __launch_bounds__(kThreads, 1)
    scan_kernel(ScanArgs a, const __grid_constant__ Maps maps, int64_t tpq, int64_t total) {
  using P = Plan<FMT>;
  using R = Ring<FMT, TPS>;
  using Lo = Layout<FMT, TPS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + (sbase - raw) + Lo::kShared);
  const int warp = threadIdx.x >> 5;
  griddep_launch_dependents();

  const int64_t per = total / gridDim.x, rem = total % gridDim.x;
  const int64_t bx = blockIdx.x;
  const int64_t t_begin = bx * per + (bx < rem ? bx : rem);
  const int n_tiles = static_cast<int>(per + (bx < rem ? 1 : 0));

  if (threadIdx.x == 0) {
    for (int h = 0; h < 2; ++h) {
      for (int s = 0; s < R::kStages; ++s) {
        // raw_full: the producer's expect_tx arrival + one cp.async arrival per lane
        mbar_init(&sh.raw_full[h][s], 1 + 32);
        // raw_empty: the MMA's commit (bf16), or the four warps of the math set
        // once they converted the stage's last tile (MX formats)
        mbar_init(&sh.raw_empty[h][s], FMT == DSA_FMT_BF16 ? 1 : 4);
      }
    }
    for (int q = 0; q < kSlots; ++q) {
      mbar_init(&sh.op_full[q], 4);
      mbar_init(&sh.acc_full[q], 1);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&sh.tmem_base, P::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The previous kernel's outputs (scores, ids, pooled keys) are final past
  // this wait; with defer_wait only the producer takes it, before the tiles
  // that the tail pool writes (nothing else here reads a library output).
  if (!a.defer_wait) griddep_wait();

  if (warp < kMmaWarp) {
    producer<FMT, TPS>(a, maps, sh, sbase, t_begin, n_tiles, tpq, warp);
  } else if (warp == kMmaWarp || warp == kMmaWarp2) {
    if ((threadIdx.x & 31) == 0) {
      mma_issuer<FMT, TPS>(a, sh, sbase, n_tiles, warp == kMmaWarp ? 0 : 1);
    }
    __syncwarp();
  } else {
    math<FMT, TPS>(a, sh, sbase, t_begin, n_tiles, tpq);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, P::kTmemCols);
  }
}

template <int FMT, int TPS>
cudaError_t launch_fmt(const ScanArgs& args, int num_sms, cudaStream_t s) {
  ScanArgs a = args;
  using Lo = Layout<FMT, TPS>;
  const int64_t tpq = (a.n_rows + kTile - 1) / kTile;
  const int64_t total = tpq * a.B;
  if (total == 0) return cudaSuccess;
  // Rows the tensor map covers: every sequence's stride, and only the last
  // sequence's own rows (a box reaching past them reads zeros). MXFP4 arrays
  // are read in pairs of rows; the caller's buffer holds whole pairs.
  int64_t last_rows;
  if (a.mode == ROWS_BLOCKS) {
    last_rows = a.prefill ? a.max_latents / 8 : (a.max_latents + 7) / 8;
  } else {
    last_rows = a.max_latents;
  }
  // A paged cache: the whole pool.
  const int64_t n_seqs = a.mq > 0 ? a.B / a.mq : (a.prefill ? 1 : a.B);
  const int64_t rows = a.pages.table ? a.pages.n_pages * a.pages.rows
                                     : (n_seqs - 1) * a.key_stride + last_rows;
  a.key_rows = rows;
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  const int box_rows = (a.mode == ROWS_GATHER || a.pages.table) ? kBlock : kTile;
  cudaError_t e = cudaSuccess;
  if (rows > 0) {
    if (FMT == DSA_FMT_BF16) {
      e = encode_tma_2d(&maps.keys, a.key_data, /*elem_bytes=*/2, /*inner=*/128, rows,
                        /*row_bytes=*/256, /*box_inner=*/64, box_rows);
    } else if (FMT == DSA_FMT_MXFP8) {
      e = encode_tma_2d(&maps.keys, a.key_data, 1, 128, rows, 128, 128, box_rows);
    } else {
      e = encode_tma_2d(&maps.keys, a.key_data, 1, 128, (rows + 1) / 2, 128, 128, box_rows / 2);
    }
    if (e != cudaSuccess) return e;
  }
  const int smem = Lo::kBytes + 1024;
  static std::atomic<int> smem_set[64]{};
  e = ensure_smem(reinterpret_cast<const void*>(scan_kernel<FMT, TPS>), smem, smem_set);
  if (e != cudaSuccess) return e;
  const int64_t grid = total < num_sms ? total : num_sms;
  return launch_pdl(scan_kernel<FMT, TPS>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem,
                    s, 1, a, maps, tpq, total);
}

}  // namespace

// Tiles per ring stage: bf16 tiles are 32 KB already; MXFP8 tiles (16.5 KB)
// go two a stage, and so do MXFP4 tiles (8.5 KB): a stage is released only
// once its last tile is converted, and four MXFP4 tiles a stage (two stages a
// half) left the scans pipeline-bound at ~0.65 us a tile (the 64 x 131072
// step 117.0 us against 103.8 with two a stage, three stages a half).
// Gathered MXFP8 scans take DSA_SCAN_GATHER_TPS tiles a stage.
cudaError_t launch_scan(const ScanArgs& args, int num_sms, cudaStream_t s) {
  const bool gather = args.mode == ROWS_GATHER || args.pages.table != nullptr;
  ScanArgs a = args;
  // the deferred wait covers the contiguous decode block stage only
  if (gather || a.mode != ROWS_BLOCKS || a.prefill || a.mq > 0) a.defer_wait = 0;
  if (a.fmt == DSA_FMT_BF16) return launch_fmt<DSA_FMT_BF16, 1>(a, num_sms, s);
  if (a.fmt == DSA_FMT_MXFP8) {
    if (gather) return launch_fmt<DSA_FMT_MXFP8, DSA_SCAN_GATHER_TPS>(a, num_sms, s);
    return launch_fmt<DSA_FMT_MXFP8, 2>(a, num_sms, s);
  }
  if (a.fmt == DSA_FMT_MXFP4) {
    if (gather) return launch_fmt<DSA_FMT_MXFP4, DSA_SCAN_MXFP4_GATHER_TPS>(a, num_sms, s);
    return launch_fmt<DSA_FMT_MXFP4, DSA_SCAN_MXFP4_TPS>(a, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dsa
