// S1 / S3 of a prefill chunk with bf16 keys, batched over queries: every
// query of the chunk scores rows of one shared key array (the pooled block
// keys, or every latent's index key), so sixteen queries share each key tile
// and one tcgen05 MMA computes all their heads at once:
//   acc[key][16 q + h] = k . q_idx(q, h)   (M = 128 keys, N = 256, K = 128)
// and the epilogue forms score(q, key) = sum_h w_{q,h} * max(0, acc), in head
// order, for the keys query q may see (-inf otherwise). The indexer formula
// is that of recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier
// sparse attention" (score = sum_h w_h ReLU(q_h . k), the reading this library
// fixes); it is the same contraction as the per-query scan, sixteen times
// wider (a per-query N = 16 MMA costs nearly as much as an N = 256 one).
//
// Work items are (group of 16 queries, tile of 128 rows), group-major; each
// persistent CTA takes a contiguous range of items, so it reloads a group's
// index queries (64 KB) and weights only when the group changes. Tiles that no
// query of a group can see are skipped by every role alike.
//   warp 0     producer: TMA loads of key tiles (4 stages of 32 KB) and of
//              each group's index queries (B operand, 64 KB) and weights;
//   warp 1     MMA issuer (one thread), tensor-memory owner: two accumulators
//              of 256 columns, so one tile's epilogue overlaps the next MMA;
//   warps 2-17 epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its key
//              rows) and the columns of queries 4 ((w - 2) / 4) .. + 3 (the
//              head sums of 16 queries per key row are the kernel's longest
//              step, so they are spread over sixteen warps).
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kTile = 128;       // key rows per tile (MMA M)
constexpr int kGroup = 16;       // queries per group
constexpr int kN = kGroup * kIdxHeads;  // 256 MMA columns
constexpr int kStages = 4;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);  // 320
constexpr int kTileBytes = kTile * kIdxDim * 2;          // 32 KB: two K-atoms of 16 KB
constexpr int kQBytes = kN * kIdxDim * 2;                // 64 KB: two K-atoms of 32 KB
constexpr int kTmemCols = 2 * kN;                        // two accumulators

struct Shared {
  uint64_t a_full[kStages], a_empty[kStages];
  uint64_t b_full, grp_done;
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort;
  alignas(16) float w[kGroup * kIdxHeads];  // the current group's weights (bulk copy target)
};

constexpr int kA = 0;                               // [stage] key tiles
constexpr int kB = kA + kStages * kTileBytes;       // the group's index queries
constexpr int kShared = kB + kQBytes;
constexpr int kSmemBytes = kShared + static_cast<int>(sizeof(Shared)) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct Maps {
  CUtensorMap keys;  // bf16 [rows][128], box {64, 128}
  CUtensorMap q;     // bf16 [n_q * 16][128], box {64, 256}
};

// Keys query q (position ctx + q) may see: its visible latents, or (blocks)
// its complete blocks; a partially visible block is scored elsewhere.
__device__ __forceinline__ int64_t visible_rows(const BatchedScanArgs& a, int64_t q) {
  const int64_t n_vis = (a.ctx + q + 1) / a.ratio;
  return a.mode == ROWS_BLOCKS ? n_vis / kBlock : n_vis;
}

// Rows of group g's score rows the kernel writes: every row for block scores
// (the selection reads them all); for latent scores, up to the end of the
// last visible block of the group's last query (the token selection reads
// only tokens of selected blocks).
__device__ __forceinline__ int64_t cover_rows(const BatchedScanArgs& a, int g) {
  if (a.mode == ROWS_BLOCKS) return a.n_cols;
  const int64_t q_last = min(static_cast<int64_t>(g) * kGroup + kGroup, a.n_q) - 1;
  const int64_t r = (visible_rows(a, q_last) + kBlock - 1) / kBlock * kBlock;
  return r < a.n_cols ? r : a.n_cols;
}

// Walk over a CTA's items [i0, i1) (item i = group i / T, tile i % T) without
// a division per item; `cover` is the current group's rows to write.
struct Walk {
  int g, t;
  int64_t cover;
  __device__ void init(const BatchedScanArgs& a, int64_t i0, int64_t T) {
    g = static_cast<int>(i0 / T);
    t = static_cast<int>(i0 - static_cast<int64_t>(g) * T);
    cover = cover_rows(a, g);
  }
  __device__ bool skip() const { return static_cast<int64_t>(t) * kTile >= cover; }
  // The tile is the last of its group that this walk visits (before i1).
  __device__ bool group_ends(int64_t i, int64_t i1, int64_t T) const {
    return i + 1 >= i1 || t + 1 == T || static_cast<int64_t>(t + 1) * kTile >= cover;
  }
  __device__ void next(const BatchedScanArgs& a, int64_t T) {
    if (++t == T) {
      t = 0;
      ++g;
      cover = cover_rows(a, g);
    }
  }
};

__device__ void producer(const BatchedScanArgs& a, const Maps& maps, Shared& sh, uint32_t sbase,
                         int64_t i0, int64_t i1, int64_t T) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    tma_prefetch_map(&maps.keys);
    tma_prefetch_map(&maps.q);
  }
  int cur_g = -1, groups = 0, s = 0;
  uint32_t kpar = 0;
  int64_t n_done = 0;
  Walk it;
  it.init(a, i0, T);
  for (int64_t i = i0; i < i1; ++i, it.next(a, T)) {
    if (it.skip()) continue;
    if (it.g != cur_g) {
      // The previous group's epilogue is done (so are its MMAs): B and the
      // weights may be replaced.
      if (groups > 0 && !mbar_wait_abortable(&sh.grp_done, static_cast<uint32_t>((groups - 1) & 1),
                                             &sh.abort, a.status, SITE_SCAN)) {
        return;
      }
      if (lane == 0) {
        const int64_t nq = min(static_cast<int64_t>(kGroup), a.n_q - static_cast<int64_t>(it.g) * kGroup);
        const uint32_t wbytes = static_cast<uint32_t>(nq) * kIdxHeads * 4;
        mbar_arrive_expect_tx(&sh.b_full, kQBytes + wbytes);
        tma_load_2d(sbase + kB, &maps.q, 0, it.g * kN, &sh.b_full);
        tma_load_2d(sbase + kB + kQBytes / 2, &maps.q, 64, it.g * kN, &sh.b_full);
        bulk_g2s(smem_u32(sh.w), a.w + static_cast<int64_t>(it.g) * kGroup * kIdxHeads, wbytes,
                 &sh.b_full);
      }
      __syncwarp();
      cur_g = it.g;
      ++groups;
    }
    if (n_done >= kStages &&
        !mbar_wait_abortable(&sh.a_empty[s], kpar ^ 1u, &sh.abort, a.status, SITE_SCAN)) {
      return;
    }
    if (lane == 0) {
      const uint32_t dst = sbase + kA + s * kTileBytes;
      const int y = it.t * kTile;
      mbar_arrive_expect_tx(&sh.a_full[s], kTileBytes);
      tma_load_2d(dst, &maps.keys, 0, y, &sh.a_full[s]);
      tma_load_2d(dst + kTileBytes / 2, &maps.keys, 64, y, &sh.a_full[s]);
    }
    __syncwarp();
    ++n_done;
    if (++s == kStages) {
      s = 0;
      kpar ^= 1u;
    }
  }
}

__device__ void mma_issuer(const BatchedScanArgs& a, Shared& sh, uint32_t sbase, int64_t i0,
                           int64_t i1, int64_t T) {
  constexpr uint32_t idesc = mma_idesc(kTile, kN, true, false, false);
  const uint32_t tmem = sh.tmem_base;
  int cur_g = -1, groups = 0, s = 0;
  uint32_t kpar = 0;
  int64_t n_done = 0;
  const uint64_t bd0 = sw128_desc(sbase + kB, 16, 1024);
  Walk it;
  it.init(a, i0, T);
  for (int64_t i = i0; i < i1; ++i, it.next(a, T)) {
    if (it.skip()) continue;
    if (it.g != cur_g) {
      if (!mbar_wait_abortable(&sh.b_full, static_cast<uint32_t>(groups & 1), &sh.abort, a.status,
                               SITE_SCAN)) {
        return;
      }
      cur_g = it.g;
      ++groups;
    }
    if (!mbar_wait_abortable(&sh.a_full[s], kpar, &sh.abort, a.status, SITE_SCAN)) return;
    const int slot = static_cast<int>(n_done & 1);
    if (n_done >= 2 && !mbar_wait_abortable(&sh.acc_empty[slot],
                                            static_cast<uint32_t>(((n_done >> 1) - 1) & 1),
                                            &sh.abort, a.status, SITE_SCAN)) {
      return;
    }
    tc_fence_after();
    // Descriptors step by their start-address field (16-byte units; every
    // operand lies below 256 KB, so no carry).
    const uint64_t ad0 = sw128_desc(sbase + kA + s * kTileBytes, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < kIdxDim / 16; ++ks) {
      const uint64_t ad = ad0 + (((ks >> 2) * (kTileBytes / 2) + (ks & 3) * 32) >> 4);
      const uint64_t bd = bd0 + (((ks >> 2) * (kQBytes / 2) + (ks & 3) * 32) >> 4);
      mma_f16(tmem + static_cast<uint32_t>(slot) * kN, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    mma_commit(&sh.acc_full[slot]);
    mma_commit(&sh.a_empty[s]);
    ++n_done;
    if (++s == kStages) {
      s = 0;
      kpar ^= 1u;
    }
  }
}

__device__ void epilogue(const BatchedScanArgs& a, Shared& sh, int64_t i0, int64_t i1, int64_t T) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;                   // TMEM lanes this warp may read
  const int quarter = (warp - kEpiWarp0) >> 2;  // queries 4 quarter .. + 3 of the group
  const int row = 32 * quad + lane;
  const uint32_t tmem = sh.tmem_base;
  const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
  int64_t n_done = 0;
  // Per group: this warp's four queries' visible rows (-1: no such query).
  int cur_g = -1;
  int vis[4];
  Walk it;
  it.init(a, i0, T);
  for (int64_t i = i0; i < i1; ++i, it.next(a, T)) {
    if (it.skip()) continue;
    if (it.g != cur_g) {
      cur_g = it.g;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t q = static_cast<int64_t>(cur_g) * kGroup + 4 * quarter + j;
        vis[j] = q < a.n_q ? static_cast<int>(visible_rows(a, q)) : -1;
      }
    }
    const int slot = static_cast<int>(n_done & 1);
    if (!mbar_wait_abortable(&sh.acc_full[slot], static_cast<uint32_t>((n_done >> 1) & 1),
                             &sh.abort, a.status, SITE_SCAN)) {
      return;
    }
    tc_fence_after();
    const int r = it.t * kTile + row;
    const bool in_cols = r < a.n_cols;
    float* out = a.scores + (static_cast<int64_t>(it.g) * kGroup + 4 * quarter) * a.n_cols + r;
    // One tensor-memory load of the four queries' 64 columns, then the
    // ReLU-weighted head sums in head order.
    {
      float v[64];
      tmem_ld64(tmem + lane_base + static_cast<uint32_t>(slot * kN + 16 * (4 * quarter)), v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = k;
        const int qj = 4 * quarter + j;  // query within the group
        if (vis[j] >= 0 && in_cols) {
          float sc = -INFINITY;
          if (r < vis[j]) {
            sc = 0.f;
            const float4* w4 = reinterpret_cast<const float4*>(sh.w + qj * kIdxHeads);
#pragma unroll
            for (int h4 = 0; h4 < kIdxHeads / 4; ++h4) {
              const float4 ww = w4[h4];
              sc = fmaf(ww.x, fmaxf(v[16 * k + 4 * h4], 0.f), sc);
              sc = fmaf(ww.y, fmaxf(v[16 * k + 4 * h4 + 1], 0.f), sc);
              sc = fmaf(ww.z, fmaxf(v[16 * k + 4 * h4 + 2], 0.f), sc);
              sc = fmaf(ww.w, fmaxf(v[16 * k + 4 * h4 + 3], 0.f), sc);
            }
          }
          // Streaming store (evict first): the score rows must not push the
          // shared key array, re-read by every group, out of L2.
          __stcs(out + j * a.n_cols, sc);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sh.acc_empty[slot]);
      // Last tile of the group in this CTA: the producer may replace B and w.
      if (it.group_ends(i, i1, T)) mbar_arrive(&sh.grp_done);
    }
    ++n_done;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    batched_scan_kernel(BatchedScanArgs a, const __grid_constant__ Maps maps, int64_t T,
                        int64_t total) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw + (sbase - raw) + kShared);
  const int warp = threadIdx.x >> 5;
  griddep_launch_dependents();
  const int64_t per = total / gridDim.x, rem = total % gridDim.x;
  const int64_t bx = blockIdx.x;
  const int64_t i0 = bx * per + (bx < rem ? bx : rem);
  const int64_t i1 = i0 + per + (bx < rem ? 1 : 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.a_full[s], 1);
      mbar_init(&sh.a_empty[s], 1);
    }
    mbar_init(&sh.b_full, 1);
    mbar_init(&sh.grp_done, kEpiWarps);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sh.acc_full[k], 1);
      mbar_init(&sh.acc_empty[k], kEpiWarps);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // the previous kernel's outputs (pooled keys, scores) are final

  if (warp == 0) {
    producer(a, maps, sh, sbase, i0, i1, T);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) mma_issuer(a, sh, sbase, i0, i1, T);
    __syncwarp();
  } else {
    epilogue(a, sh, i0, i1, T);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_scan_batched(const BatchedScanArgs& a, int num_sms, cudaStream_t s) {
  if (a.n_q <= 0 || a.n_cols <= 0) return cudaSuccess;
  if (a.key_rows <= 0) return cudaErrorInvalidValue;
  const int64_t groups = (a.n_q + kGroup - 1) / kGroup;
  const int64_t T = (a.n_cols + kTile - 1) / kTile;
  const int64_t total = groups * T;
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  cudaError_t e = encode_tma_2d(&maps.keys, a.key_data, 2, kIdxDim, static_cast<uint64_t>(a.key_rows),
                                kIdxDim * 2, 64, kTile);
  if (e != cudaSuccess) return e;
  e = encode_tma_2d(&maps.q, a.q_idx, 2, kIdxDim, static_cast<uint64_t>(a.n_q) * kIdxHeads,
                    kIdxDim * 2, 64, kN);
  if (e != cudaSuccess) return e;
  static std::atomic<int> smem_set[64]{};
  e = ensure_smem(reinterpret_cast<const void*>(batched_scan_kernel), kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int64_t grid = total < num_sms ? total : num_sms;
  return launch_pdl(batched_scan_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads),
                    kSmemBytes, s, 1, a, maps, T, total);
}

}  // namespace dsa
