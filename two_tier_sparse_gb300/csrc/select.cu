// S2 / S4: keep the k best candidates of each query by (score desc, index asc)
// (the candidate stage's 2048 blocks and the indexer's best 512 latents,
// recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention";
// ties to the lower index, the rule this library fixes).
//
// One CTA per query (the register-resident kernel: a cluster of 2 or 4 CTAs
// per query while those clusters fit the SMs at once). Scores map to
// order-preserving 32-bit keys (larger score, larger key; -0 as +0). The
// selection then works on exact integers
// t = key - kmin (kmin the smallest valid key of the query):
//   1. a radix select on t with 12-bit digits taken from the top of t's range
//      (so the first histogram already spans the keys' own spread) narrows,
//      level by level, to the digit bin that holds the k-th best key and how
//      many of its members are still needed; it stops once that bin holds at
//      most 256 candidates or all its members share one key;
//   2. a small bin is ranked exactly by (key desc, index asc) and its best
//      members are marked; in a bin of equal keys the first ones in index
//      order are taken;
//   3. one compaction pass in index order writes every key above the bin and
//      the chosen bin members, so ids come out ascending with no sort.
#include <algorithm>

#include "kernels.h"

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;            // 12-bit digits
constexpr int kBinMax = 256;           // bin size that is ranked exactly
constexpr int64_t kCacheMax = 40960;   // keys cached in shared memory (160 KB)

enum Mode { TAKE_ALL = 0, BY_BIN = 1 };

struct SelShared {
  uint32_t hist[kBins];
  uint32_t bin_idx[kBinMax];
  uint32_t bin_key[kBinMax];
  uint32_t warp_a[kWarps], warp_b[kWarps], warp_c[kWarps];
  uint32_t kmin, kmax, n_valid, bstar, need, count, total, mode, take_eq;
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

struct KeySrc {
  const float* sc;
  const uint32_t* cache;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const {
    return cache ? cache[i] : score_key(sc[i]);
  }
};

__global__ void __launch_bounds__(kThreads, 1) select_kernel(SelectArgs a, int use_cache) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ uint32_t cache_mem[];
  __shared__ SelShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = a.n;
  const uint32_t k = static_cast<uint32_t>(a.k);
  const float* sc = a.scores + static_cast<int64_t>(b) * n;

  // Block ids of the token stage, kept in shared memory for the compaction.
  int32_t* bids = reinterpret_cast<int32_t*>(cache_mem + (use_cache ? n : 0));
  if (a.block_ids) {
    // The candidate list must be ascending block ids with -1 padding at the
    // end: the lower-index tie rule and the ascending output rely on it.
    const int32_t* bl = a.block_ids + static_cast<int64_t>(b) * a.k_blocks;
    for (int i = tid; i < a.k_blocks; i += kThreads) {
      const int x = bl[i];
      bids[i] = x;
      if (i + 1 < a.k_blocks) {
        const int y = bl[i + 1];
        if (y >= 0 && (x < 0 || y <= x)) {
          record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_SELECT, static_cast<uint32_t>(i));
        }
      }
    }
  }

  // 1. keys (cached when they fit), valid count, smallest and largest valid
  // key; loads go out eight at a time so their latencies overlap.
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u, cnt = 0;
  constexpr int kBatch = 8;
  for (int64_t base = 0; base < n; base += static_cast<int64_t>(kThreads) * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t i = base + tid + static_cast<int64_t>(j) * kThreads;
      v[j] = i < n ? sc[i] : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t i = base + tid + static_cast<int64_t>(j) * kThreads;
      const uint32_t key = score_key(v[j]);
      if (use_cache && i < n) cache_mem[i] = key;
      if (key > kInvalidKey) {
        kmin = min(kmin, key);
        kmax = max(kmax, key);
        ++cnt;
      }
    }
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (lane == 0) {
    sh.warp_a[warp] = kmin;
    sh.warp_b[warp] = kmax;
    sh.warp_c[warp] = cnt;
  }
  for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
  if (tid == 0) sh.count = 0;
  __syncthreads();
  if (warp == 0) {
    const uint32_t mn = __reduce_min_sync(0xFFFFFFFFu, sh.warp_a[lane]);
    const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, sh.warp_b[lane]);
    const uint32_t c = __reduce_add_sync(0xFFFFFFFFu, sh.warp_c[lane]);
    if (lane == 0) {
      sh.kmin = mn;
      sh.kmax = mx;
      sh.n_valid = c;
      sh.mode = (c <= k) ? TAKE_ALL : BY_BIN;
    }
  }
  __syncthreads();
  const KeySrc key_at{sc, use_cache ? cache_mem : nullptr};
  kmin = sh.kmin;
  const uint32_t span = sh.kmax - kmin;
  // Level state: candidates are valid keys with (t >> hs) == P (hs = 32: all);
  // the final bin is {t : t >> s == P}.
  uint32_t P = 0, s_cur = 32;
  bool ties = false;  // the final bin holds one key value
  if (sh.mode == BY_BIN) {
    uint32_t need = k;
    // first digit: the smallest shift that fits t's range into 12 bits
    uint32_t s_next = span < kBins ? 0u : static_cast<uint32_t>(32 - __clz(span)) - 12u;
    for (int level = 0; level < 4; ++level) {
      const uint32_t hs = s_cur, s_lv = s_next;
      const uint32_t width = hs - s_lv;                // 1..12 bits
      const uint32_t dmask = width >= 32 ? 0xFFFFFFFFu : (1u << width) - 1u;
      for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < n; i += kThreads) {
        const uint32_t key = key_at(i);
        if (key <= kInvalidKey) continue;
        const uint32_t t = key - kmin;
        if (hs < 32 && (t >> hs) != P) continue;
        atomicAdd(&sh.hist[(t >> s_lv) & dmask], 1u);
      }
      __syncthreads();
      // suffix sums from the top digit down: thread t owns digits 4095 - 4t - j
      uint32_t h[4], local = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = sh.hist[kBins - 1 - (4 * tid + j)];
        local += h[j];
      }
      const uint32_t incl = warp_incl_scan(local);
      if (lane == 31) sh.warp_a[warp] = incl;
      __syncthreads();
      uint32_t run = incl - local;
      for (int w = 0; w < warp; ++w) run += sh.warp_a[w];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (run < need && run + h[j] >= need) {
          sh.bstar = static_cast<uint32_t>(kBins - 1 - (4 * tid + j));
          sh.need = need - run;
          sh.count = h[j];
        }
        run += h[j];
      }
      __syncthreads();
      P = (hs < 32 ? (P << width) : 0u) | sh.bstar;
      need = sh.need;
      s_cur = s_lv;
      const uint32_t c = sh.count;
      __syncthreads();
      if (s_lv == 0) {
        ties = true;  // every member of the bin has the same t
        break;
      }
      if (c <= kBinMax) break;
      s_next = s_lv > 12 ? s_lv - 12 : 0;
    }
    if (!ties) {
      // collect the final bin, rank its members exactly, mark the best `need`
      if (tid == 0) sh.count = 0;
      __syncthreads();
      for (int64_t i = tid; i < n; i += kThreads) {
        const uint32_t key = key_at(i);
        if (key > kInvalidKey && ((key - kmin) >> s_cur) == P) {
          const uint32_t slot = atomicAdd(&sh.count, 1u);
          sh.bin_idx[slot] = static_cast<uint32_t>(i);
          sh.bin_key[slot] = key;
        }
      }
      __syncthreads();
      const uint32_t c = sh.count;
      bool take = false;
      if (tid < c) {
        const uint32_t ke = sh.bin_key[tid], ie = sh.bin_idx[tid];
        uint32_t rank = 0;
        for (uint32_t o = 0; o < c; ++o) {
          const uint32_t ko = sh.bin_key[o];
          rank += (ko > ke || (ko == ke && sh.bin_idx[o] < ie)) ? 1u : 0u;
        }
        take = rank < need;
      }
      __syncthreads();  // every rank is computed before any index word is marked
      if (take) sh.bin_idx[tid] |= 0x80000000u;
    } else if (tid == 0) {
      sh.take_eq = need;
    }
    __syncthreads();
  }

  // 3. compaction in index order: each warp owns a contiguous segment
  const uint32_t mode = sh.mode;
  const uint32_t c = ties ? 0u : sh.count;
  // marked members of the final bin are looked up in a bitmap (hist reused)
  uint32_t* marked = sh.hist;
  const bool bitmap = (mode == BY_BIN) && !ties && ((n + 31) / 32 <= kBins);
  if (mode == BY_BIN && !ties) {
    for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    if (bitmap) {
      for (uint32_t e = tid; e < c; e += kThreads) {
        const uint32_t w = sh.bin_idx[e];
        if (w & 0x80000000u) {
          const uint32_t i = w & 0x7FFFFFFFu;
          atomicOr(&marked[i >> 5], 1u << (i & 31));
        }
      }
    }
    __syncthreads();
  }
  auto is_marked = [&](int64_t i) -> bool {
    if (bitmap) return (marked[i >> 5] >> (i & 31)) & 1u;
    for (uint32_t e = 0; e < c; ++e) {
      if (sh.bin_idx[e] == (static_cast<uint32_t>(i) | 0x80000000u)) return true;
    }
    return false;
  };
  auto flags = [&](int64_t i, bool& gt, bool& eq) {
    gt = false;
    eq = false;
    const uint32_t key = key_at(i);
    if (key <= kInvalidKey) return;
    if (mode == TAKE_ALL) {
      gt = true;
      return;
    }
    const uint32_t hi = (key - kmin) >> s_cur;
    if (hi > P) {
      gt = true;
    } else if (hi == P) {
      if (ties) {
        eq = true;
      } else {
        gt = is_marked(i);
      }
    }
  };
  const int64_t seg = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int64_t s0 = static_cast<int64_t>(warp) * seg;
  const int64_t s1 = min(n, s0 + seg);
  uint32_t gt_cnt = 0, eq_cnt = 0;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t i = base + lane;
    bool gt = false, eq = false;
    if (i < s1) flags(i, gt, eq);
    gt_cnt += __popc(__ballot_sync(0xFFFFFFFFu, gt));
    eq_cnt += __popc(__ballot_sync(0xFFFFFFFFu, eq));
  }
  __syncthreads();
  if (lane == 0) {
    sh.warp_a[warp] = gt_cnt;
    sh.warp_b[warp] = eq_cnt;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t take_eq_total = (mode == BY_BIN && ties) ? sh.take_eq : 0u;
    const uint32_t eq = sh.warp_b[lane], gt = sh.warp_a[lane];
    const uint32_t eq_incl = warp_incl_scan(eq);
    const uint32_t eq_before = eq_incl - eq;
    const uint32_t take_eq = take_eq_total > eq_before ? min(eq, take_eq_total - eq_before) : 0u;
    const uint32_t sel = gt + take_eq;
    const uint32_t sel_incl = warp_incl_scan(sel);
    sh.warp_a[lane] = sel_incl - sel;  // output offset of this warp
    sh.warp_b[lane] = take_eq;
    if (lane == 31) sh.total = sel_incl;
  }
  __syncthreads();
  int32_t* out = a.out_ids + static_cast<int64_t>(b) * a.k;
  uint32_t pos = sh.warp_a[warp];
  const uint32_t take_eq = sh.warp_b[warp];
  uint32_t eq_seen = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t i = base + lane;
    bool gt = false, eq = false;
    if (i < s1) flags(i, gt, eq);
    const uint32_t eq_b = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eq_b & lt_mask) < take_eq);
    const uint32_t tb = __ballot_sync(0xFFFFFFFFu, take);
    if (take) {
      int32_t id = static_cast<int32_t>(i);
      if (a.block_ids) id = bids[i >> 3] * 8 + static_cast<int32_t>(i & 7);
      out[pos + __popc(tb & lt_mask)] = id;
    }
    pos += __popc(tb);
    eq_seen += __popc(eq_b);
  }
  const uint32_t total = sh.total;
  for (int64_t j = total + tid; j < a.k; j += kThreads) out[j] = -1;
}

// Register-resident variant for n <= KPT * 1024: warp w owns the contiguous
// candidates [32 KPT w, 32 KPT (w + 1)), lane l holding 32 j + l of them at
// slot j, so every pass runs on registers and each warp lays out its own part
// of the output; only the warps' totals need a block-wide scan.
constexpr int kRankMax = 64;  // final bins at most this large are ranked exactly
// Dense score rows (a prefill chunk's token stage scores every latent): each
// kept block's 8 scores (32 bytes) are copied to shared memory in candidate
// order by asynchronous 16-byte copies, issued as soon as the block ids are in
// registers; the keys are then read without bank conflicts.

// The score a valid order-preserving key stands for (inverse of score_key).
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// Value-space histogram bin: non-decreasing in v for v >= vmin. t =
// (v - vmin) * vscale lies in [0, ~kBins]; adding 2^23 rounds it to an
// integer held in the low mantissa bits (every step is monotone, so the bin
// is), which avoids a float-to-integer conversion.
__device__ __forceinline__ uint32_t value_bin(float v, float vmin, float vscale) {
  const float t = (v - vmin) * vscale + 8388608.f;
  return min(__float_as_uint(t) - 0x4B000000u, static_cast<uint32_t>(kBins - 1));
}

constexpr int kMaxCluster = 4;  // CTAs a query's selection may be split over

// Arrays indexed [source CTA][...] are filled, for every CTA of a cluster, by
// the CTA that owns the values (its own entries locally, the others' by
// stores into their shared memory) before a cluster barrier; after it every
// CTA reads them locally.
struct RegShared {
  alignas(16) uint32_t hist[kBins];
  uint32_t taken[kThreads];  // bit i: candidate i of the final bin is selected (n <= 32 x 1024)
  uint32_t warp_a[kWarps];
  uint4 stat[kMaxCluster][kWarps];      // per warp: smallest and largest valid key, valid count
  uint2 bin[kMaxCluster][kRankMax];     // members of the threshold bin: key, candidate index
  uint2 tot[kMaxCluster][kWarps];       // per warp: candidates output above the bin, tied members
  uint32_t bin_src[kMaxCluster];        // the threshold bin's members in each CTA's share
  uint32_t bstar, need, count, nbin;
};

// Exclusive prefix, over the warps before this one, of the per-warp values
// v[w] (v read from shared memory at lane w), with the total; every warp
// computes it itself, so no second barrier is needed.
__device__ __forceinline__ uint32_t warps_before(uint32_t v_lane, int warp, uint32_t* total) {
  const uint32_t incl = warp_incl_scan(v_lane);
  *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  return __shfl_sync(0xFFFFFFFFu, incl - v_lane, warp);
}

// CL > 1: a query's candidates are split over a cluster of CL CTAs, rank r
// holding [r * KPT * 1024, (r + 1) * KPT * 1024). Through distributed shared
// memory the CTAs exchange their key ranges and valid counts, their members
// of the threshold bin and their output totals (each CTA stores its values
// into every CTA's copy before a cluster barrier), and read one another's
// histograms in place (after a cluster barrier; another comes before a
// histogram is cleared for the next level). Each CTA so takes the decisions
// one CTA over all the candidates would, and writes its own part of the
// ascending output. A cluster barrier costs about as much as a remote read
// round trip (~0.4-0.6 us), so small values are pushed; the 16 KB histogram
// is cheaper to read in place than to push. (Plain and second-pass
// selections only.)
template <int KPT, int CL>
__global__ void __launch_bounds__(kThreads, 1) select_reg_kernel(SelectArgs a) {
  __shared__ RegShared sh;
  extern __shared__ int32_t bids[];  // token stage: the query's block ids
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // State that depends on no input is cleared while the previous kernel ends.
  for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
  sh.taken[tid] = 0u;
  if (tid == 0) sh.nbin = 0;
  griddep_wait();
  // The CTA's candidates: all of query b's (plain), chunk c of them (first
  // pass of a two-pass selection), or the ids the first pass kept (second);
  // with CL > 1, the rank's share of them.
  const uint32_t crank = CL > 1 ? cluster_ctarank() : 0u;
  const int b = CL > 1 ? static_cast<int>(blockIdx.x / CL)
                       : (a.chunks ? static_cast<int>(blockIdx.x / a.chunks)
                                   : static_cast<int>(blockIdx.x));
  constexpr int kPerCta = KPT * kThreads;
  const int cbase = static_cast<int>(crank) * kPerCta;  // first candidate of this CTA
  const int64_t base =
      CL > 1 ? cbase : (a.chunks ? static_cast<int64_t>(blockIdx.x % a.chunks) * a.chunk : 0);
  // at most KPT x 1024 candidates: 32-bit indices from here on
  const int n_all =
      static_cast<int>(a.in_ids ? a.n_in : (a.chunks ? min(a.chunk, a.n - base) : a.n));
  const int n = CL > 1 ? max(0, min(n_all - cbase, kPerCta)) : n_all;
  const uint32_t k = static_cast<uint32_t>(a.k);
  const float* sc = a.scores + static_cast<int64_t>(b) * a.n;
  const int32_t* ids_in =
      a.in_ids ? a.in_ids + static_cast<int64_t>(b) * a.n_in + (CL > 1 ? cbase : 0) : nullptr;
  const bool dense = CL == 1 && a.dense_stride && a.block_ids;

  // The block ids (token stage) are requested first, so their latency
  // overlaps the score loads; they go to shared memory further down.
  constexpr int kBidRegs = kMaxKBlocks / kThreads;
  static_assert(kMaxKBlocks % kThreads == 0, "block ids: whole registers a thread");
  const int32_t* bl = a.block_ids ? a.block_ids + static_cast<int64_t>(b) * a.k_blocks : nullptr;
  int32_t bid_r[kBidRegs];
  if (bl) {
#pragma unroll
    for (int u = 0; u < kBidRegs; ++u) {
      const int i = tid + u * kThreads;
      bid_r[u] = i < a.k_blocks ? __ldg(bl + i) : -1;
    }
  }
  uint32_t key[KPT];
  const int wbase = warp * (32 * KPT) + lane;  // + 32 j
  // Scores that do not go through the block ids are requested first, so their
  // latency overlaps the block-id copy below.
  if (ids_in) {
    // Second pass: the kept ids ascend along the list (chunks in order, each
    // ascending, -1 padded), so list order is id order for the tie rule.
    // (The key registers hold the ids first: no second array.)
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int i = wbase + 32 * j;
      key[j] = static_cast<uint32_t>(i < n ? ids_in[i] : -1);
    }
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int32_t id = static_cast<int32_t>(key[j]);
      key[j] = score_key(id >= 0 ? sc[id] : -INFINITY);
    }
  } else if (!dense) {
    // all KPT loads go out before any is used (indices clamped into the row)
    float v[KPT];
    const float* sb = sc + (n > 0 ? base : 0);  // (a cluster rank may hold no candidate)
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int i = wbase + 32 * j;
      v[j] = __ldg(sb + (i < n ? i : 0));
    }
#pragma unroll
    for (int j = 0; j < KPT; ++j) key[j] = score_key(wbase + 32 * j < n ? v[j] : -INFINITY);
  }
  // kept blocks' scores in candidate order, after the block ids (16-byte aligned)
  float* cand_s = reinterpret_cast<float*>(bids + kMaxKBlocks);
  const int n_row_blocks = dense ? static_cast<int>(a.dense_stride / 8) : 0;
  if (dense) {
    const float* row = a.scores + static_cast<int64_t>(b) * a.dense_stride;
#pragma unroll
    for (int u = 0; u < kBidRegs; ++u) {
      const int kb = tid + u * kThreads;
      if (kb < a.k_blocks && bid_r[u] >= 0 && bid_r[u] < n_row_blocks) {
        const float* src = row + static_cast<int64_t>(bid_r[u]) * 8;
        const uint32_t dst = smem_u32(cand_s + kb * 8);
        cp_async_16(dst, src);
        cp_async_16(dst + 16, src + 4);
      }
    }
    cp_async_commit();
  }
  if (bl) {
    // to shared memory; their order is checked after the next barrier
#pragma unroll
    for (int u = 0; u < kBidRegs; ++u) {
      const int i = tid + u * kThreads;
      if (i < a.k_blocks) bids[i] = bid_r[u];
    }
  }
  if (dense) {
    cp_async_wait<0>();
    __syncthreads();  // every thread's copies and block ids are visible
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int i = wbase + 32 * j;
      const int blk = i < n ? bids[i >> 3] : -1;
      key[j] = score_key(blk >= 0 && blk < n_row_blocks ? cand_s[i] : -INFINITY);
    }
  }
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u, cnt = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    if (key[j] > kInvalidKey) {
      kmin = min(kmin, key[j]);
      kmax = max(kmax, key[j]);
      ++cnt;
    }
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (lane == 0) {
    const uint4 v = make_uint4(kmin, kmax, cnt, 0u);
    sh.stat[crank][warp] = v;
#pragma unroll
    for (uint32_t p = 1; p < CL; ++p) {
      st_cluster_u4(mapa_shared(smem_u32(&sh.stat[crank][warp]), (crank + p) % CL), v);
    }
  }
  if constexpr (CL > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (a.block_ids) {
    // Ascending block ids with -1 padding at the end are required: the tie
    // rule and the ascending output rely on it.
    for (int i = static_cast<int>(crank) * kThreads + tid; i + 1 < a.k_blocks;
         i += CL * kThreads) {
      const int x = bids[i], y = bids[i + 1];
      if (y >= 0 && (x < 0 || y <= x)) {
        record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_SELECT, static_cast<uint32_t>(i));
      }
    }
  }
  // every warp reduces the 32 warps' values (of every CTA of the cluster) itself
  uint32_t smin = 0xFFFFFFFFu, smax = 0u, scnt = 0u;
#pragma unroll
  for (int r = 0; r < CL; ++r) {
    const uint4 v = sh.stat[r][lane];
    smin = min(smin, v.x);
    smax = max(smax, v.y);
    scnt += v.z;
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, smin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, smax);
  const uint32_t n_valid = __reduce_add_sync(0xFFFFFFFFu, scnt);
  const bool take_all = n_valid <= k;
  const uint32_t span = kmax - kmin;
  uint32_t P = 0, s_cur = 32, need = k;
  bool ties = false;
  // A thread's four histogram words: digits 4092 - 4 tid .. 4095 - 4 tid
  const uint32_t hoff = static_cast<uint32_t>(kBins - 4 - 4 * tid) * 4u;
  // The histograms are complete: a barrier (CL = 1) or a cluster barrier.
  auto hist_done = [&]() {
    if constexpr (CL > 1) {
      cluster_sync();
    } else {
      __syncthreads();
    }
  };
  // Threshold search over a histogram in sh.hist: the bin holding the
  // nd-th largest key, counted from the top bin down. hist_done has run
  // after the histogram was filled; this ends with a barrier after which
  // sh.bstar / sh.need / sh.count hold the bin, the count still needed in it
  // and its size. (sh.warp_a is rewritten: its readers are behind a barrier.)
  // With CL > 1 the histogram is the sum of the cluster's CTAs' ones (read in
  // place), and sh.bin_src[r] is the bin's count in CTA r's.
  auto find_threshold = [&](uint32_t nd) {
    uint4 hr[CL];  // [p]: the words of CTA (crank + p) % CL
    hr[0] = ld_shared_v4(smem_u32(sh.hist) + hoff);
#pragma unroll
    for (uint32_t p = 1; p < CL; ++p) {
      hr[p] = ld_cluster_v4(mapa_shared(smem_u32(sh.hist) + hoff, (crank + p) % CL));
    }
    uint4 hv = hr[0];
#pragma unroll
    for (int p = 1; p < CL; ++p) {
      hv.x += hr[p].x;
      hv.y += hr[p].y;
      hv.z += hr[p].z;
      hv.w += hr[p].w;
    }
    // h[j] = digit 4095 - 4 tid - j
    uint32_t h[4] = {hv.w, hv.z, hv.y, hv.x};
    const uint32_t local = h[0] + h[1] + h[2] + h[3];
    const uint32_t incl = warp_incl_scan(local);
    if (lane == 31) sh.warp_a[warp] = incl;
    __syncthreads();
    uint32_t total;
    uint32_t run = incl - local + warps_before(sh.warp_a[lane], warp, &total);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (run < nd && run + h[j] >= nd) {
        sh.bstar = static_cast<uint32_t>(kBins - 1 - (4 * tid + j));
        sh.need = nd - run;
        sh.count = h[j];
        if constexpr (CL > 1) {
#pragma unroll
          for (uint32_t p = 0; p < CL; ++p) {
            const uint4 v = hr[p];
            sh.bin_src[(crank + p) % CL] = j == 0 ? v.w : (j == 1 ? v.z : (j == 2 ? v.y : v.x));
          }
        }
      }
      run += h[j];
    }
    __syncthreads();
  };
  // Value-space level: bin = floor((v - vmin) * 4096 / (vmax - vmin)) is
  // non-decreasing in v, so every key in a higher bin is strictly larger than
  // every key in a lower one and equal keys share a bin; for smooth score
  // distributions the threshold bin holds a handful of keys, which are then
  // ranked exactly. Otherwise the radix levels below run from the start.
  // Each candidate's bin is kept, two 16-bit bins per register.
  bool vspace = false;
  uint32_t vbin = 0;
  uint32_t binp[(KPT + 1) / 2];
#pragma unroll
  for (int j = 0; j < (KPT + 1) / 2; ++j) binp[j] = 0;
  if (!take_all) {
    const float vmin = key_value(kmin);
    const float vspan = key_value(kmax) - vmin;
    const float vscale = static_cast<float>(kBins) / vspan;
    if (vspan > 0.f && isfinite(vspan) && isfinite(vscale)) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        if (key[j] > kInvalidKey) {
          const uint32_t bj = value_bin(key_value(key[j]), vmin, vscale);
          binp[j >> 1] |= bj << (16 * (j & 1));
          atomicAdd(&sh.hist[bj], 1u);
        }
      }
      hist_done();
      find_threshold(need);
      if (sh.count <= kRankMax) {
        vspace = true;
        vbin = sh.bstar;
        need = sh.need;
      }
    }
  }
  auto bin_of = [&](int j) -> uint32_t { return (binp[j >> 1] >> (16 * (j & 1))) & 0xFFFFu; };
  if (!take_all && !vspace) {
    uint32_t s_next = span < kBins ? 0u : static_cast<uint32_t>(32 - __clz(span)) - 12u;
    for (int level = 0; level < 4; ++level) {
      const uint32_t hs = s_cur, s_lv = s_next;
      const uint32_t width = hs - s_lv;
      const uint32_t dmask = width >= 32 ? 0xFFFFFFFFu : (1u << width) - 1u;
      // (the cluster's CTAs have read this histogram's previous contents)
      if constexpr (CL > 1) cluster_sync();
      for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        if (key[j] > kInvalidKey) {
          const uint32_t t = key[j] - kmin;
          if (hs >= 32 || (t >> hs) == P) atomicAdd(&sh.hist[(t >> s_lv) & dmask], 1u);
        }
      }
      hist_done();
      find_threshold(need);
      P = (hs < 32 ? (P << width) : 0u) | sh.bstar;
      need = sh.need;
      s_cur = s_lv;
      const uint32_t c = sh.count;
      if (s_lv == 0) {
        ties = true;  // the bin holds one key value
        break;
      }
      if (c <= kRankMax) break;
      s_next = s_lv > 12 ? s_lv - 12 : 0;
      __syncthreads();
    }
  }
  // A member of the threshold bin into this CTA's list, and (CL > 1) into the
  // other CTAs' copies of it.
  auto list_member = [&](uint32_t key_j, uint32_t idx) {
    const uint32_t slot = atomicAdd(&sh.nbin, 1u);
    const uint2 m = make_uint2(key_j, idx);
    sh.bin[crank][slot] = m;
#pragma unroll
    for (uint32_t p = 1; p < CL; ++p) {
      st_cluster_u2(mapa_shared(smem_u32(&sh.bin[crank][slot]), (crank + p) % CL), m);
    }
  };
  // Classification against the threshold bin, as warp ballots over slot j:
  // gt_mask[j] = candidates strictly above the bin. The bin's members either
  // all tie (then the first `need` of them in index order are taken, and
  // sh.taken holds their ballots) or are collected here, ranked below and
  // their taken ones marked in sh.taken. Candidate wbase + 32 j is bit `lane`
  // of word warp * KPT + j, so a warp reads its slot-j word of sh.taken at once.
  uint32_t gt_mask[KPT];
  uint32_t e_w = 0;  // tied bin members in this warp
  const bool collect = !take_all && !ties;
  if (take_all) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) gt_mask[j] = __ballot_sync(0xFFFFFFFFu, key[j] > kInvalidKey);
  } else if (vspace) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const bool valid = key[j] > kInvalidKey;
      const uint32_t bj = bin_of(j);
      gt_mask[j] = __ballot_sync(0xFFFFFFFFu, valid && bj > vbin);
      if (valid && bj == vbin) {  // a value-space bin is always ranked (never ties)
        list_member(key[j], static_cast<uint32_t>(cbase + wbase + 32 * j));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const bool valid = key[j] > kInvalidKey;
      const uint32_t hi = (key[j] - kmin) >> s_cur;
      const bool inb = valid && hi == P;
      gt_mask[j] = __ballot_sync(0xFFFFFFFFu, valid && hi > P);
      if (ties) {
        const uint32_t e = __ballot_sync(0xFFFFFFFFu, inb);
        if (lane == 0) sh.taken[warp * KPT + j] = e;
        e_w += __popc(e);
      } else if (inb) {
        list_member(key[j], static_cast<uint32_t>(cbase + wbase + 32 * j));
      }
    }
    if (ties) __syncwarp();  // lane 0's words, read by the whole warp below
  }
  // a candidate index of this CTA's share: its bit in sh.taken
  auto mark_taken = [&](uint32_t ie) {
    const uint32_t li = ie - static_cast<uint32_t>(cbase);
    if (li < static_cast<uint32_t>(kPerCta)) atomicOr(&sh.taken[li >> 5], 1u << (li & 31));
  };
  if (collect) {
    // Members listed by each CTA: this one's own count, or (CL > 1) CTA r's
    // count in the final level's threshold bin.
    uint32_t cs[CL];
    if constexpr (CL > 1) {
#pragma unroll
      for (int r = 0; r < CL; ++r) cs[r] = sh.bin_src[r];
      cluster_sync();  // every CTA's members are in every list
    } else {
      __syncthreads();
      cs[0] = sh.nbin;
    }
    uint32_t c = 0;
#pragma unroll
    for (int r = 0; r < CL; ++r) c += cs[r];
    // member m of the lists taken in CTA order
    auto member = [&](uint32_t m) -> uint2 {
      int r = 0;
#pragma unroll
      for (int q = 0; q + 1 < CL; ++q) {
        if (r == q && m >= cs[q]) {
          m -= cs[q];
          r = q + 1;
        }
      }
      return sh.bin[r][m];
    };
    if (need >= c) {
      // every member is taken
      if (static_cast<uint32_t>(tid) < c) mark_taken(member(tid).y);
    } else {
      const uint32_t mi = static_cast<uint32_t>(tid >> 4), part = static_cast<uint32_t>(tid & 15);
      uint32_t rank = 0, ke = 0, ie = 0;
      if (mi < c) {
        const uint2 me = member(mi);
        ke = me.x;
        ie = me.y;
        for (uint32_t o = part; o < c; o += 16) {
          const uint2 mo = member(o);
          rank += (mo.x > ke || (mo.x == ke && mo.y < ie)) ? 1u : 0u;
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
      if (part == 0 && mi < c && rank < need) mark_taken(ie);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < KPT; ++j) gt_mask[j] |= sh.taken[warp * KPT + j];
  }
  uint32_t g_w = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) g_w += __popc(gt_mask[j]);
  // Warp totals -> (every warp scans them itself, in warp order = index
  // order) this warp's output offset and its share of the ties taken at the
  // threshold.
  if (lane == 0) {
    const uint2 v = make_uint2(g_w, e_w);
    sh.tot[crank][warp] = v;
#pragma unroll
    for (uint32_t p = 1; p < CL; ++p) {
      st_cluster_u2(mapa_shared(smem_u32(&sh.tot[crank][warp]), (crank + p) % CL), v);
    }
  }
  // (CL > 1: the last exchange; no CTA touches another's shared memory after it)
  if constexpr (CL > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  uint32_t total, te_w;
  uint32_t pos;
  {
    const uint32_t take_eq_total = ties ? need : 0u;
    const uint2 own = sh.tot[crank][lane];
    const uint32_t e = own.y, g = own.x;
    // CL > 1: the CTAs of lower rank hold the lower candidate indices, so
    // their ties come first and their output goes first.
    uint32_t e_cta = 0, s_cta = 0, s_all = 0;  // ties and output before this CTA; all output
    if constexpr (CL > 1) {
      uint32_t e_acc = 0;
#pragma unroll
      for (uint32_t r = 0; r < CL; ++r) {
        const uint2 v = sh.tot[r][lane];
        const uint32_t e_r = __reduce_add_sync(0xFFFFFFFFu, v.y);
        const uint32_t g_r = __reduce_add_sync(0xFFFFFFFFu, v.x);
        const uint32_t te_r = take_eq_total > e_acc ? min(e_r, take_eq_total - e_acc) : 0u;
        if (r < crank) {
          e_cta += e_r;
          s_cta += g_r + te_r;
        }
        s_all += g_r + te_r;
        e_acc += e_r;
      }
    }
    // ties in the warps before warp `lane`
    const uint32_t e_before = e_cta + warp_incl_scan(e) - e;
    const uint32_t te = take_eq_total > e_before ? min(e, take_eq_total - e_before) : 0u;
    const uint32_t sel = g + te;
    pos = s_cta + warps_before(sel, warp, &total);  // output offset of this warp
    if constexpr (CL > 1) total = s_all;
    te_w = __shfl_sync(0xFFFFFFFFu, te, warp);  // ties this warp takes
  }
  // First pass: row b * chunks + c of the scratch, i.e. row blockIdx.x.
  int32_t* out = a.out_ids + static_cast<int64_t>(CL > 1 ? b : static_cast<int>(blockIdx.x)) * a.k;
  const uint32_t lt = (1u << lane) - 1u;
  auto out_id = [&](int j) -> int32_t {
    const int i = wbase + 32 * j;
    if (ids_in) return ids_in[i];
    const int gi = cbase + i;  // the candidate's index within the query
    return a.block_ids ? bids[gi >> 3] * 8 + static_cast<int32_t>(gi & 7)
                       : static_cast<int32_t>(base + i);
  };
  if (!ties) {
    // one loop per id source (the source is the same for every slot): slot
    // j's lanes with their bit set write at ow + (set bits below them)
    int32_t* ow = out + pos;
    if (ids_in) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const uint32_t m = gt_mask[j];
        if ((m >> lane) & 1u) ow[__popc(m & lt)] = ids_in[wbase + 32 * j];
        ow += __popc(m);
      }
    } else if (a.block_ids) {
      // candidate cbase + wbase + 32 j is token (lane & 7) of kept block
      // ((cbase + wbase) >> 3) + 4 j
      const int32_t* bw = bids + ((cbase + wbase) >> 3);
      const int32_t r = lane & 7;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const uint32_t m = gt_mask[j];
        if ((m >> lane) & 1u) ow[__popc(m & lt)] = bw[4 * j] * 8 + r;
        ow += __popc(m);
      }
    } else {
      const int32_t id0 = static_cast<int32_t>(base) + wbase;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const uint32_t m = gt_mask[j];
        if ((m >> lane) & 1u) ow[__popc(m & lt)] = id0 + 32 * j;
        ow += __popc(m);
      }
    }
  } else {
    uint32_t eq_seen = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t eqm = sh.taken[warp * KPT + j];  // the tied members of slot j
      // ties taken in this run: the first (te_w - eq_seen) tied lanes, if any left
      const uint32_t left = te_w > eq_seen ? te_w - eq_seen : 0u;
      const uint32_t eq_rank = __popc(eqm & lt);
      const bool is_gt = (gt_mask[j] >> lane) & 1u;
      const bool is_eq = ((eqm >> lane) & 1u) && eq_rank < left;
      if (is_gt || is_eq) out[pos + __popc(gt_mask[j] & lt) + min(eq_rank, left)] = out_id(j);
      const uint32_t taken_eq = min(static_cast<uint32_t>(__popc(eqm)), left);
      pos += __popc(gt_mask[j]) + taken_eq;
      eq_seen += __popc(eqm);
    }
  }
  for (int j = static_cast<int>(total) + static_cast<int>(crank) * kThreads + tid; j < a.k;
       j += CL * kThreads) {
    out[j] = -1;
  }
}

}  // namespace

// Dynamic shared memory of a selection CTA: the block ids, then (dense rows,
// CL = 1 only) the kept blocks' scores.
constexpr size_t reg_smem_max(int cl) {
  return static_cast<size_t>(kMaxKBlocks) * 4 + (cl > 1 ? 0 : static_cast<size_t>(kMaxKBlocks) * 8 * 4);
}

template <int KPT, int CL>
cudaError_t launch_reg(const SelectArgs& a, unsigned grid, cudaStream_t s) {
  size_t smem = a.block_ids ? static_cast<size_t>(a.k_blocks) * 4 : 0;
  if (CL == 1 && a.block_ids && a.dense_stride) {
    smem = static_cast<size_t>(kMaxKBlocks) * 4 + static_cast<size_t>(a.k_blocks) * 8 * 4;
  }
  static std::atomic<int> smem_set[64]{};
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(select_reg_kernel<KPT, CL>),
                              static_cast<int>(reg_smem_max(CL)), smem_set);
  if (e != cudaSuccess) return e;
  if constexpr (CL == 1) {
    return launch_pdl(select_reg_kernel<KPT, 1>, dim3(grid), dim3(kThreads), smem, s, 1, a);
  } else {
    // clusters of CL consecutive CTAs along x, with programmatic dependent launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid * CL);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, select_reg_kernel<KPT, CL>, a);
  }
}

// Register-resident selection of m <= 32 * kThreads candidates per CTA, one
// CTA (cl = 1) or a cluster of cl CTAs (2 or 4) per query.
cudaError_t launch_reg_for(const SelectArgs& a, int64_t m, unsigned grid, cudaStream_t s,
                           int cl = 1) {
  if (cl == 2 || cl == 4) {
    const int64_t per = (m + cl - 1) / cl;
    if (per <= 2 * kThreads) return cl == 2 ? launch_reg<2, 2>(a, grid, s) : launch_reg<2, 4>(a, grid, s);
    if (per <= 4 * kThreads) return cl == 2 ? launch_reg<4, 2>(a, grid, s) : launch_reg<4, 4>(a, grid, s);
    if (per <= 8 * kThreads) return cl == 2 ? launch_reg<8, 2>(a, grid, s) : launch_reg<8, 4>(a, grid, s);
    if (per <= 16 * kThreads && cl == 2) return launch_reg<16, 2>(a, grid, s);
    return cudaErrorInvalidValue;  // (m <= 32 * kThreads: not reached)
  }
  if (m <= 2 * kThreads) return launch_reg<2, 1>(a, grid, s);
  if (m <= 4 * kThreads) return launch_reg<4, 1>(a, grid, s);
  // (a prefill chunk's block stage: a few blocks over 4096)
  if (m <= 5 * kThreads) return launch_reg<5, 1>(a, grid, s);
  if (m <= 6 * kThreads) return launch_reg<6, 1>(a, grid, s);
  if (m <= 8 * kThreads) return launch_reg<8, 1>(a, grid, s);
  if (m <= 16 * kThreads) return launch_reg<16, 1>(a, grid, s);
  return launch_reg<32, 1>(a, grid, s);
}

// CTAs per query of a register-resident selection: a query's candidates are
// split over a cluster of 2 or 4 CTAs while the clusters of all B queries
// still fit on the SMs at once and each CTA keeps at least 2048 candidates
// (the per-candidate work, which bounds the kernel, then shrinks with the
// split; the cluster exchanges cost a few barriers). Not for first passes
// (chunks) or dense score rows.
// Clusters of `cl` selection CTAs (each a whole SM) that can be resident at once.
int select_max_clusters(int cl) {
  static std::atomic<int> cache[64][2]{};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int k = cl == 2 ? 0 : 1;
  int n = cache[dev][k].load(std::memory_order_relaxed);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = reg_smem_max(cl);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cl);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const void* kern = cl == 2 ? reinterpret_cast<const void*>(select_reg_kernel<8, 2>)
                             : reinterpret_cast<const void*>(select_reg_kernel<4, 4>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(reg_smem_max(cl)));
  if (e == cudaSuccess) {
    e = cl == 2 ? cudaOccupancyMaxActiveClusters(&n, select_reg_kernel<8, 2>, &cfg)
                : cudaOccupancyMaxActiveClusters(&n, select_reg_kernel<4, 4>, &cfg);
  }
  if (e != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the error the failed query left behind
    n = device_sm_count() / cl / 2;
  }
  cache[dev][k].store(n, std::memory_order_relaxed);
  return n;
}

int select_cluster(const SelectArgs& a, int64_t m) {
  if (a.chunks || a.dense_stride) return 1;
  int cl = 1;
  while (cl < 4 && m >= int64_t{2048} * cl * 2 && a.B <= select_max_clusters(cl * 2)) cl *= 2;
  return cl;
}

constexpr int64_t kRegMax = 32 * kThreads;  // candidates a register-resident CTA holds
constexpr int kMaxChunks = 64;

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s, int* launches) {
  if (launches) *launches = 0;
  if (a.B == 0) return cudaSuccess;
  if (launches) *launches = 1;
  if (a.n <= kRegMax) return launch_reg_for(a, a.n, a.B, s, select_cluster(a, a.n));
  if (a.dense_stride) return cudaErrorInvalidValue;  // dense rows: register-resident kernel only
  // Two passes over C chunks: every query's best k lies within the best k of
  // its own chunk (same order, same ids), so the second pass over the C * k
  // kept ids finds exactly the plain selection.
  if (a.tmp && !a.block_ids && a.k > 0) {
    // Enough chunks for each to fit a CTA, and for the B x C first-pass CTAs
    // to fill the SMs (a cluster of CTAs takes the second pass's C x k ids),
    // but at least as many as keep a one-CTA second pass at 16 candidates a
    // thread (the 32-a-thread kernel spills).
    const int64_t c_fit = (a.n + kRegMax - 1) / kRegMax;
    const int64_t c_sms = std::max<int64_t>(1, device_sm_count() / std::max(1, a.B));
    const int64_t c_pref = std::min<int64_t>(std::max<int64_t>(kRegMax / 2 / a.k, c_sms), kMaxChunks);
    const int64_t C = std::min<int64_t>(std::max(c_fit, c_pref), kRegMax / a.k);
    const int64_t chunk = (a.n + C - 1) / C;
    if (C >= 2 && chunk <= kRegMax && chunk > a.k) {
      SelectArgs p1 = a;
      p1.chunks = static_cast<int>(C);
      p1.chunk = chunk;
      p1.out_ids = a.tmp;
      cudaError_t e = launch_reg_for(p1, chunk, static_cast<unsigned>(a.B * C), s);
      if (e != cudaSuccess) return e;
      SelectArgs p2 = a;
      p2.in_ids = a.tmp;
      p2.n_in = C * a.k;
      if (launches) *launches = 2;
      return launch_reg_for(p2, p2.n_in, a.B, s, select_cluster(p2, p2.n_in));
    }
  }
  const int use_cache = a.n <= kCacheMax ? 1 : 0;
  const size_t smem = (use_cache ? static_cast<size_t>(a.n) * 4 : 0) +
                      (a.block_ids ? static_cast<size_t>(a.k_blocks) * 4 : 0);
  static std::atomic<int> smem_set[64]{};
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(select_kernel),
                              static_cast<int>(kCacheMax * 4 + kMaxKBlocks * 4), smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(a.B), dim3(kThreads), smem, s, 1, a, use_cache);
}

}  // namespace dsa
