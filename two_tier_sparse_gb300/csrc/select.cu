// S2 / S4: keep the k best candidates of each query by (score desc, index asc)
// (the candidate stage's 2048 blocks and the indexer's best 512 latents,
// recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention";
// ties to the lower index, the rule this library fixes).
//
// One CTA per query. Scores map to order-preserving 32-bit keys; a 4-pass
// radix select (8 bits per pass, most significant first) finds the key T of
// the k-th best candidate and how many candidates equal to T still fit. A
// compaction pass then takes, in index order, every key > T and the first
// `remaining` keys == T, so the ids come out ascending and ties resolve to the
// lower index with no sort. Keys are cached in shared memory when they fit.
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kCacheMax = 49152;  // keys cached in shared memory (192 KB)

struct SelShared {
  uint32_t hist[256];
  uint32_t warp_sum[kWarps];
  uint32_t warp_a[kWarps];
  uint32_t warp_b[kWarps];
  uint32_t prefix, mask, remaining, n_valid, digit_found;
};

__device__ __forceinline__ uint32_t load_key(const float* sc, const uint32_t* cache, int64_t i) {
  return cache ? cache[i] : score_key(sc[i]);
}

// Inclusive scan of v over the warp.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads) select_kernel(SelectArgs a, int use_cache) {
  extern __shared__ uint32_t cache_mem[];
  __shared__ SelShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = a.n;
  const float* sc = a.scores + static_cast<int64_t>(b) * n;
  const uint32_t* cache = nullptr;
  if (use_cache) {
    for (int64_t i = tid; i < n; i += kThreads) cache_mem[i] = score_key(sc[i]);
    cache = cache_mem;
  }
  if (a.block_ids) {
    // The candidate list must be ascending block ids with -1 padding at the
    // end (as the block stage writes it): the lower-index tie rule and the
    // ascending output rely on it.
    const int32_t* bl = a.block_ids + static_cast<int64_t>(b) * a.k_blocks;
    for (int i = tid; i + 1 < a.k_blocks; i += kThreads) {
      const int x = bl[i], y = bl[i + 1];
      if ((y >= 0 && (x < 0 || y <= x))) {
        record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_SELECT, static_cast<uint32_t>(i));
      }
    }
  }
  if (tid == 0) {
    sh.prefix = 0;
    sh.mask = 0;
    sh.remaining = static_cast<uint32_t>(a.k);
    sh.digit_found = 0;
  }
  bool take_all = false;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh.prefix, mask = sh.mask, rem = sh.remaining;
    uint32_t valid_cnt = 0;
    for (int64_t base = 0; base < n; base += kThreads) {
      const int64_t i = base + tid;
      bool part = false;
      uint32_t digit = 0;
      if (i < n) {
        const uint32_t key = load_key(sc, cache, i);
        const bool valid = key > kInvalidKey;
        valid_cnt += valid ? 1u : 0u;
        part = valid && ((key & mask) == prefix);
        digit = (key >> shift) & 0xFFu;
      }
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, part);
      if (part) {
        const uint32_t peers = __match_any_sync(act, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], __popc(peers));
      }
    }
    if (pass == 0) {
      valid_cnt = __reduce_add_sync(0xFFFFFFFFu, valid_cnt);
      if (lane == 0) sh.warp_sum[warp] = valid_cnt;
      __syncthreads();
      if (tid == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kWarps; ++w) t += sh.warp_sum[w];
        sh.n_valid = t;
      }
    }
    __syncthreads();
    if (pass == 0 && sh.n_valid <= static_cast<uint32_t>(a.k)) {
      take_all = true;
      break;
    }
    // Suffix sums over digits, digit 255 first: thread t < 256 holds digit 255 - t.
    uint32_t v = 0, inc = 0;
    if (tid < 256) {
      v = sh.hist[255 - tid];
      inc = warp_incl_scan(v);
      if (lane == 31) sh.warp_a[warp] = inc;
    }
    __syncthreads();
    if (tid < 256) {
      for (int w = 0; w < warp; ++w) inc += sh.warp_a[w];
      // The k-th best lands in digit d when suffix(d) >= rem > suffix(d + 1).
      if (inc >= rem && inc - v < rem) {
        const uint32_t d = 255u - static_cast<uint32_t>(tid);
        sh.prefix = prefix | (d << shift);
        sh.mask = mask | (0xFFu << shift);
        sh.remaining = rem - (inc - v);
        sh.digit_found = static_cast<uint32_t>(pass + 1);
      }
    }
    __syncthreads();
    if (sh.digit_found != static_cast<uint32_t>(pass + 1)) {
      // Cannot happen when more than k keys are valid; keep the result defined.
      if (tid == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_SELECT, pass);
      take_all = true;
      break;
    }
  }

  // Threshold T and how many keys equal to T to take.
  const uint32_t T = take_all ? kInvalidKey : sh.prefix;
  const uint32_t take_eq_total = take_all ? 0u : sh.remaining;

  // Compaction in index order: each warp owns a contiguous segment.
  const int64_t seg = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int64_t s0 = static_cast<int64_t>(warp) * seg;
  const int64_t s1 = min(n, s0 + seg);
  uint32_t gt_cnt = 0, eq_cnt = 0;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t i = base + lane;
    const uint32_t key = (i < s1) ? load_key(sc, cache, i) : 0u;
    gt_cnt += __popc(__ballot_sync(0xFFFFFFFFu, (i < s1) && key > T));
    eq_cnt += __popc(__ballot_sync(0xFFFFFFFFu, (i < s1) && !take_all && key == T));
  }
  __syncthreads();
  if (lane == 0) {
    sh.warp_a[warp] = gt_cnt;
    sh.warp_b[warp] = eq_cnt;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t eq = sh.warp_b[lane], gt = sh.warp_a[lane];
    const uint32_t eq_incl = warp_incl_scan(eq);
    const uint32_t eq_before = eq_incl - eq;
    const uint32_t take_eq = take_eq_total > eq_before ? min(eq, take_eq_total - eq_before) : 0u;
    const uint32_t sel = gt + take_eq;
    const uint32_t sel_incl = warp_incl_scan(sel);
    sh.warp_a[lane] = sel_incl - sel;  // output offset of this warp
    sh.warp_b[lane] = take_eq;
    if (lane == 31) sh.n_valid = sel_incl;  // total selected
  }
  __syncthreads();
  int32_t* out = a.out_ids + static_cast<int64_t>(b) * a.k;
  uint32_t pos = sh.warp_a[warp];
  const uint32_t take_eq = sh.warp_b[warp];
  uint32_t eq_seen = 0;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t i = base + lane;
    const uint32_t key = (i < s1) ? load_key(sc, cache, i) : 0u;
    const bool gt = (i < s1) && key > T;
    const bool eq = (i < s1) && !take_all && key == T;
    const uint32_t eq_b = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eq_b & lt_mask) < take_eq);
    const uint32_t tb = __ballot_sync(0xFFFFFFFFu, take);
    if (take) {
      int32_t id = static_cast<int32_t>(i);
      if (a.block_ids) {
        const int blk = a.block_ids[static_cast<int64_t>(b) * a.k_blocks + (i >> 3)];
        id = blk * 8 + static_cast<int32_t>(i & 7);
      }
      out[pos + __popc(tb & lt_mask)] = id;
    }
    pos += __popc(tb);
    eq_seen += __popc(eq_b);
  }
  const uint32_t total = sh.n_valid;
  for (int64_t j = total + tid; j < a.k; j += kThreads) out[j] = -1;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  const int use_cache = a.n <= kCacheMax ? 1 : 0;
  const size_t smem = use_cache ? static_cast<size_t>(a.n) * 4 : 0;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kCacheMax * 4));
  if (e != cudaSuccess) return e;
  select_kernel<<<a.B, kThreads, smem, s>>>(a, use_cache);
  return cudaGetLastError();
}

}  // namespace dsa
