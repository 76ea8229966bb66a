// Internal launch interface between the C-ABI entry points (api.cu) and the
// kernels of the two-tier sparse-attention step.
#pragma once

#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"

namespace dsa {

// Fixed dimensions the kernels are built for (miles.radixark.com
// "DeepSeek-V4.1 Flash", §1: 64 query heads, one 512-wide latent; the indexer
// of 16 heads x 128; blocks of 8 from recipes.vllm.ai "DeepSeek-V4.1-Flash",
// Overview, "Two-tier sparse attention").
constexpr int kHeads = 64;
constexpr int kLatent = 512;
constexpr int kIdxHeads = 16;
constexpr int kIdxDim = 128;
constexpr int kBlock = 8;
constexpr int kMaxKBlocks = 4096;
constexpr int kMaxKTokens = 512;
constexpr int kMaxWindow = 128;

// Paged addressing of one cache (dsa_pages_t with this cache's rows per page:
// page_rows for index keys and latents, page_rows / 8 for block keys); a null
// table means the cache is contiguous.
struct Paging {
  const int32_t* table;  // [B, per_seq]
  int rows;              // rows per page of this cache
  int per_seq;
  int64_t n_pages;
};
// Physical row of logical row r of sequence b, or -1 when the page entry is
// outside the pool (or r outside the table).
// (Logical rows are below 2^30, so the page arithmetic is 32-bit.)
__device__ __forceinline__ int64_t paged_row(const Paging& p, int b, int64_t r) {
  if (r < 0 || r >= (int64_t{1} << 30)) return -1;
  const int ri = static_cast<int>(r);
  const int pi = ri / p.rows;
  if (pi >= p.per_seq) return -1;
  const int pg = p.table[static_cast<int64_t>(b) * p.per_seq + pi];
  if (pg < 0 || pg >= p.n_pages) return -1;
  return static_cast<int64_t>(pg) * p.rows + (ri - pi * p.rows);
}

// Position of query b of a prefill-mode call: ctx + b for a chunk of one
// sequence; in a multi-query decode batch (mq queries per sequence, sequence
// s holding n_tokens[s] tokens) the (b % mq)-th of sequence b / mq's last mq
// positions.
__device__ __forceinline__ int64_t query_pos(int64_t ctx, int mq, const int32_t* n_tokens,
                                             int b) {
  return mq > 0 ? int64_t{n_tokens[b / mq]} - mq + b % mq : ctx + b;
}
__device__ __forceinline__ int query_seq(int mq, int b) { return mq > 0 ? b / mq : 0; }

struct PoolArgs {
  int fmt;
  const void* key_data;
  const uint8_t* key_scales;
  int64_t key_stride;  // rows between sequences
  const int32_t* n_latents;
  int64_t max_latents;
  int B;
  int tail_only;
  void* out_data;
  uint8_t* out_scales;
  int64_t out_stride;
  Paging key_pages, out_pages;  // paged caches (table null: contiguous)
  int64_t key_rows, out_rows;   // rows of the key and block-key arrays (debug checks)
  DeviceStatus* status;
};
cudaError_t launch_pool(const PoolArgs& a, cudaStream_t s);

// Cache append at the compression step: for each sequence whose token count
// n completes a latent (n % ratio == 0), latent n / ratio - 1 becomes
// RN_bf16(sum_i softmax(gate)_i kv_i) over its ratio positions, and its index
// key row is copied in; n_lat_out[b] = n / ratio for the tail pooling after.
struct AppendArgs {
  int B;
  int ratio;                 // 1..32
  const int32_t* n_tokens;   // [B]
  const uint16_t* kv;        // bf16 [B, ratio, 512]
  const float* gate;         // [B, ratio]
  int fmt;
  const uint8_t* new_key;    // [B, row bytes] in the key format
  const uint8_t* new_scales; // [B, 4] (MX formats)
  uint16_t* latents;
  int64_t lat_stride;
  uint8_t* key_data;
  uint8_t* key_scales;
  int64_t key_stride;
  Paging pages;              // latents and keys paged by one table (table null: contiguous)
  int64_t max_latents;
  int32_t* n_lat_out;        // [B]
  DeviceStatus* status;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

// Indexer scores of key rows, one row per MMA lane:
//   score = sum_h w_h * max(0, q_idx_h . key)
// Row r of query b is
//   mode ROWS_BLOCKS:  pooled key r,            valid for r < ceil(n_latents[b]/8)
//   mode ROWS_LATENTS: index key r,             valid for r < n_latents[b]
//   mode ROWS_GATHER:  index key 8*ids[r/8]+r%8, valid when ids[r/8] >= 0 and
//                      the key is < n_latents[b]
// Invalid rows score -inf.
enum RowMode { ROWS_BLOCKS = 0, ROWS_LATENTS = 1, ROWS_GATHER = 2 };

struct ScanArgs {
  int fmt;
  const void* key_data;
  const uint8_t* key_scales;
  int64_t key_stride;  // rows between sequences
  const uint16_t* q_idx;  // bf16 [B, 16, 128]
  const float* w;         // [B, 16]
  const int32_t* n_latents;
  int64_t max_latents;
  int mode;
  const int32_t* block_ids;  // ROWS_GATHER: [B, k_blocks]
  int k_blocks;
  int64_t n_rows;  // rows per query (score row stride)
  float* scores;   // [B, n_rows]
  int B;
  // Prefill: query b sees n_latents = (ctx + b + 1) / ratio latents of one
  // shared key array (key_stride 0). Multi-query decode (mq > 0): prefill mode
  // over B / mq sequences of key_stride rows, query b at query_pos().
  int prefill;
  int64_t ctx;
  int ratio;
  int mq;
  const int32_t* n_tokens;
  // Paged cache (table null: contiguous, key_stride rows per sequence). Rows
  // are then read in groups of 8 (one TMA box each), like gathered blocks.
  Paging pages;
  int64_t key_rows;  // rows of the key array (set by launch_scan; debug checks)
  // Block stage of a decode step whose previous kernel is the tail pool
  // (which rewrites only each sequence's last block): the dependency wait is
  // taken by the producer just before the first tile that holds a sequence's
  // last block, so every other tile streams while the pool still runs.
  // Contiguous caches only.
  int defer_wait;
  DeviceStatus* status;
};
// In prefill ROWS_BLOCKS mode only complete blocks are scored; a query's
// partially visible last block is left at -inf for launch_prefill_partial.
cudaError_t launch_scan(const ScanArgs& a, int num_sms, cudaStream_t s);

// Prefill indexer scores of n_q queries (positions ctx .. ctx + n_q - 1) over
// one shared bf16 key array, sixteen queries per MMA. mode ROWS_BLOCKS: rows
// are complete pooled blocks, query q sees ((ctx + q + 1) / ratio) / 8 of
// them, and every column of its score row is written (-inf where unseen).
// mode ROWS_LATENTS: rows are latents, query q sees (ctx + q + 1) / ratio,
// and columns are written up to the end of the last block any query of its
// group of sixteen can see.
struct BatchedScanArgs {
  const uint16_t* key_data;  // bf16 [key_rows][128]
  int64_t key_rows;
  const uint16_t* q_idx;     // bf16 [n_q][16][128]
  const float* w;            // [n_q][16]
  int64_t n_q;
  int64_t ctx;
  int ratio;
  int mode;
  float* scores;             // [n_q][n_cols]
  int64_t n_cols;
  DeviceStatus* status;
};
cudaError_t launch_scan_batched(const BatchedScanArgs& a, int num_sms, cudaStream_t s);

// Prefill: for each query whose last visible block is incomplete, pool that
// block over its visible members (fp32 sum in order, / count, rounded to the
// key format), score it against the query's index heads and store the score
// at scores[b * n_rows + block].
struct PartialArgs {
  int fmt;
  const void* key_data;
  const uint8_t* key_scales;
  const uint16_t* q_idx;
  const float* w;
  int n_q;
  int64_t ctx;
  int ratio;
  int mq;                    // multi-query decode: queries per sequence (0: one sequence)
  const int32_t* n_tokens;   //   [n_q / mq] tokens per sequence
  int64_t key_stride;        //   key rows per sequence
  int64_t key_rows;          // rows of the key array (debug checks)
  float* scores;
  int64_t n_rows;
};
cudaError_t launch_prefill_partial(const PartialArgs& a, cudaStream_t s);

// Tensor map of a row-major 2-D array [rows][row_bytes] of elem_bytes-sized
// elements (inner extent `inner` elements), 128-byte swizzle, box
// {box_inner, box_rows}.
cudaError_t encode_tma_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_rows);

// Top-k by (score desc, index asc) among candidates with score > -inf; ids
// are written ascending, padded with -1.
struct SelectArgs {
  const float* scores;  // [B, n]
  int64_t n;
  int k;
  int B;
  const int32_t* block_ids;  // map candidate i -> 8*block_ids[i/8] + i%8 (may be null)
  int k_blocks;
  int32_t* out_ids;  // [B, k]
  DeviceStatus* status;
  // Scratch of B * 32768 ids (may be null) that lets a query with more than
  // 32768 candidates be selected in two passes: the best k of each of C
  // chunks of its candidates, then the best k of those C * k (C * k <= 32768).
  int32_t* tmp;
  // Set by launch_select for the two passes (zero for a plain selection):
  int chunks;              // pass 1: CTA b * chunks + c takes chunk c of query b
  int64_t chunk;           //         candidates [c * chunk, (c + 1) * chunk)
  const int32_t* in_ids;   // pass 2: candidate i of query b is id in_ids[b * n_in + i]
  int64_t n_in;
  // Non-zero (with block_ids): scores are dense rows over every token,
  // scores[b * dense_stride + t]; candidate i is token 8 * block_ids[i / 8] + i % 8.
  int64_t dense_stride;
};
// Returns the number of kernels launched in `launches` (1, or 2 for a
// two-pass selection).
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s, int* launches = nullptr);

struct AttnArgs {
  const uint16_t* q;        // bf16 [B, 64, 512]
  const uint16_t* latents;  // bf16, sequence stride lat_stride rows
  int64_t lat_stride;
  const int32_t* n_latents;  // [B] (ids are checked against it)
  const int32_t* token_ids;  // [B, k_tokens]
  int k_tokens;
  const uint16_t* swa;      // decode: [B, window, 512]; prefill: [n_q + window - 1, 512]
  const int32_t* swa_len;   // decode: [B]
  int window;
  int B;
  float scale_log2;  // tau * log2(e)
  uint16_t* out;     // bf16 [B, 64, 512]
  float* lse;        // [B, 64] or null
  // Prefill: query b is at position ctx + b, n_latents = (ctx + b + 1) / ratio,
  // window rows from the shared buffer. Multi-query decode (mq > 0): query b
  // at query_pos(), sequence b / mq's latents at lat_stride rows a sequence
  // and its window buffer at swa_seq_rows rows a sequence.
  int prefill;
  int64_t ctx;
  int ratio;
  int mq;
  const int32_t* n_tokens;
  int64_t swa_seq_rows;
  // Split-KV: with splits = S in {2, 4, 8} each query's window rows and
  // selected latents are each cut in S parts handled by the S CTAs of a
  // cluster (merged on chip); 1: one CTA per query.
  int splits;
  // KV rows per tile: 32 (four ring slots) or 64 (two ring slots; half the
  // QK^T instructions per row).
  int tile_rows;
  // Paged latent pool (table null: contiguous, lat_stride rows per sequence).
  Paging pages;
  int64_t lat_rows;  // rows of the latent array (debug checks)
  int64_t swa_rows;  // rows of the window buffer (set by launch_attn; debug checks)
  // fp8 KV cache (split kernel only): latents and window rows are E4M3 codes
  // (512 bytes a row; the pointers above are then byte arrays) standing for
  // code * kv_scale.
  int kv_fp8;
  float kv_scale;
  DeviceStatus* status;
};
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);
// Split-KV runs S CTAs per query, the largest S in {8, 4, 2} for which the
// queries' clusters fit the device at once (attn_max_clusters).
constexpr int kMaxAttnSplits = 8;
int attn_max_clusters(int splits);

// block_ids[b] = 0, 1, ..., ceil(n_latents[b] / 8) - 1, then -1.
cudaError_t launch_identity_blocks(const int32_t* n_latents, int B, int k_blocks,
                                   int32_t* block_ids, cudaStream_t s);

int device_sm_count();

// One CTA waits, bounded by limit_cycles, on a barrier that nothing arrives
// at, and records DSA_ERR_TIMEOUT (site SITE_SELFTEST) in `st`.
cudaError_t launch_timeout_selftest(DeviceStatus* st, long long limit_cycles, cudaStream_t s);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device): `cache` is the caller's per-kernel array.
// Host threads may race here; the attribute call is idempotent and the cache
// is atomic.
inline cudaError_t ensure_smem(const void* kernel, int bytes, std::atomic<int> (&cache)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev].load(std::memory_order_acquire) >= bytes) {
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev].store(bytes, std::memory_order_release);
  return e;
}

// Launches `kernel` on `s` with programmatic dependent launch allowed (the
// kernel starts while the previous one drains and waits for it with
// griddep_wait before touching global memory), optionally as clusters of
// (1, cluster_y, 1) CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int cluster_y, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = static_cast<unsigned>(cluster_y);
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace dsa
