// Internal launch interface between the C-ABI entry points (api.cu) and the
// kernels of the two-tier sparse-attention step.
#pragma once

#include <cuda_fp8.h>

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
  // Prefill: query b sees (ctx + b + 1) / ratio latents of one shared key
  // array (key_stride 0); only a partially visible last block is pooled, into
  // output row b. Queries whose last block is complete write nothing.
  int prefill;
  int64_t ctx;
  int ratio;
  DeviceStatus* status;
};
cudaError_t launch_pool(const PoolArgs& a, cudaStream_t s);

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
  // Prefill: query b sees n_latents = (ctx + b + 1) / ratio and, in
  // ROWS_BLOCKS mode, a partially visible last block is pooled on the fly.
  int prefill;
  int64_t ctx;
  int ratio;
  const void* partial_data;       // prefill ROWS_BLOCKS: pooled partial block of query b
  const uint8_t* partial_scales;  // at row b
  DeviceStatus* status;
};
cudaError_t launch_scan(const ScanArgs& a, int num_sms, cudaStream_t s);

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
};
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);

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
  // window rows from the shared buffer.
  int prefill;
  int64_t ctx;
  int ratio;
  DeviceStatus* status;
};
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);

// block_ids[b] = 0, 1, ..., ceil(n_latents[b] / 8) - 1, then -1.
cudaError_t launch_identity_blocks(const int32_t* n_latents, int B, int k_blocks,
                                   int32_t* block_ids, cudaStream_t s);

int device_sm_count();

}  // namespace dsa
