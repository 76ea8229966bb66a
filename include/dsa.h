/*
 * dsa.h - two-tier sparse attention on one GB300 (sm_103a): C ABI.
 *
 * The method is the two-tier sparse-attention step of DeepSeek-V4.1:
 *   - recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, bullet "Two-tier sparse
 *     attention": every layer attends over a 128-token sliding window; layers
 *     with a compression ratio (1 or 2) add compressed KV latents; an indexer
 *     side attention scores the latents and keeps the best 512 per query,
 *     pre-filtered by a candidate stage that keeps 2048 blocks of 8.
 *   - miles.radixark.com "DeepSeek-V4.1 Flash", §1 Model Introduction,
 *     "Architecture": one 512-wide latent per position is both key and value
 *     for all 64 query heads (no value projection); "Sparse retrieval": a
 *     top-512 candidate set per retrieving layer and a coarser candidate-block
 *     pass.
 * The pages leave the indexer open; this library fixes it as
 *     score(k) = sum_h w_h * ReLU(q_h . k)        (16 index heads x 128),
 * the block key as the mean of the block's 8 index keys, and ties in both
 * top-k stages to the lower index.
 *
 * Conventions shared by every call
 *   - Memory: every tensor pointer is DEVICE memory owned by the caller. The
 *     library allocates nothing and keeps no pointer after a call returns.
 *     Scratch lives in a caller-supplied workspace (see dsa_workspace_size);
 *     one workspace must not serve two calls that may run at the same time.
 *   - Streams: calls enqueue work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and return without synchronising, except
 *     dsa_read_device_status.
 *   - Threads: calls may come from several host threads at once, each with
 *     its own workspace; the library's host-side caches and launch counters
 *     are atomic. The profiling hook dsa_profile_events is the exception.
 *   - Layout: row-major, innermost dimension last. bf16 tensors are passed as
 *     raw 16-bit patterns. Every base pointer must be 16-byte aligned.
 *   - Dimensions: the kernels are built for 64 query heads, latent width 512,
 *     16 index heads of width 128, blocks of 8. Other values of those fields
 *     return DSA_ERR_UNSUPPORTED. k_blocks (1..4096), k_tokens (1..512),
 *     window (1..128), ratio (>= 1) and sm_scale are free.
 *   - Errors: every call returns a status and never aborts. Argument errors are
 *     found on the host before any launch. Conditions only the device can see
 *     (an n_latents entry above max_latents, a token id outside its sequence,
 *     block ids not ascending) are recorded in a status word inside the
 *     workspace, the offending element is skipped, and
 *     dsa_read_device_status reports DSA_ERR_DEVICE_CHECK.
 *   - Determinism: results are bit-identical from run to run (no floating-point
 *     atomics; every reduction has a fixed order).
 *   - Tracing: each call marks its phases as NVTX ranges (dsa.decode_step,
 *     dsa.decode_multi, dsa.prefill, dsa.compress_append, dsa.pool, dsa.block_stage,
 *     dsa.token_stage, dsa.attention) that a profiler shows on its timeline;
 *     with no tool attached a range costs two calls into empty stubs.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* dsa_stream_t; /* a cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, ... */
  DSA_ERR_MISALIGNED = 2,   /* a base pointer is not 16-byte aligned */
  DSA_ERR_UNSUPPORTED = 3,  /* dimensions the kernels are not built for */
  DSA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  DSA_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  DSA_ERR_DEVICE_CHECK = 6, /* a kernel flagged bad input (dsa_read_device_status) */
  DSA_ERR_TIMEOUT = 7       /* a bounded device wait ran out (dsa_read_device_status) */
} dsa_status_t;

/* Storage format of index keys and of block-pooled keys (recipes.vllm.ai
 * "DeepSeek-V4.1-Flash" names an MXFP8 and an MXFP4 indexer cache: the
 * "Mixed MXFP4/MXFP8 checkpoint" bullet and indexer_kv_dtype mxfp4 in its
 * serving configurations). */
typedef enum {
  DSA_FMT_BF16 = 0,  /* data: bf16 [rows, 128]; scales: NULL */
  DSA_FMT_MXFP8 = 1, /* data: e4m3 bytes [rows, 128]; scales: UE8M0 bytes [rows, 4]
                        (OCP MX v1.0: one power-of-two scale 2^(s-127) per 32 values) */
  DSA_FMT_MXFP4 = 2  /* data: e2m1 codes two a byte [rows, 64], element 2i in the low
                        nibble of byte i; scales: UE8M0 bytes [rows, 4] (OCP MX v1.0).
                        The kernels read these arrays in pairs of rows: seq_stride_rows
                        must be even, and a buffer whose last sequence's rows are odd in
                        number must hold one row more (it is read, never used). */
} dsa_fmt_t;

typedef struct {
  int n_heads;     /* query heads: 64 */
  int latent_dim;  /* latent width, key = value: 512 */
  int n_idx_heads; /* indexer heads: 16 */
  int idx_dim;     /* indexer width: 128 */
  int block;       /* latents per candidate block: 8 */
  int k_blocks;    /* blocks kept by the candidate stage: 2048 */
  int k_tokens;    /* latents kept per query: 512 */
  int window;      /* sliding-window rows: 128 */
  int ratio;       /* positions per compressed latent: 1 or 2 */
  float sm_scale;  /* softmax scale tau; <= 0 selects 1/sqrt(latent_dim) */
  int kv_fmt;      /* dsa_kv_fmt_t of the latents and window rows the attention reads */
  float kv_scale;  /* DSA_KV_FP8_E4M3: a row holds code * kv_scale; finite, > 0 */
} dsa_config_t;

/* Storage of the latent cache and of the window rows (key = value rows of
 * the attention). The serving pages run an fp8 KV cache (recipes.vllm.ai
 * "DeepSeek-V4.1-Flash", serving configurations, --kv-cache-dtype fp8) and
 * name no scale granularity; this library reads it as OCP E4M3 codes with one
 * scale for the whole cache. fp8 rows are taken by dsa_sparse_attn_decode, its
 * paged form and dsa_decode_step; the prefill, multi-query and append calls
 * return DSA_ERR_UNSUPPORTED for them. The attention converts each code to f16
 * exactly and takes the query to f16 with a power-of-two scale per head (exact
 * unless an element is below 2^-24 of its head's largest), so its MMAs run on
 * f16 operands; the probabilities are f16 too (bf16 with bf16 rows). */
typedef enum {
  DSA_KV_BF16 = 0,     /* bf16 rows of 512: 1024 bytes a row */
  DSA_KV_FP8_E4M3 = 1  /* E4M3 codes, 512 bytes a row, standing for code * kv_scale */
} dsa_kv_fmt_t;

/*
 * Paged layout of a decode batch's caches (a block table, as serving engines
 * keep KV caches in fixed-size pages; the candidate-block indexer reads its
 * keys through one, miles.radixark.com "DeepSeek-V4.1 Flash", §4.1). Each
 * cache is a pool of physical pages shared by the B sequences: logical row r
 * of sequence b lives in physical page
 *     page_table[b * pages_per_seq + r / R]   at row r % R of that page,
 * with R = page_rows for index keys and latents and R = page_rows / 8 for
 * block keys (a page of page_rows tokens holds page_rows / 8 blocks). So the
 * pools are laid out as [n_pages * R] rows of the cache's own row format
 * (latents: 512 bf16, or 512 E4M3 codes with an fp8 KV cache; keys: their dsa_fmt_t
 * row, MX scales [n_pages * R, 4]).
 *   page_table:    device int32 [B, pages_per_seq]; an entry outside
 *                  [0, n_pages) is a device-detected error (DSA_ERR_DEVICE_CHECK,
 *                  the rows of that page are skipped)
 *   page_rows:     tokens per page, a positive multiple of 64
 *   pages_per_seq: row stride of page_table, at least ceil(max_latents / page_rows)
 *   n_pages:       physical pages in each pool; n_pages * page_rows < 2^31
 */
typedef struct {
  const int32_t* page_table;
  int32_t page_rows;
  int32_t pages_per_seq;
  int64_t n_pages;
} dsa_pages_t;

/* A key cache (index keys or block-pooled keys) of B sequences. Contiguous
 * (pages == NULL): sequence b's row r is at data + (b * seq_stride_rows + r) *
 * row_bytes, and MX scales are laid out the same way with 4 bytes per row.
 * Paged (pages != NULL): rows are found through the page table above and
 * seq_stride_rows is not used. Paged caches are taken by dsa_pool_index_keys,
 * dsa_index_blocks, dsa_topk, dsa_topk_noalloc and dsa_decode_step (decode
 * only; prefill reads one contiguous sequence). */
typedef struct {
  dsa_fmt_t fmt;
  const void* data;
  const uint8_t* scales;
  int64_t seq_stride_rows;
  const dsa_pages_t* pages;
} dsa_keys_t;

/* The writable form, for dsa_pool_index_keys' output. */
typedef struct {
  dsa_fmt_t fmt;
  void* data;
  uint8_t* scales;
  int64_t seq_stride_rows;
  const dsa_pages_t* pages;
} dsa_keys_out_t;

/* Fills *cfg with the DeepSeek-V4.1 values above (ratio 1, sm_scale 0). */
void dsa_default_config(dsa_config_t* cfg);

/* Human-readable name of a status. Never NULL. */
const char* dsa_status_string(dsa_status_t s);

/*
 * Workspace bytes needed by any call below for up to `n_queries` queries
 * (decode: the batch B; prefill: n_q) whose sequences hold at most
 * `max_latents` latents each. Any larger workspace works too. The buffer must
 * be 256-byte aligned device memory, zeroed once before its first use (its
 * first 16 bytes hold the device status word), and is reused across calls.
 */
dsa_status_t dsa_workspace_size(const dsa_config_t* cfg, int n_queries, int64_t max_latents,
                                size_t* bytes);

/*
 * S0, block keys (the candidate stage's "blocks of 8", recipes.vllm.ai
 * "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention"; the block key is
 * the mean of the block's index keys, the rule this library fixes).
 * For each sequence b and each block j < ceil(n_latents[b] / 8) (or only the
 * block holding latent n_latents[b] - 1 when tail_only != 0):
 *     pooled[b][j] = RN_fmt( fp32_sum_in_order(keys[b][8j .. 8j+c-1]) / c ),
 * c = min(8, n_latents[b] - 8j). RN_fmt is round-to-nearest-even to bf16, or
 * the OCP MX conversion (X = floor(log2 amax) - emax per 32 values, emax 8
 * for e4m3 and 2 for e2m1, elements rounded to nearest even with saturation).
 * pooled->fmt must equal keys->fmt.
 *   n_latents: device int32 [B], each in [0, max_latents].
 */
dsa_status_t dsa_pool_index_keys(const dsa_config_t* cfg, const dsa_keys_t* keys,
                                 const int32_t* n_latents, int B, int64_t max_latents,
                                 int tail_only, const dsa_keys_out_t* pooled, void* workspace,
                                 size_t workspace_bytes, dsa_stream_t stream);

/*
 * S1 + S2, candidate-block stage: per query b, score every block j <
 * ceil(n_latents[b] / 8) with score = sum_h w_h ReLU(q_idx[b][h] . pooled[b][j])
 * and keep the k_blocks best by (score desc, j asc). When a query has at most
 * k_blocks blocks, all are kept.
 *   q_idx:        device bf16 [B, 16, 128]
 *   w:            device fp32 [B, 16]
 *   pooled:       block keys, as written by dsa_pool_index_keys
 *   n_latents:    device int32 [B]
 *   block_ids:    out, device int32 [B, k_blocks], ascending, -1 padded
 *   block_scores: out (optional, may be NULL), device fp32 [B, ceil(max_latents/8)];
 *                 entries past a query's block count are -inf
 */
dsa_status_t dsa_index_blocks(const dsa_config_t* cfg, const void* q_idx, const float* w,
                              const dsa_keys_t* pooled, const int32_t* n_latents, int B,
                              int64_t max_latents, int32_t* block_ids, float* block_scores,
                              void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * S3 + S4, token stage: per query b, score every visible latent t of the kept
 * blocks (t = 8 * block_ids[b][i] + r, r < 8, t < n_latents[b]) and keep the
 * k_tokens best by (score desc, t asc).
 *   block_ids:    device int32 [B, k_blocks], ascending with -1 padding at the
 *                 end (as dsa_index_blocks writes it), or NULL for "every block"
 *   token_ids:    out, device int32 [B, k_tokens], ascending, -1 padded
 *   token_scores: out (optional), device fp32 [B, n_cand]: the score of
 *                 candidate i (i.e. latent 8 * block_ids[b][i / 8] + i % 8), or of
 *                 latent i when block_ids is NULL; -inf where no latent exists.
 *                 n_cand = 8 * k_blocks, or max_latents rounded up to 8 when
 *                 block_ids is NULL.
 */
dsa_status_t dsa_topk(const dsa_config_t* cfg, const void* q_idx, const float* w,
                      const dsa_keys_t* keys, const int32_t* block_ids,
                      const int32_t* n_latents, int B, int64_t max_latents, int32_t* token_ids,
                      float* token_scores, void* workspace, size_t workspace_bytes,
                      dsa_stream_t stream);

/*
 * S5 - S7, attention (miles.radixark.com "DeepSeek-V4.1 Flash", §1: the latent
 * is key and value for all 64 heads). For query b the rows are
 *     KV = latents[b][token_ids[b][i]] for every id >= 0, then swa[b][0 .. swa_len[b]-1]
 * (selected latents and the sliding window, concatenated), and every head h
 *     z_j = tau * q[b][h] . KV_j,   out[b][h] = sum_j softmax(z)_j KV_j,
 *     lse[b][h] = log sum_j exp(z_j)   (natural log; -inf when there are no rows).
 *   q:        device bf16 [B, 64, 512]
 *   latents:  device bf16, sequence b's row r at (b * latent_seq_stride_rows + r) * 512
 *             (cfg->kv_fmt DSA_KV_FP8_E4M3: uint8 E4M3 codes, the same row layout)
 *   n_latents: device int32 [B]; an id >= n_latents[b] is flagged and skipped
 *   token_ids: device int32 [B, k_tokens], -1 entries are skipped
 *   swa:      device bf16 [B, window, 512]; slot s holds position T - swa_len[b] + s
 *             (DSA_KV_FP8_E4M3: uint8 E4M3 codes [B, window, 512])
 *   swa_len:  device int32 [B], each in [0, window]
 *   out:      out, device bf16 [B, 64, 512]
 *   lse:      out (optional), device fp32 [B, 64]
 */
dsa_status_t dsa_sparse_attn_decode(const dsa_config_t* cfg, const void* q, const void* latents,
                                    int64_t latent_seq_stride_rows, const int32_t* n_latents,
                                    const int32_t* token_ids, const void* swa,
                                    const int32_t* swa_len, int B, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    dsa_stream_t stream);

/*
 * dsa_sparse_attn_decode over a paged latent pool: latent id t of sequence b
 * is row page_table[b * pages_per_seq + t / page_rows] * page_rows + t % page_rows
 * of `latents` (bf16 [pages->n_pages * page_rows, 512], or E4M3 codes with an fp8 KV
 * cache). Ids whose page entry
 * is out of range are skipped and reported like ids past n_latents.
 */
dsa_status_t dsa_sparse_attn_decode_paged(const dsa_config_t* cfg, const void* q,
                                          const void* latents, const dsa_pages_t* pages,
                                          const int32_t* n_latents, const int32_t* token_ids,
                                          const void* swa, const int32_t* swa_len, int B,
                                          void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, dsa_stream_t stream);

/*
 * The whole decode step for B sequences, the query of sequence b at position
 * T_b - 1 with n_latents[b] = T_b / ratio visible latents: pool the newest
 * block (when update_pool != 0), the candidate-block stage (skipped when no
 * sequence can have more than k_blocks blocks), the token stage and the
 * attention, as the four calls above would in sequence.
 *   pooled:        block keys, read by the block stage; also written (newest
 *                  block only) when update_pool != 0
 *   keys, pooled:  both contiguous, or both paged with the same page table;
 *                  paged keys make the latents paged by that table too (and
 *                  latent_seq_stride_rows is then not used)
 *   block_ids:     out (optional), device int32 [B, k_blocks]
 *   token_ids:     out (optional), device int32 [B, k_tokens]
 */
dsa_status_t dsa_decode_step(const dsa_config_t* cfg, const void* q, const void* q_idx,
                             const float* w, const dsa_keys_t* keys, const dsa_keys_out_t* pooled,
                             int update_pool, const void* latents,
                             int64_t latent_seq_stride_rows, const int32_t* n_latents,
                             int64_t max_latents, const void* swa, const int32_t* swa_len, int B,
                             int32_t* block_ids, int32_t* token_ids, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * Prefill: n_q queries appended after ctx_len tokens of one sequence, query i
 * at position P = ctx_len + i. Each query has its own causal selection: it sees
 * floor((P + 1) / ratio) latents; a block that it sees only in part is pooled
 * over its visible members on the fly; its window is positions
 * max(0, P - window + 1) .. P.
 *   q:         device bf16 [n_q, 64, 512]
 *   q_idx:     device bf16 [n_q, 16, 128];  w: device fp32 [n_q, 16]
 *   latents:   device bf16 [n_lat, 512], n_lat = (ctx_len + n_q) / ratio
 *   keys:      index keys [n_lat, 128] (seq_stride_rows ignored)
 *   pooled:    block keys of the complete blocks [n_lat / 8, 128]
 *   swa:       device bf16 [n_q + window - 1, 512]; row r holds position
 *              ctx_len - window + 1 + r (rows before position 0 are never read)
 *   out:       out, device bf16 [n_q, 64, 512];  lse: out (optional) fp32 [n_q, 64]
 *   token_ids: out (optional), device int32 [n_q, k_tokens]
 */
dsa_status_t dsa_sparse_attn_prefill(const dsa_config_t* cfg, int n_q, int64_t ctx_len,
                                     const void* q, const void* q_idx, const float* w,
                                     const void* latents, const dsa_keys_t* keys,
                                     const dsa_keys_t* pooled, const void* swa, void* out,
                                     float* lse, int32_t* token_ids, void* workspace,
                                     size_t workspace_bytes, dsa_stream_t stream);

/*
 * Cache append at the compression step (recipes.vllm.ai "DeepSeek-V4.1-Flash",
 * Overview, "Two-tier sparse attention": layers with a compression ratio keep
 * latents "pooled by a learned softmax gate", one latent per ratio positions).
 * For each sequence b whose token count T_b = n_tokens[b] completes a latent
 * (T_b % ratio == 0), latent j = T_b / ratio - 1 becomes
 *     RN_bf16( sum_i softmax(gate[b])_i * kv[b][i] ),   i = 0 .. ratio - 1
 * (softmax over the group's ratio logits, in fp32), its index key row becomes
 * new_keys' row b, and the block key of the block holding j is re-pooled as
 * dsa_pool_index_keys(tail_only) does. Sequences that complete no latent are
 * left as they are. The gate's learned projection is not on the pages: its
 * logits are inputs.
 *   n_tokens:  device int32 [B]
 *   kv:        device bf16 [B, ratio, 512]: the group's per-position KV vectors
 *   gate:      device fp32 [B, ratio]
 *   new_keys:  the new index key of each sequence, one row per sequence (data
 *              [B, row], MX scales [B, 4]; seq_stride_rows not used)
 *   latents:   bf16, contiguous with latent_seq_stride_rows rows a sequence, or
 *              paged by keys->pages like the keys
 *   keys, pooled: the index-key and block-key caches (written)
 *   max_latents: the caches' capacity; a latent at or past it is a device check
 * ratio must be at most 32 (DSA_ERR_UNSUPPORTED otherwise). The workspace is
 * sized for B queries.
 */
dsa_status_t dsa_compress_append(const dsa_config_t* cfg, int B, const int32_t* n_tokens,
                                 const void* kv, const float* gate, const dsa_keys_t* new_keys,
                                 void* latents, int64_t latent_seq_stride_rows,
                                 const dsa_keys_out_t* keys, const dsa_keys_out_t* pooled,
                                 int64_t max_latents, void* workspace, size_t workspace_bytes,
                                 dsa_stream_t stream);

/*
 * Multi-query decode: n_q queries per sequence at its last n_q positions, as
 * when a block of draft tokens is verified in one pass (recipes.vllm.ai
 * "DeepSeek-V4.1-Flash", Overview, bullet "DSpark draft head"). Sequence b
 * holds T_b = n_tokens[b] tokens and its query i sits at position
 * P = T_b - n_q + i. Each query is causal with its own two-tier selection over
 * floor((P + 1) / ratio) latents (a block it sees in part is pooled over its
 * visible members on the fly, as in prefill) and its own window of positions
 * max(0, P - window + 1) .. P; the queries of a sequence read the same caches.
 *   n_tokens:    device int32 [B], each >= n_q (the queries of a shorter
 *                sequence that have no position get no rows, reported as
 *                DSA_ERR_DEVICE_CHECK)
 *   q:           device bf16 [B, n_q, 64, 512]; q_idx bf16 [B, n_q, 16, 128];
 *                w fp32 [B, n_q, 16]
 *   keys:        index keys of each sequence, contiguous (seq_stride_rows >=
 *                max_latents)
 *   pooled:      block keys of each sequence's complete blocks, as
 *                dsa_pool_index_keys writes them (seq_stride_rows >= max_latents / 8)
 *   latents:     bf16, sequence b's row r at (b * latent_seq_stride_rows + r) * 512
 *   max_latents: at least floor(n_tokens[b] / ratio) for every b
 *   swa:         device bf16 [B, window + n_q - 1, 512]; row r of sequence b
 *                holds position T_b - n_q - window + 1 + r (rows before
 *                position 0 are never read)
 *   out:         out, bf16 [B, n_q, 64, 512]; lse: out (optional) fp32 [B, n_q, 64]
 *   token_ids:   out (optional), int32 [B, n_q, k_tokens]
 * The workspace is sized for B * n_q queries (dsa_workspace_size).
 */
dsa_status_t dsa_decode_multi(const dsa_config_t* cfg, int n_q, const int32_t* n_tokens,
                              const void* q, const void* q_idx, const float* w,
                              const dsa_keys_t* keys, const dsa_keys_t* pooled,
                              const void* latents, int64_t latent_seq_stride_rows,
                              int64_t max_latents, const void* swa, int B, void* out, float* lse,
                              int32_t* token_ids, void* workspace, size_t workspace_bytes,
                              dsa_stream_t stream);

/*
 * dsa_topk without a workspace. The pages have no counterpart to this call; it
 * serves callers that cannot allocate device memory: a plugin that runs inside
 * a host framework which owns all device memory and lends it none, or a
 * serving loop under a fixed memory budget that forbids allocation once it has
 * started. It computes exactly what dsa_topk computes (same kernels, same
 * arguments, bit-identical token_ids) but keeps its candidate scores in a
 * scratch array that the library defines statically in device memory:
 * DSA_TOPK_NOALLOC_MAX_SCORES fp32 values (8 MiB), held on every GPU that
 * loads the library until the process exits. It calls no allocator.
 *   - Limit: B * n_cand <= DSA_TOPK_NOALLOC_MAX_SCORES, where n_cand is
 *     8 * k_blocks (block_ids given) or max_latents rounded up to 8 (block_ids
 *     NULL); larger requests return DSA_ERR_WORKSPACE before any launch.
 *   - Set-up: the first call on each device looks up that device's address of
 *     the scratch array (the calling thread's current device must be the one
 *     the stream belongs to); make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same scratch array, which keeps
 *     the last call's contents (every score the kernels read is written first
 *     by the same call, so nothing needs clearing). Calls that may overlap on
 *     the GPU (different streams without ordering) race on it: serialise them.
 *   - No status word: device-side input checks (ids outside a sequence,
 *     unordered block ids) skip the offending elements and report nothing,
 *     and a bounded device wait that runs out (DSA_ERR_TIMEOUT in the other
 *     calls) is not reported either. After such a timeout the scan leaves
 *     score slots unwritten, so the selection may rank scores left in the
 *     scratch by an earlier call while the call still returns DSA_OK. Use
 *     dsa_topk with a workspace where these conditions must be seen.
 */
#define DSA_TOPK_NOALLOC_MAX_SCORES (1 << 21)
dsa_status_t dsa_topk_noalloc(const dsa_config_t* cfg, const void* q_idx, const float* w,
                              const dsa_keys_t* keys, const int32_t* block_ids,
                              const int32_t* n_latents, int B, int64_t max_latents,
                              int32_t* token_ids, dsa_stream_t stream);

/* Kernel kinds, for the timing hook and the launch counters below. */
typedef enum {
  DSA_KERNEL_POOL = 0,    /* block-key pooling */
  DSA_KERNEL_SCAN = 1,    /* indexer scores (block stage and token stage) */
  DSA_KERNEL_SELECT = 2,  /* top-k selection */
  DSA_KERNEL_ATTN = 3,    /* attention */
  DSA_KERNEL_OTHER = 4,   /* small helpers (identity block lists) */
  DSA_KERNEL_KINDS = 5
} dsa_kernel_kind_t;

/*
 * Optional timing hook for profiling and benchmarks (no counterpart on the
 * pages). With n > 0, each later launch of kernel `kind` is bracketed on its
 * stream by cudaEventRecord(starts[i % n]) and cudaEventRecord(ends[i % n]),
 * where i counts that kind's launches since this call; n = 0 switches it off.
 * starts/ends hold caller-owned cudaEvent_t handles and must outlive their use.
 * The setting is process-wide and not thread-safe. Recording inside CUDA-graph
 * capture does not give timings; use it on plain stream launches.
 */
dsa_status_t dsa_profile_events(int kind, void* const* starts, void* const* ends, int n);

/*
 * Number of kernel launches per kind (counts[DSA_KERNEL_KINDS]) issued by this
 * process since it started or since the last call with reset != 0.
 */
dsa_status_t dsa_launch_counts(uint64_t* counts, int reset);

/*
 * Waits for `stream`, then reads and clears the status word in `workspace`:
 * DSA_OK, DSA_ERR_DEVICE_CHECK or DSA_ERR_TIMEOUT (the earliest recorded).
 * If info is not NULL it receives the recorded detail word (0 if none): bits
 * 24..31 name the kernel (1 block-key pooling, 2 indexer scan, 3 top-k
 * selection, 4 attention, 5 prefill partial block, 6 the self-test below),
 * bits 0..23 a detail (for
 * DSA_ERR_TIMEOUT the shared-memory address of the barrier waited on; for
 * DSA_ERR_DEVICE_CHECK the offending sequence index or id).
 */
dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, uint32_t* info);

/*
 * Self-test of the device failure report (no counterpart on the pages): a
 * kernel waits on a barrier that nothing arrives at, under the bounded-wait
 * scheme the step's kernels use but with a limit of about one millisecond,
 * gives up and records DSA_ERR_TIMEOUT in `workspace`'s status word. A
 * following dsa_read_device_status returns DSA_ERR_TIMEOUT with site 6; the
 * device stays usable. Returns DSA_ERR_INVALID_ARG without a workspace.
 */
dsa_status_t dsa_selftest_timeout(void* workspace, size_t workspace_bytes, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
