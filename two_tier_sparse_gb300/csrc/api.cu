// C-ABI entry points (declared in include/dsa.h): argument checks on the host,
// workspace layout, and the launch sequence of each call on the caller's stream.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <mutex>

#include "kernels.h"

namespace dsa {

namespace {

// NVTX range over a scope: the call's phases show by name in a profiler's
// timeline (Nsight Systems, ncu --nvtx); without a tool attached a push or pop
// is one call into an empty stub.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace regions for n queries over sequences of at most max_latents latents.
struct Layout {
  size_t status, block_scores, token_scores, block_ids, token_ids, select_tmp, total;
  int64_t nb_max, n_cand;
  bool has_select_tmp;
};

// Candidates per query above which the selection runs in two passes through
// a scratch of 32768 ids per query.
constexpr int64_t kSelectOnePass = 32768;

Layout layout(const dsa_config_t& c, int n, int64_t max_latents) {
  Layout L{};
  L.nb_max = (max_latents + kBlock - 1) / kBlock;
  const int64_t gathered = static_cast<int64_t>(c.k_blocks) * kBlock;
  const int64_t all = (max_latents + 7) / 8 * 8;
  L.n_cand = std::max(gathered, all);
  size_t off = 0;
  L.status = off;
  off = align_up(off + sizeof(DeviceStatus));
  L.block_scores = off;
  off = align_up(off + static_cast<size_t>(n) * L.nb_max * 4);
  L.token_scores = off;
  off = align_up(off + static_cast<size_t>(n) * L.n_cand * 4);
  L.block_ids = off;
  off = align_up(off + static_cast<size_t>(n) * c.k_blocks * 4);
  L.token_ids = off;
  off = align_up(off + static_cast<size_t>(n) * c.k_tokens * 4);
  L.select_tmp = off;
  L.has_select_tmp = std::max(L.nb_max, L.n_cand) > kSelectOnePass;
  if (L.has_select_tmp) off = align_up(off + static_cast<size_t>(n) * kSelectOnePass * 4);
  L.total = off;
  return L;
}

dsa_status_t check_config(const dsa_config_t* c) {
  if (c == nullptr) return DSA_ERR_INVALID_ARG;
  if (c->n_heads != kHeads || c->latent_dim != kLatent || c->n_idx_heads != kIdxHeads ||
      c->idx_dim != kIdxDim || c->block != kBlock) {
    return DSA_ERR_UNSUPPORTED;
  }
  if (c->k_blocks < 1 || c->k_blocks > kMaxKBlocks || c->k_tokens < 1 ||
      c->k_tokens > kMaxKTokens || c->window < 1 || c->window > kMaxWindow || c->ratio < 1 ||
      !(c->sm_scale == c->sm_scale) || isinf(c->sm_scale)) {
    return DSA_ERR_INVALID_ARG;
  }
  if (c->kv_fmt != DSA_KV_BF16 && c->kv_fmt != DSA_KV_FP8_E4M3) return DSA_ERR_INVALID_ARG;
  if (c->kv_fmt == DSA_KV_FP8_E4M3 && !(c->kv_scale > 0.f && !isinf(c->kv_scale))) {
    return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

float tau(const dsa_config_t& c) {
  return c.sm_scale > 0.f ? c.sm_scale : 1.0f / sqrtf(static_cast<float>(c.latent_dim));
}

// A page table covering sequences of up to max_latents latents.
dsa_status_t check_pages(const dsa_pages_t* pg, int64_t max_latents) {
  if (pg->page_table == nullptr || pg->page_rows <= 0 || pg->page_rows % 64 != 0 ||
      pg->n_pages < 1 || pg->pages_per_seq < 1) {
    return DSA_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(pg->page_table) & 3u) return DSA_ERR_MISALIGNED;
  if (static_cast<int64_t>(pg->pages_per_seq) * pg->page_rows < max_latents) {
    return DSA_ERR_INVALID_ARG;
  }
  if (pg->n_pages * pg->page_rows >= (int64_t(1) << 31)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// Paged addressing of a cache with `div` tokens per row (1: keys, latents;
// 8: block keys); a null table for a contiguous cache.
Paging paging_of(const dsa_pages_t* pg, int div) {
  Paging p{};
  if (pg != nullptr) {
    p.table = pg->page_table;
    p.rows = pg->page_rows / div;
    p.per_seq = pg->pages_per_seq;
    p.n_pages = pg->n_pages;
  }
  return p;
}

// Rows of a cache array of B sequences that hold at most `rows` rows each
// (contiguous: every sequence's stride but the last's own rows; paged: the
// pool), for the debug checks of the kernels.
int64_t cache_rows(const dsa_pages_t* pg, int div, int B, int64_t stride, int64_t rows) {
  if (pg != nullptr) return pg->n_pages * (pg->page_rows / div);
  return B > 0 ? (B - 1) * stride + rows : 0;
}

bool same_pages(const dsa_pages_t* a, const dsa_pages_t* b) {
  if (a == nullptr || b == nullptr) return a == b;
  return a->page_table == b->page_table && a->page_rows == b->page_rows &&
         a->pages_per_seq == b->pages_per_seq && a->n_pages == b->n_pages;
}

// Key cache checks. Contiguous: at least min_stride rows per sequence (when
// need_stride). Paged: a valid table for sequences of max_latents latents.
dsa_status_t check_keys(const dsa_keys_t* k, int64_t min_stride, bool need_stride,
                        int64_t max_latents = 0) {
  if (k == nullptr || k->data == nullptr) return DSA_ERR_INVALID_ARG;
  if (k->fmt != DSA_FMT_BF16 && k->fmt != DSA_FMT_MXFP8 && k->fmt != DSA_FMT_MXFP4) {
    return DSA_ERR_INVALID_ARG;
  }
  const bool mx = k->fmt != DSA_FMT_BF16;
  if (mx && k->scales == nullptr) return DSA_ERR_INVALID_ARG;
  if (!aligned16(k->data)) return DSA_ERR_MISALIGNED;
  if (mx && (reinterpret_cast<uintptr_t>(k->scales) & 3u)) return DSA_ERR_MISALIGNED;
  if (k->pages != nullptr) return check_pages(k->pages, max_latents);
  if (need_stride && k->seq_stride_rows < min_stride) return DSA_ERR_INVALID_ARG;
  // MXFP4 rows are read two at a time (128 bytes): sequences start on a pair.
  if (k->fmt == DSA_FMT_MXFP4 && need_stride && (k->seq_stride_rows & 1)) {
    return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

dsa_status_t check_ws(const dsa_config_t& c, int n, int64_t max_latents, void* ws, size_t bytes,
                      Layout* L) {
  *L = layout(c, n, max_latents);
  if (ws == nullptr || bytes < L->total) return DSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return DSA_ERR_MISALIGNED;
  return DSA_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

dsa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// Launch shape of an attention call over n queries: split-KV over the most
// CTAs per query (8, 4 or 2) whose n clusters are all resident at once, else
// one; 64-row tiles for prefill chunks, 32-row tiles for decode.
// An fp8 KV cache (decode only) is read by the split kernel alone: at least
// two CTAs a query, in several waves when the batch is large.
void set_splits(AttnArgs& a, const dsa_config_t& c, int n) {
  a.tile_rows = a.prefill ? 64 : 32;
  a.splits = 1;
  const int sms = device_sm_count();
  for (int sp = kMaxAttnSplits; sp >= 2; sp /= 2) {
    if (static_cast<int64_t>(sp) * n <= sms && n <= attn_max_clusters(sp)) {
      a.splits = sp;
      break;
    }
  }
  a.kv_fp8 = c.kv_fmt == DSA_KV_FP8_E4M3 ? 1 : 0;
  a.kv_scale = c.kv_scale;
  if (a.kv_fp8 && a.splits == 1) a.splits = 2;
}

#define DSA_TRY(expr)                  \
  do {                                 \
    dsa_status_t _s = (expr);          \
    if (_s != DSA_OK) return _s;       \
  } while (0)
#define DSA_CUDA(expr) DSA_TRY(cuda_status(expr))

constexpr int64_t kMaxLatents = int64_t(1) << 30;

// Timing hook and launch counters (dsa_profile_events, dsa_launch_counts).
struct Profile {
  void* const* starts = nullptr;
  void* const* ends = nullptr;
  int n = 0;
  uint64_t next = 0;
};
Profile g_profile[DSA_KERNEL_KINDS];
std::atomic<uint64_t> g_launches[DSA_KERNEL_KINDS]{};

template <typename F>
cudaError_t launch(int kind, cudaStream_t s, F&& f) {
  Profile& p = g_profile[kind];
  const bool timed = p.n > 0;
  const int slot = timed ? static_cast<int>(p.next % static_cast<uint64_t>(p.n)) : 0;
  if (timed) {
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(p.starts[slot]), s);
    if (e != cudaSuccess) return e;
  }
  int n_launched = 1;
  cudaError_t e = f(&n_launched);
  if (e != cudaSuccess) return e;
  g_launches[kind].fetch_add(static_cast<uint64_t>(n_launched), std::memory_order_relaxed);
  if (timed) {
    ++p.next;
    return cudaEventRecord(static_cast<cudaEvent_t>(p.ends[slot]), s);
  }
  return cudaSuccess;
}

// The workspace's selection scratch, or null when no query can have more than
// kSelectOnePass candidates.
int32_t* select_tmp(void* workspace, const Layout& L) {
  return L.has_select_tmp ? reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.select_tmp)
                          : nullptr;
}

// Prefill with bf16 keys runs its indexer stages batched over queries (one
// shared key array, sixteen queries per MMA) when the array has rows.
bool prefill_batched(const dsa_keys_t& k, int prefill, int64_t rows) {
  return prefill && k.fmt == DSA_FMT_BF16 && rows > 0;
}

// Multi-query decode: mq queries per sequence, each sequence holding
// n_tokens[s] tokens (mq = 0: a plain decode batch or one prefill chunk).
struct MultiQuery {
  int mq = 0;
  const int32_t* n_tokens = nullptr;
};

// Launch sequences shared by the public calls. `sel_tmp`: scratch of
// 32768 ids per query for two-pass selections (may be null).
dsa_status_t run_block_stage(const dsa_config_t& c, const uint16_t* q_idx, const float* w,
                             const dsa_keys_t& pooled, const int32_t* n_lat, int B,
                             int64_t max_latents, int32_t* block_ids, float* scores,
                             DeviceStatus* st, int32_t* sel_tmp, cudaStream_t s, int prefill,
                             int64_t ctx, const dsa_keys_t* partial_keys,
                             MultiQuery m = MultiQuery{}, int after_tail_pool = 0) {
  Range range("dsa.block_stage");
  const int64_t nb_max = (max_latents + kBlock - 1) / kBlock;
  if (m.mq == 0 && prefill_batched(pooled, prefill, max_latents / kBlock)) {
    BatchedScanArgs ba{};
    ba.key_data = static_cast<const uint16_t*>(pooled.data);
    ba.key_rows = max_latents / kBlock;  // complete blocks
    ba.q_idx = q_idx;
    ba.w = w;
    ba.n_q = B;
    ba.ctx = ctx;
    ba.ratio = c.ratio;
    ba.mode = ROWS_BLOCKS;
    ba.scores = scores;
    ba.n_cols = nb_max;
    ba.status = st;
    DSA_CUDA(launch(DSA_KERNEL_SCAN, s, [&](int*) { return launch_scan_batched(ba, device_sm_count(), s); }));
  } else {
    ScanArgs sa{};
    sa.fmt = pooled.fmt;
    sa.key_data = pooled.data;
    sa.key_scales = pooled.scales;
    sa.key_stride = prefill && m.mq == 0 ? 0 : pooled.seq_stride_rows;
    sa.q_idx = q_idx;
    sa.w = w;
    sa.n_latents = n_lat;
    sa.max_latents = max_latents;
    sa.mq = m.mq;
    sa.n_tokens = m.n_tokens;
    sa.mode = ROWS_BLOCKS;
    sa.pages = paging_of(pooled.pages, kBlock);
    sa.n_rows = nb_max;
    sa.scores = scores;
    sa.B = B;
    sa.prefill = prefill;
    sa.ctx = ctx;
    sa.ratio = c.ratio;
    sa.defer_wait = after_tail_pool;
    sa.status = st;
    DSA_CUDA(launch(DSA_KERNEL_SCAN, s, [&](int*) { return launch_scan(sa, device_sm_count(), s); }));
  }
  if (prefill) {
    PartialArgs pa{};
    pa.fmt = pooled.fmt;
    pa.key_data = partial_keys->data;
    pa.key_scales = partial_keys->scales;
    pa.q_idx = q_idx;
    pa.w = w;
    pa.n_q = B;
    pa.ctx = ctx;
    pa.ratio = c.ratio;
    pa.mq = m.mq;
    pa.n_tokens = m.n_tokens;
    pa.key_stride = m.mq > 0 ? partial_keys->seq_stride_rows : 0;
    pa.key_rows = m.mq > 0 ? cache_rows(nullptr, 1, B / m.mq, pa.key_stride, max_latents)
                           : max_latents;
    pa.scores = scores;
    pa.n_rows = nb_max;
    DSA_CUDA(launch(DSA_KERNEL_POOL, s, [&](int*) { return launch_prefill_partial(pa, s); }));
  }
  SelectArgs se{};
  se.scores = scores;
  se.n = nb_max;
  se.k = c.k_blocks;
  se.B = B;
  se.out_ids = block_ids;
  se.status = st;
  se.tmp = sel_tmp;
  DSA_CUDA(launch(DSA_KERNEL_SELECT, s, [&](int* nl) { return launch_select(se, s, nl); }));
  return DSA_OK;
}

dsa_status_t run_token_stage(const dsa_config_t& c, const uint16_t* q_idx, const float* w,
                             const dsa_keys_t& keys, const int32_t* block_ids,
                             const int32_t* n_lat, int B, int64_t max_latents, int32_t* token_ids,
                             float* scores, DeviceStatus* st, int32_t* sel_tmp, cudaStream_t s,
                             int prefill, int64_t ctx, MultiQuery m = MultiQuery{}) {
  Range range("dsa.token_stage");
  SelectArgs se{};
  if (block_ids && m.mq == 0 && prefill_batched(keys, prefill, max_latents)) {
    // Dense token scores over every latent, read by the selection through
    // the block ids.
    BatchedScanArgs ba{};
    ba.key_data = static_cast<const uint16_t*>(keys.data);
    ba.key_rows = max_latents;
    ba.q_idx = q_idx;
    ba.w = w;
    ba.n_q = B;
    ba.ctx = ctx;
    ba.ratio = c.ratio;
    ba.mode = ROWS_LATENTS;
    ba.scores = scores;
    ba.n_cols = (max_latents + 7) / 8 * 8;
    ba.status = st;
    DSA_CUDA(launch(DSA_KERNEL_SCAN, s, [&](int*) { return launch_scan_batched(ba, device_sm_count(), s); }));
    se.scores = scores;
    se.n = static_cast<int64_t>(c.k_blocks) * kBlock;
    se.dense_stride = ba.n_cols;
  } else {
    ScanArgs sa{};
    sa.fmt = keys.fmt;
    sa.key_data = keys.data;
    sa.key_scales = keys.scales;
    sa.key_stride = prefill && m.mq == 0 ? 0 : keys.seq_stride_rows;
    sa.q_idx = q_idx;
    sa.w = w;
    sa.n_latents = n_lat;
    sa.max_latents = max_latents;
    sa.mq = m.mq;
    sa.n_tokens = m.n_tokens;
    sa.pages = paging_of(keys.pages, 1);
    if (block_ids) {
      sa.mode = ROWS_GATHER;
      sa.block_ids = block_ids;
      sa.k_blocks = c.k_blocks;
      sa.n_rows = static_cast<int64_t>(c.k_blocks) * kBlock;
    } else {
      sa.mode = ROWS_LATENTS;
      sa.n_rows = (max_latents + 7) / 8 * 8;
    }
    sa.scores = scores;
    sa.B = B;
    sa.prefill = prefill;
    sa.ctx = ctx;
    sa.ratio = c.ratio;
    sa.status = st;
    DSA_CUDA(launch(DSA_KERNEL_SCAN, s, [&](int*) { return launch_scan(sa, device_sm_count(), s); }));
    se.scores = scores;
    se.n = sa.n_rows;
  }
  se.k = c.k_tokens;
  se.B = B;
  se.block_ids = block_ids;
  se.k_blocks = c.k_blocks;
  se.out_ids = token_ids;
  se.status = st;
  se.tmp = sel_tmp;
  DSA_CUDA(launch(DSA_KERNEL_SELECT, s, [&](int* nl) { return launch_select(se, s, nl); }));
  return DSA_OK;
}

}  // namespace

cudaError_t encode_tma_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_rows) {
  // Looked up once, under the thread-safe initialisation of a local static.
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      fn = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (encode == nullptr) return cudaErrorNotSupported;
  const CUtensorMapDataType dt =
      elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int device_sm_count() {
  static std::atomic<int> cached[64]{};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      n = 152;
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

__global__ void identity_blocks_kernel(const int32_t* n_latents, int k_blocks, int32_t* out) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.x;
  const int nb = (n_latents[b] + 7) / 8;
  for (int i = threadIdx.x; i < k_blocks; i += blockDim.x) {
    out[static_cast<int64_t>(b) * k_blocks + i] = i < nb ? i : -1;
  }
}

}  // namespace

cudaError_t launch_identity_blocks(const int32_t* n_latents, int B, int k_blocks,
                                   int32_t* block_ids, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(identity_blocks_kernel, dim3(B), dim3(256), 0, s, 1, n_latents, k_blocks,
                             block_ids);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa

using namespace dsa;

extern "C" {

void dsa_default_config(dsa_config_t* c) {
  if (c == nullptr) return;
  c->n_heads = kHeads;
  c->latent_dim = kLatent;
  c->n_idx_heads = kIdxHeads;
  c->idx_dim = kIdxDim;
  c->block = kBlock;
  c->k_blocks = 2048;
  c->k_tokens = 512;
  c->window = 128;
  c->ratio = 1;
  c->sm_scale = 0.f;
  c->kv_fmt = DSA_KV_BF16;
  c->kv_scale = 1.f;
}

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

dsa_status_t dsa_workspace_size(const dsa_config_t* cfg, int n_queries, int64_t max_latents,
                                size_t* bytes) {
  DSA_TRY(check_config(cfg));
  if (bytes == nullptr || n_queries < 0 || max_latents < 0 || max_latents > kMaxLatents) {
    return DSA_ERR_INVALID_ARG;
  }
  *bytes = layout(*cfg, n_queries, max_latents).total;
  return DSA_OK;
}

dsa_status_t dsa_pool_index_keys(const dsa_config_t* cfg, const dsa_keys_t* keys,
                                 const int32_t* n_latents, int B, int64_t max_latents,
                                 int tail_only, const dsa_keys_out_t* pooled, void* workspace,
                                 size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents || pooled == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  DSA_TRY(check_keys(keys, max_latents, true, max_latents));
  const dsa_keys_t pk{pooled->fmt, pooled->data, pooled->scales, pooled->seq_stride_rows,
                      pooled->pages};
  DSA_TRY(check_keys(&pk, (max_latents + 7) / 8, true, max_latents));
  if (pooled->fmt != keys->fmt || n_latents == nullptr) return DSA_ERR_INVALID_ARG;
  if (!same_pages(keys->pages, pooled->pages)) return DSA_ERR_INVALID_ARG;
  Layout L;
  DSA_TRY(check_ws(*cfg, B, max_latents, workspace, workspace_bytes, &L));
  if (B == 0 || max_latents == 0) return DSA_OK;
  Range range("dsa.pool");
  PoolArgs a{};
  a.fmt = keys->fmt;
  a.key_data = keys->data;
  a.key_scales = keys->scales;
  a.key_stride = keys->seq_stride_rows;
  a.n_latents = n_latents;
  a.max_latents = max_latents;
  a.B = B;
  a.tail_only = tail_only;
  a.out_data = pooled->data;
  a.out_scales = pooled->scales;
  a.out_stride = pooled->seq_stride_rows;
  a.key_pages = paging_of(keys->pages, 1);
  a.out_pages = paging_of(pooled->pages, kBlock);
  a.key_rows = cache_rows(keys->pages, 1, B, keys->seq_stride_rows, max_latents);
  a.out_rows = cache_rows(pooled->pages, kBlock, B, pooled->seq_stride_rows,
                          (max_latents + kBlock - 1) / kBlock);
  a.status = at<DeviceStatus>(workspace, L.status);
  DSA_CUDA(launch(DSA_KERNEL_POOL, static_cast<cudaStream_t>(stream), [&](int*) { return launch_pool(a, static_cast<cudaStream_t>(stream)); }));
  return DSA_OK;
}

dsa_status_t dsa_index_blocks(const dsa_config_t* cfg, const void* q_idx, const float* w,
                              const dsa_keys_t* pooled, const int32_t* n_latents, int B,
                              int64_t max_latents, int32_t* block_ids, float* block_scores,
                              void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents) return DSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || w == nullptr || n_latents == nullptr || block_ids == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(block_ids) ||
      (block_scores && !aligned16(block_scores))) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(pooled, (max_latents + 7) / 8, true, max_latents));
  Layout L;
  DSA_TRY(check_ws(*cfg, B, max_latents, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  float* scores = block_scores ? block_scores : at<float>(workspace, L.block_scores);
  return run_block_stage(*cfg, static_cast<const uint16_t*>(q_idx), w, *pooled, n_latents, B,
                         max_latents, block_ids, scores, at<DeviceStatus>(workspace, L.status),
                         select_tmp(workspace, L), static_cast<cudaStream_t>(stream), 0, 0,
                         nullptr);
}

dsa_status_t dsa_topk(const dsa_config_t* cfg, const void* q_idx, const float* w,
                      const dsa_keys_t* keys, const int32_t* block_ids,
                      const int32_t* n_latents, int B, int64_t max_latents, int32_t* token_ids,
                      float* token_scores, void* workspace, size_t workspace_bytes,
                      dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents) return DSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || w == nullptr || n_latents == nullptr || token_ids == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(token_ids) ||
      (block_ids && !aligned16(block_ids)) || (token_scores && !aligned16(token_scores))) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(keys, max_latents, true, max_latents));
  Layout L;
  DSA_TRY(check_ws(*cfg, B, max_latents, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  float* scores = token_scores ? token_scores : at<float>(workspace, L.token_scores);
  return run_token_stage(*cfg, static_cast<const uint16_t*>(q_idx), w, *keys, block_ids,
                         n_latents, B, max_latents, token_ids, scores,
                         at<DeviceStatus>(workspace, L.status), select_tmp(workspace, L),
                         static_cast<cudaStream_t>(stream), 0, 0);
}

}  // extern "C"

namespace {

// dsa_sparse_attn_decode and its paged form (pages != nullptr).
dsa_status_t attn_decode(const dsa_config_t* cfg, const void* q, const void* latents,
                         int64_t latent_seq_stride_rows, const dsa_pages_t* pages,
                         const int32_t* n_latents, const int32_t* token_ids, const void* swa,
                         const int32_t* swa_len, int B, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || latent_seq_stride_rows < 0) return DSA_ERR_INVALID_ARG;
  if (q == nullptr || latents == nullptr || n_latents == nullptr || token_ids == nullptr ||
      swa == nullptr || swa_len == nullptr || out == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q) || !aligned16(latents) || !aligned16(swa) || !aligned16(out) ||
      !aligned16(token_ids) || (lse && !aligned16(lse))) {
    return DSA_ERR_MISALIGNED;
  }
  if (pages != nullptr) DSA_TRY(check_pages(pages, 0));
  Layout L;
  DSA_TRY(check_ws(*cfg, B, 0, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.latents = static_cast<const uint16_t*>(latents);
  a.lat_stride = latent_seq_stride_rows;
  a.lat_rows = static_cast<int64_t>(B) * latent_seq_stride_rows;
  if (pages != nullptr) {
    a.pages = paging_of(pages, 1);
    a.lat_stride = static_cast<int64_t>(pages->pages_per_seq) * pages->page_rows;
    a.lat_rows = pages->n_pages * pages->page_rows;
  }
  a.n_latents = n_latents;
  a.token_ids = token_ids;
  a.k_tokens = cfg->k_tokens;
  a.swa = static_cast<const uint16_t*>(swa);
  a.swa_len = swa_len;
  a.window = cfg->window;
  a.B = B;
  a.scale_log2 = tau(*cfg) * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = at<DeviceStatus>(workspace, L.status);
  set_splits(a, *cfg, B);
  Range range("dsa.attention");
  DSA_CUDA(launch(DSA_KERNEL_ATTN, static_cast<cudaStream_t>(stream), [&](int*) { return launch_attn(a, static_cast<cudaStream_t>(stream)); }));
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status_t dsa_sparse_attn_decode(const dsa_config_t* cfg, const void* q, const void* latents,
                                    int64_t latent_seq_stride_rows, const int32_t* n_latents,
                                    const int32_t* token_ids, const void* swa,
                                    const int32_t* swa_len, int B, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    dsa_stream_t stream) {
  return attn_decode(cfg, q, latents, latent_seq_stride_rows, nullptr, n_latents, token_ids, swa,
                     swa_len, B, out, lse, workspace, workspace_bytes, stream);
}

dsa_status_t dsa_sparse_attn_decode_paged(const dsa_config_t* cfg, const void* q,
                                          const void* latents, const dsa_pages_t* pages,
                                          const int32_t* n_latents, const int32_t* token_ids,
                                          const void* swa, const int32_t* swa_len, int B,
                                          void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, dsa_stream_t stream) {
  if (pages == nullptr) return DSA_ERR_INVALID_ARG;
  return attn_decode(cfg, q, latents, 0, pages, n_latents, token_ids, swa, swa_len, B, out, lse,
                     workspace, workspace_bytes, stream);
}

dsa_status_t dsa_decode_step(const dsa_config_t* cfg, const void* q, const void* q_idx,
                             const float* w, const dsa_keys_t* keys, const dsa_keys_out_t* pooled,
                             int update_pool, const void* latents,
                             int64_t latent_seq_stride_rows, const int32_t* n_latents,
                             int64_t max_latents, const void* swa, const int32_t* swa_len, int B,
                             int32_t* block_ids, int32_t* token_ids, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents || pooled == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (keys != nullptr && keys->pages == nullptr && latent_seq_stride_rows < max_latents) {
    return DSA_ERR_INVALID_ARG;
  }
  if (q == nullptr || q_idx == nullptr || w == nullptr || latents == nullptr ||
      n_latents == nullptr || swa == nullptr || swa_len == nullptr || out == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(w) || !aligned16(latents) ||
      !aligned16(swa) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (block_ids && !aligned16(block_ids)) || (token_ids && !aligned16(token_ids))) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(keys, max_latents, true, max_latents));
  const dsa_keys_t pk{pooled->fmt, pooled->data, pooled->scales, pooled->seq_stride_rows,
                      pooled->pages};
  DSA_TRY(check_keys(&pk, (max_latents + 7) / 8, true, max_latents));
  if (pooled->fmt != keys->fmt) return DSA_ERR_INVALID_ARG;
  if (!same_pages(keys->pages, pooled->pages)) return DSA_ERR_INVALID_ARG;
  Layout L;
  DSA_TRY(check_ws(*cfg, B, max_latents, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  Range range("dsa.decode_step");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(workspace, L.status);
  if (update_pool && max_latents > 0) {
    Range pool_range("dsa.pool");
    PoolArgs a{};
    a.fmt = keys->fmt;
    a.key_data = keys->data;
    a.key_scales = keys->scales;
    a.key_stride = keys->seq_stride_rows;
    a.n_latents = n_latents;
    a.max_latents = max_latents;
    a.B = B;
    a.tail_only = 1;
    a.out_data = pooled->data;
    a.out_scales = pooled->scales;
    a.out_stride = pooled->seq_stride_rows;
    a.key_pages = paging_of(keys->pages, 1);
    a.out_pages = paging_of(pooled->pages, kBlock);
    a.key_rows = cache_rows(keys->pages, 1, B, keys->seq_stride_rows, max_latents);
    a.out_rows = cache_rows(pooled->pages, kBlock, B, pooled->seq_stride_rows,
                            (max_latents + kBlock - 1) / kBlock);
    a.status = st;
    DSA_CUDA(launch(DSA_KERNEL_POOL, s, [&](int*) { return launch_pool(a, s); }));
  }
  const uint16_t* qi = static_cast<const uint16_t*>(q_idx);
  int32_t* bids = block_ids ? block_ids : at<int32_t>(workspace, L.block_ids);
  const int32_t* gather_ids = nullptr;
  if (L.nb_max > cfg->k_blocks) {
    // right after the tail pool, the block scan streams every block the pool
    // does not rewrite before it waits for the pool
    DSA_TRY(run_block_stage(*cfg, qi, w, pk, n_latents, B, max_latents, bids,
                            at<float>(workspace, L.block_scores), st, select_tmp(workspace, L), s,
                            0, 0, nullptr, MultiQuery{},
                            update_pool && max_latents > 0 && !pk.pages ? 1 : 0));
    gather_ids = bids;
  } else if (block_ids) {
    DSA_CUDA(launch(DSA_KERNEL_OTHER, s, [&](int*) { return launch_identity_blocks(n_latents, B, cfg->k_blocks, block_ids, s); }));
  }
  int32_t* tids = token_ids ? token_ids : at<int32_t>(workspace, L.token_ids);
  DSA_TRY(run_token_stage(*cfg, qi, w, *keys, gather_ids, n_latents, B, max_latents, tids,
                          at<float>(workspace, L.token_scores), st, select_tmp(workspace, L), s, 0,
                          0));
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.latents = static_cast<const uint16_t*>(latents);
  a.lat_stride = latent_seq_stride_rows;
  a.lat_rows = static_cast<int64_t>(B) * latent_seq_stride_rows;
  if (keys->pages) {  // the latents share the keys' page table
    a.pages = paging_of(keys->pages, 1);
    a.lat_stride = static_cast<int64_t>(keys->pages->pages_per_seq) * keys->pages->page_rows;
    a.lat_rows = keys->pages->n_pages * keys->pages->page_rows;
  }
  a.n_latents = n_latents;
  a.token_ids = tids;
  a.k_tokens = cfg->k_tokens;
  a.swa = static_cast<const uint16_t*>(swa);
  a.swa_len = swa_len;
  a.window = cfg->window;
  a.B = B;
  a.scale_log2 = tau(*cfg) * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = st;
  set_splits(a, *cfg, B);
  Range attn_range("dsa.attention");
  DSA_CUDA(launch(DSA_KERNEL_ATTN, s, [&](int*) { return launch_attn(a, s); }));
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn_prefill(const dsa_config_t* cfg, int n_q, int64_t ctx_len,
                                     const void* q, const void* q_idx, const float* w,
                                     const void* latents, const dsa_keys_t* keys,
                                     const dsa_keys_t* pooled, const void* swa, void* out,
                                     float* lse, int32_t* token_ids, void* workspace,
                                     size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (cfg->kv_fmt != DSA_KV_BF16) return DSA_ERR_UNSUPPORTED;  // fp8 caches: decode only
  if (n_q < 0 || ctx_len < 0) return DSA_ERR_INVALID_ARG;
  const int64_t n_lat = (ctx_len + n_q) / cfg->ratio;
  if (n_lat > kMaxLatents) return DSA_ERR_INVALID_ARG;
  if (q == nullptr || q_idx == nullptr || w == nullptr || latents == nullptr || swa == nullptr ||
      out == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(w) || !aligned16(latents) ||
      !aligned16(swa) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (token_ids && !aligned16(token_ids))) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(keys, 0, false));
  DSA_TRY(check_keys(pooled, 0, false));
  if (pooled->fmt != keys->fmt) return DSA_ERR_INVALID_ARG;
  if (keys->pages != nullptr || pooled->pages != nullptr) return DSA_ERR_INVALID_ARG;
  Layout L;
  DSA_TRY(check_ws(*cfg, n_q, n_lat, workspace, workspace_bytes, &L));
  if (n_q == 0) return DSA_OK;
  Range range("dsa.prefill");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(workspace, L.status);
  const uint16_t* qi = static_cast<const uint16_t*>(q_idx);
  int32_t* bids = at<int32_t>(workspace, L.block_ids);
  DSA_TRY(run_block_stage(*cfg, qi, w, *pooled, nullptr, n_q, n_lat, bids,
                          at<float>(workspace, L.block_scores), st, select_tmp(workspace, L), s, 1,
                          ctx_len, keys));
  int32_t* tids = token_ids ? token_ids : at<int32_t>(workspace, L.token_ids);
  DSA_TRY(run_token_stage(*cfg, qi, w, *keys, bids, nullptr, n_q, n_lat, tids,
                          at<float>(workspace, L.token_scores), st, select_tmp(workspace, L), s, 1,
                          ctx_len));
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.latents = static_cast<const uint16_t*>(latents);
  a.lat_stride = n_lat;
  a.lat_rows = n_lat;
  a.token_ids = tids;
  a.k_tokens = cfg->k_tokens;
  a.swa = static_cast<const uint16_t*>(swa);
  a.window = cfg->window;
  a.B = n_q;
  a.scale_log2 = tau(*cfg) * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.prefill = 1;
  a.ctx = ctx_len;
  a.ratio = cfg->ratio;
  a.status = st;
  set_splits(a, *cfg, n_q);
  Range attn_range("dsa.attention");
  DSA_CUDA(launch(DSA_KERNEL_ATTN, s, [&](int*) { return launch_attn(a, s); }));
  return DSA_OK;
}

dsa_status_t dsa_decode_multi(const dsa_config_t* cfg, int n_q, const int32_t* n_tokens,
                              const void* q, const void* q_idx, const float* w,
                              const dsa_keys_t* keys, const dsa_keys_t* pooled,
                              const void* latents, int64_t latent_seq_stride_rows,
                              int64_t max_latents, const void* swa, int B, void* out, float* lse,
                              int32_t* token_ids, void* workspace, size_t workspace_bytes,
                              dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (cfg->kv_fmt != DSA_KV_BF16) return DSA_ERR_UNSUPPORTED;  // fp8 caches: single-query decode
  if (n_q < 1 || B < 0 || max_latents < 0 || max_latents > kMaxLatents ||
      latent_seq_stride_rows < max_latents || static_cast<int64_t>(B) * n_q > (1 << 30)) {
    return DSA_ERR_INVALID_ARG;
  }
  if (n_tokens == nullptr || q == nullptr || q_idx == nullptr || w == nullptr ||
      latents == nullptr || swa == nullptr || out == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(w) || !aligned16(latents) ||
      !aligned16(swa) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (token_ids && !aligned16(token_ids)) || (reinterpret_cast<uintptr_t>(n_tokens) & 3u)) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(keys, max_latents, true));
  DSA_TRY(check_keys(pooled, max_latents / kBlock, true));
  if (pooled->fmt != keys->fmt) return DSA_ERR_INVALID_ARG;
  if (keys->pages != nullptr || pooled->pages != nullptr) return DSA_ERR_INVALID_ARG;
  const int nq_total = B * n_q;
  Layout L;
  DSA_TRY(check_ws(*cfg, nq_total, max_latents, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  Range range("dsa.decode_multi");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(workspace, L.status);
  const uint16_t* qi = static_cast<const uint16_t*>(q_idx);
  const MultiQuery m{n_q, n_tokens};
  int32_t* bids = at<int32_t>(workspace, L.block_ids);
  DSA_TRY(run_block_stage(*cfg, qi, w, *pooled, nullptr, nq_total, max_latents, bids,
                          at<float>(workspace, L.block_scores), st, select_tmp(workspace, L), s, 1,
                          0, keys, m));
  int32_t* tids = token_ids ? token_ids : at<int32_t>(workspace, L.token_ids);
  DSA_TRY(run_token_stage(*cfg, qi, w, *keys, bids, nullptr, nq_total, max_latents, tids,
                          at<float>(workspace, L.token_scores), st, select_tmp(workspace, L), s, 1,
                          0, m));
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.latents = static_cast<const uint16_t*>(latents);
  a.lat_stride = latent_seq_stride_rows;
  a.lat_rows = static_cast<int64_t>(B) * latent_seq_stride_rows;
  a.token_ids = tids;
  a.k_tokens = cfg->k_tokens;
  a.swa = static_cast<const uint16_t*>(swa);
  a.window = cfg->window;
  a.B = nq_total;
  a.scale_log2 = tau(*cfg) * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.prefill = 1;
  a.ratio = cfg->ratio;
  a.mq = n_q;
  a.n_tokens = n_tokens;
  a.swa_seq_rows = cfg->window + n_q - 1;
  a.status = st;
  set_splits(a, *cfg, nq_total);
  Range attn_range("dsa.attention");
  DSA_CUDA(launch(DSA_KERNEL_ATTN, s, [&](int*) { return launch_attn(a, s); }));
  return DSA_OK;
}

dsa_status_t dsa_compress_append(const dsa_config_t* cfg, int B, const int32_t* n_tokens,
                                 const void* kv, const float* gate, const dsa_keys_t* new_keys,
                                 void* latents, int64_t latent_seq_stride_rows,
                                 const dsa_keys_out_t* keys, const dsa_keys_out_t* pooled,
                                 int64_t max_latents, void* workspace, size_t workspace_bytes,
                                 dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (cfg->ratio > 32) return DSA_ERR_UNSUPPORTED;
  if (cfg->kv_fmt != DSA_KV_BF16) return DSA_ERR_UNSUPPORTED;  // it writes bf16 latents
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents || keys == nullptr ||
      pooled == nullptr || new_keys == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (n_tokens == nullptr || kv == nullptr || gate == nullptr || latents == nullptr ||
      new_keys->data == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  const bool paged = keys->pages != nullptr;
  if (!paged && latent_seq_stride_rows < max_latents) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(latents) || !aligned16(new_keys->data) ||
      (reinterpret_cast<uintptr_t>(n_tokens) & 3u) || (reinterpret_cast<uintptr_t>(gate) & 3u)) {
    return DSA_ERR_MISALIGNED;
  }
  const dsa_keys_t kk{keys->fmt, keys->data, keys->scales, keys->seq_stride_rows, keys->pages};
  DSA_TRY(check_keys(&kk, max_latents, true, max_latents));
  const dsa_keys_t pk{pooled->fmt, pooled->data, pooled->scales, pooled->seq_stride_rows,
                      pooled->pages};
  DSA_TRY(check_keys(&pk, (max_latents + 7) / 8, true, max_latents));
  if (pooled->fmt != keys->fmt || new_keys->fmt != keys->fmt) return DSA_ERR_INVALID_ARG;
  if (new_keys->fmt != DSA_FMT_BF16 && new_keys->scales == nullptr) return DSA_ERR_INVALID_ARG;
  if (!same_pages(keys->pages, pooled->pages)) return DSA_ERR_INVALID_ARG;
  Layout L;
  DSA_TRY(check_ws(*cfg, B, max_latents, workspace, workspace_bytes, &L));
  if (B == 0) return DSA_OK;
  Range range("dsa.compress_append");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus* st = at<DeviceStatus>(workspace, L.status);
  int32_t* n_lat = at<int32_t>(workspace, L.token_ids);  // B entries: the new latent counts
  AppendArgs ap{};
  ap.B = B;
  ap.ratio = cfg->ratio;
  ap.n_tokens = n_tokens;
  ap.kv = static_cast<const uint16_t*>(kv);
  ap.gate = gate;
  ap.fmt = keys->fmt;
  ap.new_key = static_cast<const uint8_t*>(new_keys->data);
  ap.new_scales = new_keys->scales;
  ap.latents = static_cast<uint16_t*>(latents);
  ap.lat_stride = latent_seq_stride_rows;
  ap.key_data = static_cast<uint8_t*>(keys->data);
  ap.key_scales = keys->scales;
  ap.key_stride = keys->seq_stride_rows;
  ap.pages = paging_of(keys->pages, 1);
  ap.max_latents = max_latents;
  ap.n_lat_out = n_lat;
  ap.status = st;
  DSA_CUDA(launch(DSA_KERNEL_POOL, s, [&](int*) { return launch_append(ap, s); }));
  PoolArgs a{};
  a.fmt = keys->fmt;
  a.key_data = keys->data;
  a.key_scales = keys->scales;
  a.key_stride = keys->seq_stride_rows;
  a.n_latents = n_lat;
  a.max_latents = max_latents;
  a.B = B;
  a.tail_only = 1;
  a.out_data = pooled->data;
  a.out_scales = pooled->scales;
  a.out_stride = pooled->seq_stride_rows;
  a.key_pages = paging_of(keys->pages, 1);
  a.out_pages = paging_of(pooled->pages, kBlock);
  a.key_rows = cache_rows(keys->pages, 1, B, keys->seq_stride_rows, max_latents);
  a.out_rows = cache_rows(pooled->pages, kBlock, B, pooled->seq_stride_rows,
                          (max_latents + kBlock - 1) / kBlock);
  a.status = st;
  DSA_CUDA(launch(DSA_KERNEL_POOL, s, [&](int*) { return launch_pool(a, s); }));
  return DSA_OK;
}

dsa_status_t dsa_profile_events(int kind, void* const* starts, void* const* ends, int n) {
  if (kind < 0 || kind >= DSA_KERNEL_KINDS || n < 0) return DSA_ERR_INVALID_ARG;
  if (n > 0 && (starts == nullptr || ends == nullptr)) return DSA_ERR_INVALID_ARG;
  Profile& p = g_profile[kind];
  p.starts = n > 0 ? starts : nullptr;
  p.ends = n > 0 ? ends : nullptr;
  p.n = n;
  p.next = 0;
  return DSA_OK;
}

dsa_status_t dsa_launch_counts(uint64_t* counts, int reset) {
  if (counts == nullptr) return DSA_ERR_INVALID_ARG;
  for (int k = 0; k < DSA_KERNEL_KINDS; ++k) {
    counts[k] = reset ? g_launches[k].exchange(0, std::memory_order_relaxed)
                      : g_launches[k].load(std::memory_order_relaxed);
  }
  return DSA_OK;
}

dsa_status_t dsa_selftest_timeout(void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  if (workspace == nullptr || workspace_bytes < sizeof(DeviceStatus)) return DSA_ERR_INVALID_ARG;
  // about 1 ms at the GB300's 2.07 GHz maximum SM clock
  constexpr long long kLimitCycles = 2000000;
  DSA_CUDA(launch(DSA_KERNEL_OTHER, static_cast<cudaStream_t>(stream), [&](int*) {
    return launch_timeout_selftest(static_cast<DeviceStatus*>(workspace), kLimitCycles,
                                   static_cast<cudaStream_t>(stream));
  }));
  return DSA_OK;
}

dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, uint32_t* info) {
  if (workspace == nullptr) return DSA_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus h{};
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    return DSA_ERR_CUDA;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  if (h.code != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), s) != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  }
  if (info) *info = h.info;
  return static_cast<dsa_status_t>(h.code);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dsa_topk_noalloc: the token stage with its candidate scores in a statically
// defined device array, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------

namespace {

// Candidate-score scratch of dsa_topk_noalloc (8 MiB on every device that
// loads the library). Device code could name it directly; host code must use
// the address cudaGetSymbolAddress returns for the current device, since the
// symbol itself is only a host-side stand-in.
static __device__ __align__(256) float g_topk_scratch[DSA_TOPK_NOALLOC_MAX_SCORES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_topk_scratch on the current device, looked up once per
// device (the first call on a device does this set-up).
dsa_status_t topk_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) {
      return DSA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" dsa_status_t dsa_topk_noalloc(const dsa_config_t* cfg, const void* q_idx,
                                         const float* w, const dsa_keys_t* keys,
                                         const int32_t* block_ids, const int32_t* n_latents,
                                         int B, int64_t max_latents, int32_t* token_ids,
                                         dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (B < 0 || max_latents < 0 || max_latents > kMaxLatents) return DSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || w == nullptr || n_latents == nullptr || token_ids == nullptr) {
    return DSA_ERR_INVALID_ARG;
  }
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(token_ids) ||
      (block_ids && !aligned16(block_ids))) {
    return DSA_ERR_MISALIGNED;
  }
  DSA_TRY(check_keys(keys, max_latents, true, max_latents));
  const int64_t n_cand = block_ids ? static_cast<int64_t>(cfg->k_blocks) * kBlock
                                   : (max_latents + 7) / 8 * 8;
  if (static_cast<int64_t>(B) * n_cand > DSA_TOPK_NOALLOC_MAX_SCORES) return DSA_ERR_WORKSPACE;
  if (B == 0) return DSA_OK;
  float* scores = nullptr;
  DSA_TRY(topk_scratch(&scores));
  return run_token_stage(*cfg, static_cast<const uint16_t*>(q_idx), w, *keys, block_ids,
                         n_latents, B, max_latents, token_ids, scores, nullptr, nullptr,
                         static_cast<cudaStream_t>(stream), 0, 0);
}
