// S5 - S7: attention over the gathered latents and the sliding window under one
// softmax (miles.radixark.com "DeepSeek-V4.1 Flash", §1 "Architecture": one
// 512-wide latent per position is both key and value for all 64 query heads;
// recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention":
// the 128-token window plus the selected latents).
//
// A CTA's rows (its share of the window rows, then its share of the selected
// latents in id order) stream through shared memory in tiles of 32 rows; two tcgen05 MMAs per tile run
// with fp32 accumulators in tensor memory:
//   S   = Q . KV^T    (M = 128 with the 64 heads in lanes 0..63, N = 32 rows, K = 512)
//   O^T += KV^T . P^T (four M = 128 slices of the 512 latent dims, N = 64 heads,
//                      K = 32 rows; the KV tile is read as an MN-major operand)
// Warp roles: warps 0-3 math (softmax for the 64 heads by warps 0-1, one head
// per thread; O rescaling by all four, thread = TMEM lane; the epilogue by
// these four and the four loader warps, which are idle by then),
// warps 4-7 loaders (every loader warp copies its quarter of the rows of each
// tile by cp.async, the 1 KB rows gathered at random; each lane's completion
// arrives on the slot's mbarrier by itself, so the four warps' copies of a
// tile are in flight together and no warp waits for its own; Q comes by
// eight TMA boxes that land in the swizzled operand layout), warp 8 issues
// the QK^T MMAs and warp 9 the PV MMAs (a barrier wait costs a single thread
// a few hundred cycles; two issuers overlap their waits). Four 32 KB slots
// keep several tiles in flight. S is double-buffered in tensor memory so QK^T of tile t + 1
// runs while the softmax of tile t does. The running maximum only moves when
// it grows by more than 2^8 (the stale maximum keeps every P value <= 256,
// exact enough in bf16 and fp32), so rescaling O is rare.
//
// The window rows are inputs of the step: they stream while the previous
// kernel (the token selection) still runs, and only the tiles holding
// selected latents wait for its ids (programmatic dependent launch).
//
// Split-KV: while S x queries CTAs fit the SMs (S = 8, 4 or 2), the window
// rows and the selected latents of a query are each cut in S parts handled by
// the S CTAs of a cluster. CTA r finishes the latent dims [r D, r D + D),
// D = 512 / S: once every CTA's MMAs are done (a cluster barrier), each stores
// straight into each peer's idle ring (distributed shared memory) its
// unnormalised O for that peer's dims and its (max, sum); after a second
// cluster barrier each merges its dims and writes them.
//
// The epilogue works in chunks of 16 heads in rolled loops and writes the
// output from registers (a warp stores 32 consecutive dims of a head at a
// time): it runs once per CTA, so its code is fetched cold, and a compact
// loop costs far less than a fully unrolled one.
#include <algorithm>
#include <cstddef>

#include "kernels.h"

namespace dsa {

namespace {

constexpr int kLoadWarp0 = 4;
constexpr int kLoadWarps = 4;
constexpr int kMaxSlots = 4;
constexpr int kMmaWarp = kLoadWarp0 + kLoadWarps;  // 8: QK^T issuer (and TMEM owner)
constexpr int kPvWarp = kMmaWarp + 1;          // 9: PV issuer
constexpr int kThreads = 32 * (kPvWarp + 1);   // 320
constexpr int kMathBar = 1;         // named barrier of the 128 math threads
constexpr int kEpiBar = 2;          // named barrier of the epilogue (math + loader warps)
constexpr int kLoadBar = 3;         // named barrier of the 128 loader threads
constexpr int kEpiThreads = 32 * kMmaWarp;  // 256

// Shared-memory plan (offsets from a 1024-aligned base). The QK^T MMA reads
// 64 rows past each Q atom (they only feed unused accumulator lanes); past
// the last atom they land in the P buffers, which is harmless.
constexpr int kQ = 0;                              // 8 atoms x 64 heads x 128 B; output staging
constexpr int kP = kQ + 8 * kHeads * 128;          // 2 x (64 heads x 128 B: up to 64 rows bf16)
constexpr int kPBytes = kHeads * 128;
constexpr int kKV = kP + 2 * kPBytes;              // the ring: 128 KB of tiles
constexpr int kKVBytes = 128 * 1024;
constexpr int kIds = kKV + kKVBytes;               // compacted latent ids

// Tiles of ROWS rows (32 or 64): 128 / ROWS ring slots of 8 atoms (64 dims x
// ROWS rows x 128 B each); each loader warp fills 32 rows of its slot's tiles.
template <int ROWS>
struct TileShape {
  static_assert(ROWS == 32 || ROWS == 64, "tile rows");
  static constexpr int kSlots = kKVBytes / (ROWS * 1024);
  static constexpr int kAtomBytes = ROWS * 128;
  static constexpr int kSlotBytes = 8 * kAtomBytes;
};
constexpr int kMisc = kIds + kMaxKTokens * 4;
constexpr int kMiscBytes = 2048;
constexpr int kSmemBytes = kMisc + kMiscBytes + 1024;  // + alignment slack of the base
constexpr int kTmemCols = 512;  // S[b]: cols [64 b, 64 b + 32); O^T slice m: [128 + 64 m, ...)
constexpr uint32_t kQBytes = kHeads * kLatent * 2;  // one query's bf16 Q, 8 atoms
static_assert(kP - kQ == static_cast<int>(kQBytes), "Q region");
// Split-KV exchange payload from a sender to the CTA finishing dims
// [p D, p D + D): the sender's unnormalised O for those dims, bf16, one
// 128-byte row of 64 heads per dim (16-byte chunk c of row dd stored at chunk
// c ^ (dd & 7)), then the sender's (max, sum) per head.
__host__ __device__ constexpr int xchg_bytes(int S) { return (kLatent / S) * 128 + kHeads * 8; }
constexpr int kRecv = kKV;   // incoming payloads: slot s from sender s, in the ring
static_assert(2 * xchg_bytes(2) <= kKVBytes && 4 * xchg_bytes(4) <= kKVBytes &&
                  kMaxAttnSplits * xchg_bytes(kMaxAttnSplits) <= kKVBytes,
              "receive areas fit the ring");
constexpr int kWgt = kP;     // [S][64 h] merge weights, in the P buffers
static_assert(kWgt + kMaxAttnSplits * kHeads * 4 <= kKV, "merge weights fit the P buffers");

struct Misc {
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots], s_full[2], s_free[2], p_full[2], p_empty[2];
  uint64_t q_done, ids_ready;
  uint64_t q_conv;                   // (fp8 cache) Q is in f16, scaled per head
  uint64_t o_done;                   // every MMA of the CTA has completed
  alignas(16) float q_unscale[kHeads];  // (fp8 cache) kv_scale * 2^-e_h of head h
  uint32_t tmem_base;
  int abort;
  int n_sel;
  int warp_cnt[4];
  alignas(16) float alpha[kHeads];
  alignas(16) float inv_l[kHeads];  // read four at a time (16-byte loads)
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block");
static_assert(offsetof(Misc, inv_l) % 16 == 0 && kMisc % 16 == 0 && kWgt % 16 == 0,
              "16-byte loads of inv_l and of the merge weights");

// A tile's raw scores of this thread's head (TMEM columns [addr, addr + R)),
// -inf past the tile's valid rows: one TMEM load, one wait. The softmax scale
// (positive) is applied by max_scores and exp_pack.
template <int R>
__device__ __forceinline__ void load_scores(uint32_t addr, int valid, float (&z)[R]) {
  if constexpr (R == 64) {
    tmem_ld64(addr, z);
  } else {
    static_assert(R == 32, "tile rows");
    tmem_ld32(addr, z);
  }
#pragma unroll
  for (int i = 0; i < R; ++i) z[i] = i < valid ? z[i] : -INFINITY;
}
// scale * max_i z[i] (log2 units; equal to max_i (scale * z[i]) for scale > 0),
// the maximum as four independent chains
template <int R>
__device__ __forceinline__ float max_scores(const float (&z)[R], float scale) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < R; ++i) m4[i & 3] = fmaxf(m4[i & 3], z[i]);
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale;
}
// 2^x by the ex2 instruction (flushing subnormal results to zero: a
// probability below 2^-126 of the running maximum's is dropped)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// p_i = 2^(scale z_i - m) (one fused multiply-add a score) packed as bf16
// pairs into pk; returns sum_i p_i over the fp32 probabilities (four partial
// sums)
template <int R, bool F16 = false>
__device__ __forceinline__ float exp_pack(const float (&z)[R], float scale, float m,
                                          uint32_t (&pk)[R / 2]) {
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < R; i += 2) {
    const float p0 = ex2_ftz(fmaf(z[i], scale, -m)), p1 = ex2_ftz(fmaf(z[i + 1], scale, -m));
    s4[(i >> 1) & 3] += p0 + p1;
    if constexpr (F16) {  // the PV operands of an fp8 cache are f16
      const __half2 p2 = __floats2half2_rn(p0, p1);
      pk[i / 2] = *reinterpret_cast<const uint32_t*>(&p2);
    } else {
      const __nv_bfloat162 p2 = __floats2bfloat162_rn(p0, p1);
      pk[i / 2] = *reinterpret_cast<const uint32_t*>(&p2);
    }
  }
  return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

// 8 E4M3 codes (two words, byte i = code i) -> 8 f16 (exact: every E4M3 value
// is an f16 normal, subnormal or zero), element i in the low half of word i / 2.
__device__ __forceinline__ uint4 e4m3x8_to_f16(uint2 c) {
  uint4 r;
  asm("{\n .reg .b16 a, b, c, d;\n mov.b32 {a, b}, %4;\n mov.b32 {c, d}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n"
      " cvt.rn.f16x2.e4m3x2 %2, c;\n cvt.rn.f16x2.e4m3x2 %3, d;\n}\n"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "r"(c.x), "r"(c.y));
  return r;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* m,
                                         DeviceStatus* st) {
  return mbar_wait_abortable(bar, parity, &m->abort, st, SITE_ATTN);
}

template <int ROWS, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap) {
  using TS = TileShape<ROWS>;
  constexpr int kRows = ROWS;
  constexpr int kSlots = TS::kSlots;
  constexpr int kAtomBytes = TS::kAtomBytes;
  constexpr int kSlotBytes = TS::kSlotBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  Misc* misc = reinterpret_cast<Misc*>(gbase + kMisc);
  int32_t* ids = reinterpret_cast<int32_t*>(gbase + kIds);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int split = blockIdx.y;  // rank in the cluster
  const int S = a.splits;
  const bool paired = S > 1;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&misc->kv_full[i], 32 * kLoadWarps);  // every loader thread, per tile
      mbar_init(&misc->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&misc->s_full[i], 1);
      mbar_init(&misc->s_free[i], 2);
      mbar_init(&misc->p_full[i], 2);
      mbar_init(&misc->p_empty[i], 1);
    }
    mbar_init(&misc->q_done, 1);    // the TMA loads of Q (expect-tx arrival + 64 KB)
    mbar_init(&misc->q_conv, 1);    // (fp8 cache) the math warps' conversion of Q
    mbar_init(&misc->ids_ready, 1);  // the math warps compacted the token ids
    mbar_init(&misc->o_done, 1);     // the PV issuer's last commit
    misc->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&misc->tmem_base, kTmemCols);
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  tc_fence_after();
  // The partner's barriers are initialised before any remote arrival: every
  // thread arrives here and waits before its first cluster access.
  if (paired) cluster_arrive_relaxed();

  // This query's visible latents and window rows.
  int n_vis, n_sw;
  const uint16_t* win;
  int64_t wrow0;  // row of the window buffer holding this query's first window row
  if (a.prefill) {
    int64_t P = query_pos(a.ctx, a.mq, a.n_tokens, b);
    if (P < 0) {
      // a multi-query sequence with fewer tokens than queries: this query has
      // no position, hence no rows
      if (tid == 0 && split == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, b);
      P = -1;
    }
    n_vis = static_cast<int>((P + 1) / a.ratio);
    const int64_t first = P - a.window + 1 > 0 ? P - a.window + 1 : 0;
    // the window buffer's row 0 holds position (first query's position) - window + 1
    const int64_t base_pos = (a.mq > 0 ? P - b % a.mq : a.ctx) - a.window + 1;
    wrow0 = static_cast<int64_t>(query_seq(a.mq, b)) * a.swa_seq_rows + (first - base_pos);
    win = a.swa + wrow0 * kLatent;
    n_sw = static_cast<int>(P - first + 1);
  } else {
    n_vis = a.n_latents[b];
    n_sw = a.swa_len[b];
    if (n_sw < 0 || n_sw > a.window) {
      if (tid == 0 && split == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, b);
      n_sw = n_sw < 0 ? 0 : a.window;
    }
    wrow0 = static_cast<int64_t>(b) * a.window;
    win = a.swa + wrow0 * kLatent;
  }
  if (n_vis > a.lat_stride) n_vis = static_cast<int>(a.lat_stride);
  // Latent rows: ids index this sequence's rows, or (paged) the compaction
  // below turns them into rows of the shared pool.
  const bool paged = a.pages.table != nullptr;
  const int lat_seq = a.prefill ? query_seq(a.mq, b) : (paged ? 0 : b);
  const int64_t lat_row0 = static_cast<int64_t>(lat_seq) * a.lat_stride;  // its first row
  // This CTA's rows: its part of the window rows first (they are inputs of the
  // step, so they stream while the previous kernel still selects the tokens),
  // then its part of the selected latents (known once the ids are compacted).
  const int w_part = (n_sw + S - 1) / S;
  const int w_begin = min(n_sw, split * w_part);
  const int w_cnt = min(n_sw, w_begin + w_part) - w_begin;
  auto sel_range = [&](int n_sel, int& s_begin, int& s_cnt) {
    const int h = (n_sel + S - 1) / S;
    s_begin = min(n_sel, split * h);
    s_cnt = min(n_sel, s_begin + h) - s_begin;
  };
  const uint32_t tmem = misc->tmem_base;
  // Cluster barrier phases of a split-KV CTA (every thread of the cluster
  // arrives at each):
  //   0 (arrived at start-up): every CTA's barriers are initialised;
  //   1: every CTA's MMAs are done and its payloads are staged, so rings may
  //      be written and payloads read;
  //   2: every CTA has received its payloads, so no copy reads or writes a
  //      CTA's memory any more (waited at exit).
  // The warps outside the exchange arrive at phase 2 at once.
  auto exchange_phases = [&]() {
    cluster_wait();
    cluster_arrive();
    cluster_wait();
    cluster_arrive();
  };

  if (warp == kLoadWarp0 && lane == 0) {
    // Q does not depend on the ids: eight boxes of 64 heads x 64 dims, each
    // landing as one 128-byte-swizzled atom of the QK^T A operand.
    tma_prefetch_map(&qmap);
    mbar_arrive_expect_tx(&misc->q_done, kQBytes);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      tma_load_2d(sbase + kQ + c * (kHeads * 128), &qmap, 64 * c, b * kHeads, &misc->q_done);
    }
  }

  // Compact the valid token ids (>= 0 and < n_vis) in order (math threads,
  // once the previous kernel's ids are final).
  if (tid < 128) {
    griddep_wait();
    const int32_t* tk = a.token_ids + static_cast<int64_t>(b) * a.k_tokens;
    constexpr int kPer = kMaxKTokens / 128;  // 4
    int my[kPer];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid * kPer + j;
      int id = -1;
      if (i < a.k_tokens) {
        id = tk[i];
        if (id >= n_vis) {
          if (split == 0) {
            record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, static_cast<uint32_t>(id));
          }
          id = -1;
        }
        if (paged && id >= 0) {
          const int64_t row = paged_row(a.pages, b, id);
          if (row < 0 && split == 0) {
            record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, static_cast<uint32_t>(id));
          }
          id = static_cast<int>(row);
        }
      }
      my[j] = id;
      cnt += id >= 0 ? 1 : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) misc->warp_cnt[warp] = incl;
    named_sync(kMathBar, 128);
    int before = incl - cnt;
    for (int w = 0; w < warp; ++w) before += misc->warp_cnt[w];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (my[j] >= 0) ids[before++] = my[j];
    }
    if (tid == 127) misc->n_sel = before;
    named_sync(kMathBar, 128);
    if (tid == 0) mbar_arrive(&misc->ids_ready);
    if constexpr (FP8) {
      // An fp8 cache's rows become f16 operands, so Q goes to f16 too, in
      // place, once the ids are out (the loaders start on the tiles
      // meanwhile; only the MMAs wait for it): thread t takes head
      // h = t / 2 in atoms 4 (t % 2) .. + 3 (the head's row of 8 chunks in
      // each), scales the head by 2^e_h so that its largest element lies in
      // [2^14, 2^15) (every bf16 element down to 2^-24 of it stays exact) and
      // records kv_scale * 2^-e_h for the softmax.
      wait_bar(&misc->q_done, 0u, misc, a.status);  // (a timeout is recorded)
      const int h = tid >> 1;
      const uint32_t qrow = sbase + kQ + static_cast<uint32_t>(4 * (tid & 1)) * (kHeads * 128) +
                            static_cast<uint32_t>(h) * 128;
      // chunk k of the thread's 32 (atom k / 8); the order within a row is
      // rotated by the head and the half so that the 8 lanes of a quarter
      // warp touch 8 different 16-byte bank groups
      auto qchunk = [&](int k) {
        return qrow + static_cast<uint32_t>(k >> 3) * (kHeads * 128) +
               static_cast<uint32_t>(((k & 7) + h + 4 * (tid & 1)) & 7) * 16;
      };
      float amax = 0.f;
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const uint4 v = ld_shared_v4(qchunk(k));
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(vw[i] & 0xFFFF)),
                                   fabsf(bf16_bits_to_float(vw[i] >> 16))));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      int e = 0;
      if (amax > 0.f) {
        const int E = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;
        e = min(126, max(-126, 14 - E));
      }
      const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const uint32_t addr = qchunk(k);
        const uint4 v = ld_shared_v4(addr);
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
        uint32_t hw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 x = __floats2half2_rn(bf16_bits_to_float(vw[i] & 0xFFFF) * up,
                                              bf16_bits_to_float(vw[i] >> 16) * up);
          hw[i] = *reinterpret_cast<const uint32_t*>(&x);
        }
        st_shared_v4(addr, make_uint4(hw[0], hw[1], hw[2], hw[3]));
      }
      if ((tid & 1) == 0) {
        misc->q_unscale[h] = a.kv_scale * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      }
      fence_proxy_async_smem();  // the MMA reads Q through the async proxy
      named_sync(kMathBar, 128);
      if (tid == 0) mbar_arrive(&misc->q_conv);
    }
  }

  // State the epilogue warps (math and loaders) share: the softmax statistics
  // of head tid (threads 0..63), whether every wait succeeded, and the tile count.
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  int n_tiles_e = 0;

  if (warp >= kLoadWarp0 && warp < kMmaWarp) {
    // ---------------- loaders ----------------
    // Loader warp w fills rows [kWarpRows w, kWarpRows (w + 1)) of every tile
    // t (ring slot t % kSlots): the four warps' copies of a tile are in
    // flight together, and each lane's completion arrives on the slot by
    // itself (rows without a source are zero-filled through the same path),
    // so no warp waits for its own copies. Tiles made only of window rows
    // need no ids: they load while the previous kernel still selects.
    constexpr int kWarpRows = kRows / kLoadWarps;
    const int w = warp - kLoadWarp0;
    bool have_ids = false;
    int s_begin = 0, n_rows_cta = w_cnt, n_tiles = 0;
    // An fp8 cache (32-row tiles: 8 rows a warp): lane l loads the codes
    // [8 l, 8 l + 8) and [256 + 8 l, 256 + 8 l + 8) of each of its warp's rows
    // into registers, and once the next tile's loads are out converts them to
    // f16 and stores chunks l and l + 32 of the rows, the places the bf16
    // copies fill (rows without a source: code 0, f16 zero). The load latency
    // of one tile so overlaps the previous tile's conversion.
    constexpr bool fp8 = FP8;
    static_assert(!FP8 || kRows == 32, "an fp8 cache takes 32-row tiles");
    const uint8_t* lat8 = reinterpret_cast<const uint8_t*>(a.latents);
    const uint8_t* swa8 = reinterpret_cast<const uint8_t*>(a.swa);
    // codes of even and of odd tiles (two register sets, so a tile's loads
    // are never waited on before the next tile's are out)
    uint2 alo[8], ahi[8], blo[8], bhi[8];
    const uint32_t dcol = static_cast<uint32_t>(lane >> 3) * kAtomBytes;
    auto fp8_load = [&](int r0t, int64_t arl, uint2 (&lo)[8], uint2 (&hi)[8]) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int64_t arow = __shfl_sync(0xFFFFFFFFu, arl, r);
        lo[r] = make_uint2(0u, 0u);
        hi[r] = make_uint2(0u, 0u);
        if (arow >= 0) {
          const uint8_t* src = (r0t + r < w_cnt ? swa8 : lat8) + arow * kLatent + lane * 8;
          lo[r] = __ldg(reinterpret_cast<const uint2*>(src));
          hi[r] = __ldg(reinterpret_cast<const uint2*>(src + 256));
        }
      }
    };
    auto fp8_store = [&](int tt, const uint2 (&clo)[8], const uint2 (&chi)[8]) -> bool {
      const int slt = tt % kSlots;
      if (tt >= kSlots &&
          !wait_bar(&misc->kv_empty[slt], static_cast<uint32_t>(((tt / kSlots) - 1) & 1), misc,
                    a.status)) {
        return false;
      }
      const uint32_t db = sbase + kKV + slt * kSlotBytes;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint32_t d0 = db + dcol + sw128_off(8 * w + r, lane & 7);
        st_shared_v4(d0, e4m3x8_to_f16(clo[r]));
        st_shared_v4(d0 + 4 * kAtomBytes, e4m3x8_to_f16(chi[r]));
      }
      fence_proxy_async_smem();  // the MMAs read the tile through the async proxy
      mbar_arrive(&misc->kv_full[slt]);
      return true;
    };
    for (int t = 0;; ++t) {
      const int g0 = t * kRows;
      if (!have_ids && g0 + kRows > w_cnt) {
        if (!wait_bar(&misc->ids_ready, 0u, misc, a.status)) {
          ok = false;
          break;
        }
        int s_cnt;
        sel_range(misc->n_sel, s_begin, s_cnt);
        n_rows_cta = w_cnt + s_cnt;
        n_tiles = (n_rows_cta + kRows - 1) / kRows;
        have_ids = true;
      }
      if (have_ids && t >= n_tiles) break;
      const int sl = t % kSlots;
      if (!fp8 && t >= kSlots &&
          !wait_bar(&misc->kv_empty[sl], static_cast<uint32_t>(((t / kSlots) - 1) & 1), misc,
                    a.status)) {
        ok = false;
        break;
      }
      const uint32_t dstb = sbase + kKV + sl * kSlotBytes;
      const int r0 = g0 + kWarpRows * w;  // this warp's first row of the tile
      // Lane l < kWarpRows works out the source of the warp's row l once (its
      // place in the window buffer or the latents; -1: none, zero-filled);
      // each row is then copied by the whole warp, lane l taking 16-byte
      // chunks l and l + 32, so a copy instruction covers 512 contiguous bytes.
      int64_t arow_l = -1;
      {
        const int gl = r0 + lane;
        if (lane < kWarpRows && gl < n_rows_cta) {
          arow_l = gl < w_cnt ? wrow0 + w_begin + gl : lat_row0 + ids[s_begin + gl - w_cnt];
          if (!DSA_DCHECK(arow_l >= 0 && arow_l < (gl < w_cnt ? a.swa_rows : a.lat_rows), a.status,
                          SITE_ATTN, arow_l)) {
            arow_l = -1;
          }
        }
      }
      // chunk lane of a row: atom lane / 8, 16-byte unit lane % 8 (dcol);
      // chunk lane + 32: atom 4 + lane / 8, same unit
      if constexpr (fp8) {
        bool st_ok = true;
        if ((t & 1) == 0) {
          fp8_load(r0, arow_l, alo, ahi);
          if (t > 0) st_ok = fp8_store(t - 1, blo, bhi);
        } else {
          fp8_load(r0, arow_l, blo, bhi);
          st_ok = fp8_store(t - 1, alo, ahi);
        }
        if (!st_ok) {
          ok = false;
          break;
        }
      } else {
#pragma unroll 4
        for (int r = 0; r < kWarpRows; ++r) {
          const int64_t arow = __shfl_sync(0xFFFFFFFFu, arow_l, r);
          const int row = kWarpRows * w + r;
          const uint32_t d0 = dstb + dcol + sw128_off(row, lane & 7);
          const uint32_t d1 = d0 + 4 * kAtomBytes;
          if (arow >= 0) {
            const uint16_t* src = (r0 + r < w_cnt ? a.swa : a.latents) + arow * kLatent + lane * 8;
            cp_async_16(d0, src);
            cp_async_16(d1, src + 256);
          } else {
            cp_async_16_zero(d0, a.latents);
            cp_async_16_zero(d1, a.latents);
          }
        }
        cp_async_mbar_arrive_noinc(&misc->kv_full[sl]);
      }
    }
    // (fp8) the last tile loaded
    if constexpr (fp8) {
      if (ok && have_ids && n_tiles > 0) {
        if (!((n_tiles - 1) & 1 ? fp8_store(n_tiles - 1, blo, bhi)
                                : fp8_store(n_tiles - 1, alo, ahi))) {
          ok = false;
        }
      }
    }
    n_tiles_e = have_ids ? n_tiles : 0;
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ---------------- MMA issuers ----------------
    int n_tiles = 0;
    if (lane == 0 && wait_bar(&misc->ids_ready, 0u, misc, a.status)) {
      int s_begin, s_cnt;
      sel_range(misc->n_sel, s_begin, s_cnt);
      n_tiles = (w_cnt + s_cnt + kRows - 1) / kRows;
    }
    // PV(t) is issued only after the softmax of tile t, hence after QK^T(t)
    // completed: its commit alone frees the tile's slot, and the PV issuer's
    // last commit means every MMA of the CTA has completed.
    if (lane == 0 && warp == kPvWarp) {
      // f16 operands with an fp8 cache, bf16 otherwise
      constexpr uint32_t idesc_o = mma_idesc(128, kHeads, !FP8, true, false);
      for (int t = 0; t < n_tiles; ++t) {
        const int sb = t & 1;
        if (!wait_bar(&misc->p_full[sb], static_cast<uint32_t>((t >> 1) & 1), misc, a.status)) {
          break;
        }
        tc_fence_after();
        fence_proxy_async_smem();
        // Descriptors are built once and stepped by their start-address field
        // (16-byte units; every operand lies below 256 KB, so no carry).
        const uint64_t ad0 =
            sw128_desc(sbase + kKV + (t % kSlots) * kSlotBytes, kAtomBytes, 1024);
        const uint64_t bd0 = sw128_desc(sbase + kP + sb * kPBytes, 16, 1024);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks) {
            const uint64_t ad = ad0 + ((m * 2 * kAtomBytes + ks * 16 * 128) >> 4);
            const uint64_t bd = bd0 + ((ks * 32) >> 4);
            mma_f16(tmem + 128 + 64 * m, ad, bd, idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
          }
        }
        mma_commit(&misc->kv_empty[t % kSlots]);
        mma_commit(&misc->p_empty[sb]);
      }
      if (n_tiles > 0) mma_commit(&misc->o_done);  // arrives once every MMA has completed
    }
    if (lane == 0 && warp == kMmaWarp) {
      constexpr uint32_t idesc_s = mma_idesc(128, kRows, !FP8, false, false);
      // Q as loaded, or (fp8 cache) once the math warps have taken it to f16
      bool ok = n_tiles == 0 ||
                wait_bar(FP8 ? &misc->q_conv : &misc->q_done, 0u, misc, a.status);
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int slot = t % kSlots, sb = t & 1;
        if (!wait_bar(&misc->kv_full[slot], static_cast<uint32_t>((t / kSlots) & 1), misc,
                      a.status)) {
          ok = false;
          break;
        }
        if (t >= 2 && !wait_bar(&misc->s_free[sb], static_cast<uint32_t>(((t >> 1) - 1) & 1),
                                misc, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        fence_proxy_async_smem();
        const uint64_t ad0 = sw128_desc(sbase + kQ, 16, 1024);
        const uint64_t bd0 = sw128_desc(sbase + kKV + slot * kSlotBytes, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < kLatent / 16; ++ks) {
          const uint64_t ad = ad0 + (((ks >> 2) * (kHeads * 128) + (ks & 3) * 32) >> 4);
          const uint64_t bd = bd0 + (((ks >> 2) * kAtomBytes + (ks & 3) * 32) >> 4);
          mma_f16(tmem + 64 * sb, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&misc->s_full[sb]);
      }
    }
    __syncwarp();
    if (paired) exchange_phases();
  } else {
    // ---------------- math: softmax, rescale ----------------
    int s_begin, s_cnt;
    sel_range(misc->n_sel, s_begin, s_cnt);
    const int n_rows_cta = w_cnt + s_cnt;
    const int n_tiles = (n_rows_cta + kRows - 1) / kRows;
    // A failed (timed-out) wait makes `ok` false for good; the thread then
    // skips the work but still reaches every named barrier, so the math warps
    // never part ways at a barrier.
    n_tiles_e = n_tiles;
    const uint32_t la = tmem_addr(tmem, static_cast<uint32_t>(32 * warp), 0);
    // the softmax constant of this thread's head (fp8 cache: the head's Q
    // scale undone and the cache scale applied)
    const float sl = FP8 ? a.scale_log2 * misc->q_unscale[tid & (kHeads - 1)] : a.scale_log2;
    // PV(j) is known complete through p_empty[j & 1], whose phases a thread
    // consumes in order (at most one phase ahead of its last wait), so a
    // parity wait is never more than one phase off; waiting on PV(j) early (to
    // rescale) and again later (to reuse the buffer) both read the right phase.
    auto wait_pv = [&](int j) {
      if (ok) {
        ok = wait_bar(&misc->p_empty[j & 1], static_cast<uint32_t>((j >> 1) & 1), misc, a.status);
      }
    };
    for (int t = 0; t < n_tiles; ++t) {
      const int sb = t & 1;
      const int valid = min(kRows, n_rows_cta - t * kRows);
      float z[kRows];
      float alpha = 1.f;
      bool resc = false;
      if (warp < 2) {
        if (ok) ok = wait_bar(&misc->s_full[sb], static_cast<uint32_t>((t >> 1) & 1), misc, a.status);
        tc_fence_after();
        if (ok) {
          load_scores<kRows>(la + 64 * sb, valid, z);
          const float mt = max_scores<kRows>(z, sl);
          if (t == 0) {
            m_run = mt;
          } else if (mt > m_run + 8.f) {
            alpha = exp2f(m_run - mt);
            m_run = mt;
            resc = true;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&misc->s_free[sb]);
        misc->alpha[tid] = alpha;
      }
      // O^T holds PV(0..t-1); if any head's maximum moved, scale every head's
      // column by its alpha (alpha = 1 for heads whose maximum stayed).
      const bool any_resc = named_sync_or(kMathBar, 128, resc);
      if (any_resc) {
        if (t > 0) wait_pv(t - 1);
        tc_fence_after();
        if (ok && t > 0) {
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float v[16];
              const uint32_t addr = la + 128 + 64 * m + 16 * c;
              tmem_ld16(addr, v);
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] *= misc->alpha[16 * c + i];
              tmem_st16(addr, v);
            }
          }
        }
        tc_fence_before();
        named_sync(kMathBar, 128);  // alpha is read by all before the next tile rewrites it
      }
      if (warp < 2) {
        // P[sb] was last read by PV(t - 2)
        if (t >= 2) wait_pv(t - 2);
        if (ok) {
          uint32_t pk[kRows / 2];
          // the denominator sums the fp32 probabilities
          l_run = l_run * alpha + exp_pack<kRows, FP8>(z, sl, m_run, pk);
          const uint32_t pb = sbase + kP + sb * kPBytes;
#pragma unroll
          for (int c = 0; c < kRows / 8; ++c) {
            st_shared_v4(pb + sw128_off(tid, c),
                         make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&misc->p_full[sb]);
      }
    }
  }

  if (warp < kMmaWarp) {
    // ---------------- epilogue (math and loader warps) ----------------
    // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (dims 128 m + 32 (w % 4) + lane of O^T
    // slice m) and heads [32 (w / 4), 32 (w / 4) + 32): the math warps take heads
    // 0..31, the loader warps (idle by now) heads 32..63, so eight warps share the
    // work that runs once per CTA.
    const int half = warp >> 2;
    const int et = 32 * (warp & 3) + lane;  // dim within a slice = TMEM lane
    const uint32_t lq = tmem_addr(tmem, static_cast<uint32_t>(32 * (warp & 3)), 0);
    const int n_tiles = n_tiles_e;
    // Once the PV issuer's last commit has arrived, every MMA has completed:
    // Q, P and the ring are free.
    if (n_tiles > 0) {
      if (ok) ok = wait_bar(&misc->o_done, 0u, misc, a.status);
    } else if (ok) {
      // no tiles: nothing ordered the Q copies before the staging writes below
      ok = wait_bar(&misc->q_done, 0u, misc, a.status);
    }
    tc_fence_after();
    const bool have_o = ok && n_tiles > 0;
    uint16_t* out = a.out + static_cast<int64_t>(b) * kHeads * kLatent;
    // Heads [16 hc, 16 hc + 16) of O^T slice m (dim 128 m + et in this
    // thread's lane), zeros without rows.
    auto load16 = [&](int m, int hc, float (&v)[16]) {
      if (have_o) {
        tmem_ld16(lq + 128 + 64 * m + 16 * hc, v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
    };
    // v[i] *= f[16 hc + i], f in shared memory
    auto scale16 = [&](float (&v)[16], uint32_t f, int hc) {
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 w4 = ld_shared_f4(f + (16 * hc + i) * 4);
        v[i] *= w4.x;
        v[i + 1] *= w4.y;
        v[i + 2] *= w4.z;
        v[i + 3] *= w4.w;
      }
    };
    // out[16 hc + i][d] = v[i]: each store instruction of a warp writes 32
    // consecutive dims of one head.
    auto store16 = [&](int d, int hc, const float (&v)[16]) {
      uint16_t* o = out + static_cast<int64_t>(16 * hc) * kLatent + d;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[static_cast<int64_t>(i) * kLatent] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
      }
    };
    const uint32_t inv_l_s = smem_u32(misc->inv_l);
    if (!paired) {
      if (warp < 2) {
        // (an fp8 cache's rows are code * kv_scale: O carries the scale)
        misc->inv_l[tid] = l_run > 0.f ? (FP8 ? a.kv_scale : 1.f) / l_run : 0.f;
        if (a.lse) {
          a.lse[static_cast<int64_t>(b) * kHeads + tid] =
              l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        }
      }
      named_sync(kEpiBar, kEpiThreads);
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
#pragma unroll 1
        for (int hc = 2 * half; hc < 2 * half + 2; ++hc) {
          float v[16];
          load16(m, hc, v);
          scale16(v, inv_l_s, hc);
          store16(128 * m + et, hc, v);
        }
      }
    } else {
      // CTA `split` finishes latent dims [split D, split D + D). O^T slice m
      // holds dim 128 m + et in this thread's lane, so the thread's four dims
      // go to CTAs (128 m + et) / D (a warp's 32 dims always go to one CTA).
      // Each CTA writes, straight into each peer's receive area (its ring, free
      // once the peer's MMAs are done), its unnormalised O for the peer's dims
      // in bf16 and its (max, sum) per head; its own (max, sum) go to its own
      // area, so the merge reads every CTA's the same way.
      const int D = kLatent / S;
      const uint32_t pay = static_cast<uint32_t>(xchg_bytes(S));
      const float m_own = have_o ? m_run : -INFINITY, l_own = have_o ? l_run : 0.f;
      auto recv_slot = [&](int q) -> uint32_t {  // payload from CTA q, in this CTA
        return sbase + kRecv + static_cast<uint32_t>(q) * pay;
      };
      cluster_wait();  // phase 0
      if (warp < 2) {
        float* t = reinterpret_cast<float*>(gbase + (recv_slot(split) - sbase) + D * 128);
        t[2 * tid] = m_own;
        t[2 * tid + 1] = l_own;
      }
      cluster_arrive();  // phase 1: every CTA's MMAs are done, so its ring may be written
      cluster_wait();
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + et;
        const int p = d / D;
        if (p == split) continue;
        const int dd = d - p * D;
        const uint32_t row =
            mapa_shared(recv_slot(split) + static_cast<uint32_t>(dd) * 128, static_cast<uint32_t>(p));
#pragma unroll 1
        for (int hc = 2 * half; hc < 2 * half + 2; ++hc) {
          float v[16];
          load16(m, hc, v);
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __nv_bfloat162 x = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            w8[e] = *reinterpret_cast<const uint32_t*>(&x);
          }
          st_cluster_u4(row + static_cast<uint32_t>((2 * hc) ^ (dd & 7)) * 16,
                        make_uint4(w8[0], w8[1], w8[2], w8[3]));
          st_cluster_u4(row + static_cast<uint32_t>((2 * hc + 1) ^ (dd & 7)) * 16,
                        make_uint4(w8[4], w8[5], w8[6], w8[7]));
        }
      }
      if (warp < 2) {
        for (int p = 0; p < S; ++p) {
          if (p == split) continue;
          st_cluster_f32x2(mapa_shared(recv_slot(split) + D * 128 + 8 * tid, static_cast<uint32_t>(p)),
                           m_own, l_own);
        }
      }
      cluster_arrive();  // phase 2: every payload is written (release) ...
      cluster_wait();    // ... and visible here (acquire)
      // out = sum_q w_q O_q with w_q = 2^(m_q - M) / L, M = max_q m_q,
      // L = sum_q 2^(m_q - M) l_q (a range without rows has l_q = 0), O_q the
      // unnormalised accumulator of CTA q.
      float* wgt = reinterpret_cast<float*>(gbase + kWgt);  // [S][64]
      if (warp < 2) {
        // Rolled loops over the S senders: this code runs once per CTA and is
        // fetched cold, so its size costs more than its work.
        auto ml = [&](int q) {  // sender q's (max, sum) of head tid
          return reinterpret_cast<const float2*>(gbase + (recv_slot(q) - sbase) + D * 128)[tid];
        };
        float M = -INFINITY;
#pragma unroll 1
        for (int q = 0; q < S; ++q) {
          const float2 x = ml(q);
          if (x.y > 0.f) M = fmaxf(M, x.x);
        }
        float L = 0.f;
#pragma unroll 1
        for (int q = 0; q < S; ++q) {
          const float2 x = ml(q);
          const float e = x.y > 0.f ? exp2f(x.x - M) : 0.f;
          wgt[q * kHeads + tid] = e;
          L = fmaf(e, x.y, L);
        }
        // (an fp8 cache's rows are code * kv_scale: O carries the scale)
        const float inv_L = L > 0.f ? (FP8 ? a.kv_scale : 1.f) / L : 0.f;
#pragma unroll 1
        for (int q = 0; q < S; ++q) wgt[q * kHeads + tid] *= inv_L;
        if (a.lse && split == 0) {
          a.lse[static_cast<int64_t>(b) * kHeads + tid] =
              L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
      }
      named_sync(kEpiBar, kEpiThreads);
      const uint32_t wgt_s = sbase + kWgt;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + et;
        if (d / D != split) continue;
        const int dd = d - split * D;
#pragma unroll 1
        for (int hc = 2 * half; hc < 2 * half + 2; ++hc) {
          float v[16];
          load16(m, hc, v);
          scale16(v, wgt_s + static_cast<uint32_t>(split * kHeads * 4), hc);
#pragma unroll 1
          for (int q = 0; q < S; ++q) {
            if (q == split) continue;
            const uint32_t row = recv_slot(q) + static_cast<uint32_t>(dd) * 128;
            const uint4 x0 = ld_shared_v4(row + static_cast<uint32_t>((2 * hc) ^ (dd & 7)) * 16);
            const uint4 x1 =
                ld_shared_v4(row + static_cast<uint32_t>((2 * hc + 1) ^ (dd & 7)) * 16);
            const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t wq = wgt_s + static_cast<uint32_t>(q * kHeads * 4);
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 w4 = ld_shared_f4(wq + (16 * hc + i) * 4);
              v[i] = fmaf(w4.x, bf16_bits_to_float(xs[i / 2] & 0xFFFF), v[i]);
              v[i + 1] = fmaf(w4.y, bf16_bits_to_float(xs[i / 2] >> 16), v[i + 1]);
              v[i + 2] = fmaf(w4.z, bf16_bits_to_float(xs[i / 2 + 1] & 0xFFFF), v[i + 2]);
              v[i + 3] = fmaf(w4.w, bf16_bits_to_float(xs[i / 2 + 1] >> 16), v[i + 3]);
            }
          }
          store16(d, hc, v);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // The epilogue warps have waited for phase 2 (no peer writes this CTA any
  // more); the MMA warps, which only arrived there, wait now.
  if (paired && warp >= kMmaWarp) cluster_wait();
}

// ---------------------------------------------------------------------------
// Unsplit attention (one CTA per query: prefill chunks, multi-query batches,
// decode batches too large to split), persistent: grid = min(queries, SMs),
// CTA c takes queries c, c + grid, ... and runs them through one pipeline, so
// the next query's index list, Q and first tiles load while the current
// query's last tiles and its epilogue run. The roles are those of attn_kernel
// (4 math warps, 4 loaders, QK^T and PV issuers); barrier phases follow a
// per-CTA count of tiles across the CTA's queries (tile g: ring slot g mod
// kSlots, S and P buffer g & 1).
//   * index lists: double-buffered; the math warps compact query i + 1's
//     right after their last softmax of query i, before its epilogue;
//   * Q: the QK^T issuer loads query i + 1's Q once query i's last QK^T has
//     completed (q_free);
//   * O^T: the math warps' epilogue of query i reads it before their first
//     softmax of query i + 1, which precedes PV(i + 1, 0) (the only MMA that
//     overwrites it), so no extra barrier is needed; the epilogue runs on the
//     math warps alone while the loaders stream the next query.
// ---------------------------------------------------------------------------
constexpr int kIdsB = kMisc + kMiscBytes;  // second index-list buffer
constexpr int kSmemStream = kIdsB + kMaxKTokens * 4 + 1024;

struct MiscS {
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots], s_full[2], s_free[2], p_full[2], p_empty[2];
  uint64_t q_done, q_free, o_done;
  uint32_t tmem_base;
  int abort;
  // Per-query hand-offs are counters, not barrier phases: a query without rows
  // lets a role run ahead by more than one phase.
  int ids_seq;  // queries whose index lists are compacted (loader warps)
  int ld_seq;   // queries finished by loader warps (one count per warp)
  int math_seq; // queries whose tile count the math warps have read
  int mma_seq;  // queries whose tile count the QK^T issuer has read
  int pv_seq;   // queries whose tile count the PV issuer has read
  int epi_seq;  // queries whose epilogue is done (math warps)
  int n_sel[2];
  int warp_cnt[4];
  alignas(16) float alpha[kHeads];
  alignas(16) float inv_l[kHeads];
};
static_assert(sizeof(MiscS) <= kMiscBytes, "misc block");
static_assert(offsetof(MiscS, inv_l) % 16 == 0, "16-byte loads of inv_l");

__device__ __forceinline__ bool wait_bar_s(uint64_t* bar, uint32_t parity, MiscS* m,
                                           DeviceStatus* st) {
  return mbar_wait_abortable(bar, parity, &m->abort, st, SITE_ATTN);
}

// A query's rows in the window buffer and the latents (unsplit).
struct QueryRows {
  int n_vis;      // visible latents (ids must be below)
  int n_sw;       // window rows
  int64_t wrow0;  // row of the window buffer holding its first window row
  int64_t lat_row0;  // first row of its sequence's latents (0 when paged)
};

__device__ __forceinline__ QueryRows query_rows(const AttnArgs& a, int b, bool report) {
  QueryRows r;
  if (a.prefill) {
    int64_t P = query_pos(a.ctx, a.mq, a.n_tokens, b);
    if (P < 0) {
      // a multi-query sequence with fewer tokens than queries: no rows
      if (report) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, b);
      P = -1;
    }
    r.n_vis = static_cast<int>((P + 1) / a.ratio);
    const int64_t first = P - a.window + 1 > 0 ? P - a.window + 1 : 0;
    // the window buffer's row 0 holds position (first query's position) - window + 1
    const int64_t base_pos = (a.mq > 0 ? P - b % a.mq : a.ctx) - a.window + 1;
    r.wrow0 = static_cast<int64_t>(query_seq(a.mq, b)) * a.swa_seq_rows + (first - base_pos);
    r.n_sw = static_cast<int>(P - first + 1);
  } else {
    r.n_vis = a.n_latents[b];
    r.n_sw = a.swa_len[b];
    if (r.n_sw < 0 || r.n_sw > a.window) {
      if (report) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, b);
      r.n_sw = r.n_sw < 0 ? 0 : a.window;
    }
    r.wrow0 = static_cast<int64_t>(b) * a.window;
  }
  if (r.n_vis > a.lat_stride) r.n_vis = static_cast<int>(a.lat_stride);
  const bool paged = a.pages.table != nullptr;
  const int lat_seq = a.prefill ? query_seq(a.mq, b) : (paged ? 0 : b);
  r.lat_row0 = static_cast<int64_t>(lat_seq) * a.lat_stride;
  return r;
}

// Bounded wait (all threads that call it) until *p >= v, a counter in shared
// memory that another role raises; false once it times out or the CTA aborts.
__device__ __forceinline__ bool wait_count(int* p, int v, MiscS* m, DeviceStatus* st) {
  volatile int* vp = p;
  if (*vp >= v) {
    __threadfence_block();
    return true;
  }
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (*vp >= v) {
      __threadfence_block();
      return true;
    }
    if ((it & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(&m->abort)) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        record_status(st, DSA_ERR_TIMEOUT, SITE_ATTN, smem_u32(p));
        m->abort = 1;
        return false;
      }
    }
    __nanosleep(64);
  }
}
// Raises a counter after this thread's earlier shared-memory writes.
__device__ __forceinline__ void raise_count(int* p, int v) {
  __threadfence_block();
  *reinterpret_cast<volatile int*>(p) = v;
}

template <int ROWS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_stream_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap) {
  using TS = TileShape<ROWS>;
  constexpr int kRows = ROWS;
  constexpr int kSlots = TS::kSlots;
  constexpr int kAtomBytes = TS::kAtomBytes;
  constexpr int kSlotBytes = TS::kSlotBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  MiscS* misc = reinterpret_cast<MiscS*>(gbase + kMisc);
  // index-list buffer of query index qi
  auto ids_buf = [&](int qi) -> int32_t* {
    return reinterpret_cast<int32_t*>(gbase + ((qi & 1) ? kIdsB : kIds));
  };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b0 = blockIdx.x, gstep = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&misc->kv_full[i], 32 * kLoadWarps);  // every loader thread, per tile
      mbar_init(&misc->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&misc->s_full[i], 1);
      mbar_init(&misc->s_free[i], 2);
      mbar_init(&misc->p_full[i], 2);
      mbar_init(&misc->p_empty[i], 1);
    }
    mbar_init(&misc->q_done, 1);  // a query's Q: expect-tx arrival + 64 KB
    mbar_init(&misc->q_free, 1);  // a query's QK^Ts have completed
    mbar_init(&misc->o_done, 1);  // a query's PVs have completed
    misc->abort = 0;
    misc->ids_seq = misc->ld_seq = misc->mma_seq = misc->pv_seq = misc->epi_seq = 0;
    misc->math_seq = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&misc->tmem_base, kTmemCols);
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  // Tile count of query index qi (its lists compacted): window rows + ids.
  auto tiles_of = [&](int b, int qi) -> int {
    const QueryRows qr = query_rows(a, b, false);
    return (qr.n_sw + misc->n_sel[qi & 1] + kRows - 1) / kRows;
  };

  // Compacts query index qi's valid token ids (>= 0 and < n_vis; pool rows
  // when the latents are paged) in order into buffer qi & 1: the loader
  // warps' work (thread ct of 128, warp cw of 4, named barrier kLoadBar),
  // done for the next query as soon as a query's tiles are out, so that no
  // role waits for ids at a query switch.
  auto compact = [&](int b, int qi, bool& ok) {
    const int ct = tid - 32 * kLoadWarp0, cw = warp - kLoadWarp0;
    if (qi >= 2) {
      // every other role is done with query qi - 2, whose buffer this reuses
      if (ct == 0 && ok) {
        ok = wait_count(&misc->ld_seq, kLoadWarps * (qi - 1), misc, a.status) &&
             wait_count(&misc->mma_seq, qi - 1, misc, a.status) &&
             wait_count(&misc->pv_seq, qi - 1, misc, a.status) &&
             wait_count(&misc->math_seq, qi - 1, misc, a.status);
      }
      named_sync(kLoadBar, 32 * kLoadWarps);
    }
    const QueryRows qr = query_rows(a, b, ct == 0);
    const int32_t* tk = a.token_ids + static_cast<int64_t>(b) * a.k_tokens;
    int32_t* ids = ids_buf(qi);
    constexpr int kPer = kMaxKTokens / 128;  // 4
    int my[kPer];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = ct * kPer + j;
      int id = -1;
      if (i < a.k_tokens) {
        id = tk[i];
        if (id >= qr.n_vis) {
          record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, static_cast<uint32_t>(id));
          id = -1;
        }
        if (a.pages.table != nullptr && id >= 0) {
          const int64_t row = paged_row(a.pages, b, id);
          if (row < 0) {
            record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, static_cast<uint32_t>(id));
          }
          id = static_cast<int>(row);
        }
      }
      my[j] = id;
      cnt += id >= 0 ? 1 : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) misc->warp_cnt[cw] = incl;
    named_sync(kLoadBar, 32 * kLoadWarps);
    int before = incl - cnt;
    for (int w = 0; w < cw; ++w) before += misc->warp_cnt[w];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (my[j] >= 0) ids[before++] = my[j];
    }
    if (ct == 127) misc->n_sel[qi & 1] = before;
    named_sync(kLoadBar, 32 * kLoadWarps);
    if (ct == 0) raise_count(&misc->ids_seq, qi + 1);
  };

  if (warp < kLoadWarp0) {
    // ---------------- math: index lists, softmax, epilogue ----------------
    griddep_wait();  // the previous kernel's token ids are final
    const uint32_t la = tmem_addr(tmem, static_cast<uint32_t>(32 * warp), 0);
    bool ok = true;
    int64_t gq = 0;  // this CTA's tile count before the current query
    int qi = 0;
    for (int b = b0; b < a.B; b += gstep, ++qi) {
      if (tid == 0 && ok) ok = wait_count(&misc->ids_seq, qi + 1, misc, a.status);
      named_sync(kMathBar, 128);
      const QueryRows qr = query_rows(a, b, false);
      const int n_rows = qr.n_sw + misc->n_sel[qi & 1];
      const int n_tiles = (n_rows + kRows - 1) / kRows;
      named_sync(kMathBar, 128);  // every math thread has read the tile count
      if (tid == 0) raise_count(&misc->math_seq, qi + 1);
      float m_run = -INFINITY, l_run = 0.f;  // threads 0..63: head tid
      // PV(j) is known complete through p_empty[j & 1]; the next phase of that
      // barrier needs P(j + 2), written after every wait below, so a parity
      // wait is never more than one phase off.
      auto wait_pv = [&](int64_t j) {
        if (ok) {
          ok = wait_bar_s(&misc->p_empty[j & 1], static_cast<uint32_t>((j >> 1) & 1), misc,
                          a.status);
        }
      };
      for (int t = 0; t < n_tiles; ++t) {
        const int64_t g = gq + t;
        const int sb = static_cast<int>(g & 1);
        const int valid = min(kRows, n_rows - t * kRows);
        float z[kRows];
        float alpha = 1.f;
        bool resc = false;
        if (warp < 2) {
          if (ok) {
            ok = wait_bar_s(&misc->s_full[sb], static_cast<uint32_t>((g >> 1) & 1), misc, a.status);
          }
          tc_fence_after();
          if (ok) {
            load_scores<kRows>(la + 64 * sb, valid, z);
            const float mt = max_scores<kRows>(z, a.scale_log2);
            if (t == 0) {
              m_run = mt;
            } else if (mt > m_run + 8.f) {
              alpha = exp2f(m_run - mt);
              m_run = mt;
              resc = true;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&misc->s_free[sb]);
          misc->alpha[tid] = alpha;
        }
        // O^T holds this query's PV(0..t-1); if any head's maximum moved,
        // scale every head's column by its alpha.
        const bool any_resc = named_sync_or(kMathBar, 128, resc);
        if (any_resc) {
          if (t > 0) wait_pv(g - 1);
          tc_fence_after();
          if (ok && t > 0) {
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                float v[16];
                const uint32_t addr = la + 128 + 64 * m + 16 * c;
                tmem_ld16(addr, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= misc->alpha[16 * c + i];
                tmem_st16(addr, v);
              }
            }
          }
          tc_fence_before();
          named_sync(kMathBar, 128);  // alpha is read by all before the next tile rewrites it
        }
        if (warp < 2) {
          // P[sb] was last read by PV(g - 2), of this query or the previous one
          if (g >= 2) wait_pv(g - 2);
          if (ok) {
            uint32_t pk[kRows / 2];
            // the denominator sums the fp32 probabilities
            l_run = l_run * alpha + exp_pack<kRows>(z, a.scale_log2, m_run, pk);
            const uint32_t pb = sbase + kP + sb * kPBytes;
#pragma unroll
            for (int c = 0; c < kRows / 8; ++c) {
              st_shared_v4(pb + sw128_off(tid, c),
                           make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&misc->p_full[sb]);
        }
      }
      // ---------------- epilogue (math warps) ----------------
      if (ok) ok = wait_bar_s(&misc->o_done, static_cast<uint32_t>(qi & 1), misc, a.status);
      tc_fence_after();
      const bool have_o = ok && n_tiles > 0;
      uint16_t* out = a.out + static_cast<int64_t>(b) * kHeads * kLatent;
      if (warp < 2) {
        misc->inv_l[tid] = have_o && l_run > 0.f ? 1.f / l_run : 0.f;
        if (a.lse) {
          a.lse[static_cast<int64_t>(b) * kHeads + tid] =
              have_o && l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        }
      }
      named_sync(kMathBar, 128);
      const uint32_t inv_l_s = smem_u32(misc->inv_l);
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
#pragma unroll 1
        for (int hc = 0; hc < 4; ++hc) {
          float v[16];
          if (have_o) {
            tmem_ld16(la + 128 + 64 * m + 16 * hc, v);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 w4 = ld_shared_f4(inv_l_s + (16 * hc + i) * 4);
            v[i] *= w4.x;
            v[i + 1] *= w4.y;
            v[i + 2] *= w4.z;
            v[i + 3] *= w4.w;
          }
          uint16_t* o = out + static_cast<int64_t>(16 * hc) * kLatent + 128 * m + tid;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            o[static_cast<int64_t>(i) * kLatent] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
          }
        }
      }
      tc_fence_before();
      named_sync(kMathBar, 128);  // every read of O^T is done
      if (tid == 0) raise_count(&misc->epi_seq, qi + 1);
      gq += n_tiles;
    }
  }
  else if (warp < kMmaWarp) {
    // ---------------- loaders ----------------
    // Loader warp w fills rows [kWarpRows w, kWarpRows (w + 1)) of every tile
    // g = 0, 1, ... of the CTA's queries (ring slot g % kSlots): the four
    // warps' copies of a tile are in flight together, and each lane's
    // completion arrives on the slot by itself (rows without a source are
    // zero-filled through the same path), so no warp waits for its own
    // copies: it goes on to the next tile once that tile's slot is free.
    constexpr int kWarpRows = kRows / kLoadWarps;
    const int w = warp - kLoadWarp0;
    bool ok = true;
    griddep_wait();  // the previous kernel's token ids are final
    if (b0 < a.B) compact(b0, 0, ok);
    int64_t gq = 0;
    int qi = 0;
    // Every loader warp goes through every query (and every compaction's
    // barriers), also after a failed wait, which only skips its copies.
    for (int b = b0; b < a.B; b += gstep, ++qi) {
      const QueryRows qr = query_rows(a, b, false);
      const int32_t* ids = ids_buf(qi);
      const int w_cnt = qr.n_sw;
      const int n_rows = w_cnt + misc->n_sel[qi & 1];
      const int n_tiles = (n_rows + kRows - 1) / kRows;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int64_t g = gq + t;
        const int sl = static_cast<int>(g % kSlots);
        const uint32_t u = static_cast<uint32_t>(g / kSlots);
        if (g >= kSlots &&
            !wait_bar_s(&misc->kv_empty[sl], (u - 1) & 1u, misc, a.status)) {
          ok = false;
          break;
        }
        const uint32_t dstb = sbase + kKV + sl * kSlotBytes;
        const int r0 = t * kRows + kWarpRows * w;  // this warp's first row of the tile
        // Lane l < kWarpRows works out the source of the warp's row l once
        // (-1: none, zero-filled); each row is then copied by the whole warp,
        // lane l taking 16-byte chunks l and l + 32.
        int64_t arow_l = -1;
        {
          const int gl = r0 + lane;
          if (lane < kWarpRows && gl < n_rows) {
            arow_l = gl < w_cnt ? qr.wrow0 + gl : qr.lat_row0 + ids[gl - w_cnt];
            if (!DSA_DCHECK(arow_l >= 0 && arow_l < (gl < w_cnt ? a.swa_rows : a.lat_rows),
                            a.status, SITE_ATTN, arow_l)) {
              arow_l = -1;
            }
          }
        }
        const uint32_t dcol = static_cast<uint32_t>(lane >> 3) * kAtomBytes;
#pragma unroll 4
        for (int r = 0; r < kWarpRows; ++r) {
          const int64_t arow = __shfl_sync(0xFFFFFFFFu, arow_l, r);
          const int row = kWarpRows * w + r;
          const uint32_t d0 = dstb + dcol + sw128_off(row, lane & 7);
          const uint32_t d1 = d0 + 4 * kAtomBytes;
          if (arow >= 0) {
            const uint16_t* src = (r0 + r < w_cnt ? a.swa : a.latents) + arow * kLatent + lane * 8;
            cp_async_16(d0, src);
            cp_async_16(d1, src + 256);
          } else {
            cp_async_16_zero(d0, a.latents);
            cp_async_16_zero(d1, a.latents);
          }
        }
        cp_async_mbar_arrive_noinc(&misc->kv_full[sl]);
      }
      __syncwarp();
      if (ok && lane == 0) {
        __threadfence_block();
        atomicAdd(&misc->ld_seq, 1);  // this warp no longer reads query qi's list
      }
      gq += n_tiles;
      // the next query's list, while this query's last tiles are computed
      if (b + gstep < a.B) compact(b + gstep, qi + 1, ok);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- QK^T issuer (and Q loads) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = mma_idesc(128, kRows, true, false, false);
      auto load_q = [&](int b) {
        mbar_arrive_expect_tx(&misc->q_done, kQBytes);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          tma_load_2d(sbase + kQ + c * (kHeads * 128), &qmap, 64 * c, b * kHeads, &misc->q_done);
        }
      };
      tma_prefetch_map(&qmap);
      if (b0 < a.B) load_q(b0);
      bool ok = true;
      int64_t gq = 0;
      int qi = 0;
      for (int b = b0; b < a.B && ok; b += gstep, ++qi) {
        if (!wait_count(&misc->ids_seq, qi + 1, misc, a.status)) break;
        const int n_tiles = tiles_of(b, qi);
        raise_count(&misc->mma_seq, qi + 1);
        ok = wait_bar_s(&misc->q_done, static_cast<uint32_t>(qi & 1), misc, a.status);
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int64_t g = gq + t;
          const int slot = static_cast<int>(g % kSlots), sb = static_cast<int>(g & 1);
          if (!wait_bar_s(&misc->kv_full[slot], static_cast<uint32_t>((g / kSlots) & 1), misc,
                          a.status)) {
            ok = false;
            break;
          }
          if (g >= 2 && !wait_bar_s(&misc->s_free[sb], static_cast<uint32_t>(((g >> 1) - 1) & 1),
                                    misc, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          fence_proxy_async_smem();
          const uint64_t ad0 = sw128_desc(sbase + kQ, 16, 1024);
          const uint64_t bd0 = sw128_desc(sbase + kKV + slot * kSlotBytes, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < kLatent / 16; ++ks) {
            const uint64_t ad = ad0 + (((ks >> 2) * (kHeads * 128) + (ks & 3) * 32) >> 4);
            const uint64_t bd = bd0 + (((ks >> 2) * kAtomBytes + (ks & 3) * 32) >> 4);
            mma_f16(tmem + 64 * sb, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
          }
          mma_commit(&misc->s_full[sb]);
        }
        mma_commit(&misc->q_free);  // arrives once this query's QK^Ts have completed
        gq += n_tiles;
        if (ok && b + gstep < a.B) {
          ok = wait_bar_s(&misc->q_free, static_cast<uint32_t>(qi & 1), misc, a.status);
          if (ok) load_q(b + gstep);
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- PV issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_o = mma_idesc(128, kHeads, true, true, false);
      bool ok = true;
      int64_t gq = 0;
      int qi = 0;
      for (int b = b0; b < a.B && ok; b += gstep, ++qi) {
        if (!wait_count(&misc->ids_seq, qi + 1, misc, a.status)) break;
        const int n_tiles = tiles_of(b, qi);
        raise_count(&misc->pv_seq, qi + 1);
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int64_t g = gq + t;
          const int slot = static_cast<int>(g % kSlots), sb = static_cast<int>(g & 1);
          if (!wait_bar_s(&misc->p_full[sb], static_cast<uint32_t>((g >> 1) & 1), misc,
                          a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          fence_proxy_async_smem();
          const uint64_t ad0 = sw128_desc(sbase + kKV + slot * kSlotBytes, kAtomBytes, 1024);
          const uint64_t bd0 = sw128_desc(sbase + kP + sb * kPBytes, 16, 1024);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int ks = 0; ks < kRows / 16; ++ks) {
              const uint64_t ad = ad0 + ((m * 2 * kAtomBytes + ks * 16 * 128) >> 4);
              const uint64_t bd = bd0 + ((ks * 32) >> 4);
              mma_f16(tmem + 128 + 64 * m, ad, bd, idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
            }
          }
          mma_commit(&misc->kv_empty[slot]);
          mma_commit(&misc->p_empty[sb]);
        }
        // o_done's phases stay one per query in step with the epilogues:
        // this query's commit waits for the previous query's epilogue.
        if (ok) ok = wait_count(&misc->epi_seq, qi, misc, a.status);
        mma_commit(&misc->o_done);  // arrives once this query's PVs have completed
        gq += n_tiles;
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}
}  // namespace

// Clusters of `splits` CTAs (32-row tiles) that can be resident at once on
// the current device (clusters must fit a GPC; several GPCs cannot hold as
// many 8-CTA clusters as SMs / 8). Cached per device and size.
int attn_max_clusters(int splits) {
  static std::atomic<int> cache[64][4]{};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int k = splits == 2 ? 0 : splits == 4 ? 1 : splits == 8 ? 2 : 3;
  int n = cache[dev][k].load(std::memory_order_relaxed);
  if (n > 0) return n;
  static std::atomic<int> smem_set[64]{};
  if (ensure_smem(reinterpret_cast<const void*>(attn_kernel<32, false>), kSmemBytes, smem_set) !=
      cudaSuccess) {
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 1;
  attr.val.clusterDim.y = static_cast<unsigned>(splits);
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<32, false>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the error the failed query left behind
    n = device_sm_count() / splits;
  }
  cache[dev][k].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  if (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8) {
    return cudaErrorInvalidValue;
  }
  // Q as rows of 512 bf16 (one per query head), boxes of 64 heads x 64 dims.
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  cudaError_t e = encode_tma_2d(&qmap, a.q, 2, kLatent, static_cast<uint64_t>(a.B) * kHeads,
                                kLatent * 2, 64, kHeads);
  if (e != cudaSuccess) return e;
  // Rows of the window buffer (decode: B x window rows; prefill: n_q + window - 1).
  const uint64_t wrows =
      a.prefill ? (a.mq > 0 ? static_cast<uint64_t>(a.B / a.mq) * a.swa_seq_rows
                            : static_cast<uint64_t>(a.B) + a.window - 1)
                : static_cast<uint64_t>(a.B) * a.window;
  // an fp8 cache is read by the split kernel with 32-row tiles only
  if (a.kv_fp8 && (a.splits == 1 || a.tile_rows != 32)) return cudaErrorInvalidValue;
  AttnArgs args = a;
  args.swa_rows = static_cast<int64_t>(wrows);
  if (a.splits == 1) {
    // unsplit: persistent CTAs, one per SM at most, each walking its queries
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(a.B, device_sm_count()));
    if (a.tile_rows == 64) {
      static std::atomic<int> smem_set[64]{};
      e = ensure_smem(reinterpret_cast<const void*>(attn_stream_kernel<64>), kSmemStream, smem_set);
      if (e != cudaSuccess) return e;
      return launch_pdl(attn_stream_kernel<64>, dim3(grid), dim3(kThreads), kSmemStream, s, 1, args,
                        qmap);
    }
    if (a.tile_rows != 32) return cudaErrorInvalidValue;
    static std::atomic<int> smem_set[64]{};
    e = ensure_smem(reinterpret_cast<const void*>(attn_stream_kernel<32>), kSmemStream, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_stream_kernel<32>, dim3(grid), dim3(kThreads), kSmemStream, s, 1, args,
                      qmap);
  }
  if (a.tile_rows == 64) {
    static std::atomic<int> smem_set[64]{};
    e = ensure_smem(reinterpret_cast<const void*>(attn_kernel<64, false>), kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_kernel<64, false>, dim3(a.B, a.splits), dim3(kThreads), kSmemBytes, s,
                      a.splits, args, qmap);
  }
  if (a.tile_rows != 32) return cudaErrorInvalidValue;
  static std::atomic<int> smem_set[64]{};
  if (a.kv_fp8) {
    static std::atomic<int> smem_set8[64]{};
    e = ensure_smem(reinterpret_cast<const void*>(attn_kernel<32, true>), kSmemBytes, smem_set8);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_kernel<32, true>, dim3(a.B, a.splits), dim3(kThreads), kSmemBytes, s,
                      a.splits, args, qmap);
  }
  e = ensure_smem(reinterpret_cast<const void*>(attn_kernel<32, false>), kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<32, false>, dim3(a.B, a.splits), dim3(kThreads), kSmemBytes, s,
                    a.splits, args, qmap);
}

}  // namespace dsa
