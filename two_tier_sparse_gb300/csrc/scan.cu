// S1 / S3: indexer scores (the indexer side attention of recipes.vllm.ai
// "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention"; the formula
// score = sum_h w_h * ReLU(q_h . k) is the one this library fixes).
//
// Per query the scores are one skinny contraction: keys [rows x 128] times
// q_idx^T [128 x 16 heads]. Tiles of 128 key rows are the M side of a
// tcgen05.mma (M = 128, N = 16, fp32 accumulators in tensor memory), so the
// key stream stays HBM-bound instead of CUDA-core-bound (4096 flop per key).
//
//  * bf16 keys are copied into 128-byte-swizzled shared tiles by cp.async and
//    used directly as the bf16 A operand.
//  * MXFP8 keys (e4m3 codes + one UE8M0 scale per 32 values) are converted
//    code by code to f16 (exact: every e4m3 value is an f16 normal) and each
//    32-wide group gets its own accumulator (4 x 16 TMEM columns), so the
//    power-of-two group scales are applied exactly in the epilogue. The index
//    query is taken to f16 with a power-of-two scale per head that puts its
//    largest element in [2^14, 2^15); a bf16 value is then exact in f16 unless
//    it is below 2^-31 of its head's largest element.
// The epilogue thread of TMEM lane r reads the 16 head dot products of row r
// and writes score = sum_h w_h * max(0, dot_h), summed in head order.
#include <algorithm>

#include "kernels.h"

namespace dsa {

namespace {

constexpr int kThreads = 128;
constexpr int kTile = 128;   // key rows per MMA (M)
template <int FMT>
struct Plan;

// Shared-memory plan (offsets from a 1024-aligned base); kStages is the
// depth of the cp.async ring (kStages - 1 tiles in flight).
template <>
struct Plan<DSA_FMT_BF16> {
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kTile * 256;            // 2 K-atoms x 128 rows x 128 B
  static constexpr int kRing = 0;
  static constexpr int kQ = kRing + kStages * kStageBytes;  // 2 atoms x 16 rows x 128 B
  static constexpr int kMisc = kQ + 4096;
  static constexpr int kBytes = kMisc + 1024;
  static constexpr int kTmemCols = 32;
};
template <>
struct Plan<DSA_FMT_MXFP8> {
  static constexpr int kStages = 6;
  static constexpr int kStageBytes = kTile * 128;            // raw codes, swizzled
  static constexpr int kRing = 0;
  static constexpr int kScales = kRing + kStages * kStageBytes;  // kStages x 128 rows x 4 B
  static constexpr int kOp = kScales + kStages * kTile * 4;       // 2 x f16 operand tiles
  static constexpr int kOpBytes = kTile * 256;
  static constexpr int kQ = kOp + 2 * kOpBytes;
  static constexpr int kMisc = kQ + 4096;
  static constexpr int kBytes = kMisc + 1024;
  static constexpr int kTmemCols = 64;
};

struct Misc {
  uint64_t bar;
  uint32_t tmem_base;
  float w[kIdxHeads];
  float qinv[kIdxHeads];  // 2^-s_h (f16 path) or 1
};

__device__ __forceinline__ int visible_latents(const ScanArgs& a, int b) {
  if (a.prefill) return static_cast<int>((a.ctx + b + 1) / a.ratio);
  return a.n_latents[b];
}

// Key row of output row r of query b, or -1 if the row holds no key.
__device__ __forceinline__ int64_t key_row(const ScanArgs& a, int b, int n_vis, int64_t r) {
  if (r >= a.n_rows) return -1;
  if (a.mode == ROWS_BLOCKS) {
    const int64_t nb = (n_vis + 7) / 8;
    return r < nb ? r : -1;
  }
  if (a.mode == ROWS_LATENTS) return r < n_vis ? r : -1;
  const int64_t bi = r >> 3;
  if (bi >= a.k_blocks) return -1;
  const int blk = a.block_ids[static_cast<int64_t>(b) * a.k_blocks + bi];
  if (blk < 0) return -1;
  const int64_t t = static_cast<int64_t>(blk) * 8 + (r & 7);
  return t < n_vis ? t : -1;
}

// Prefill block rows: the last block of a query that sees it only in part is
// read from the per-query partial-block buffer instead of the pooled cache.
__device__ __forceinline__ bool is_partial(const ScanArgs& a, int n_vis, int64_t kr) {
  return a.prefill && a.mode == ROWS_BLOCKS && (n_vis & 7) != 0 && kr == (n_vis >> 3);
}
__device__ __forceinline__ const uint8_t* row_src(const ScanArgs& a, int b, int n_vis, int64_t kr,
                                                  int64_t seq, const uint8_t* kd, int row_bytes) {
  if (is_partial(a, n_vis, kr)) {
    return static_cast<const uint8_t*>(a.partial_data) + static_cast<int64_t>(b) * row_bytes;
  }
  return kd + (seq + kr) * row_bytes;
}

template <int FMT>
__device__ __forceinline__ void issue_tile_load(const ScanArgs& a, uint32_t sbase, int stage,
                                                int64_t tile, int64_t tpq) {
  using P = Plan<FMT>;
  const int tid = threadIdx.x;
  const int b = static_cast<int>(tile / tpq);
  const int64_t r0 = (tile % tpq) * kTile;
  int n_vis = visible_latents(a, b);
  if (n_vis > a.max_latents) n_vis = static_cast<int>(a.max_latents);
  const int64_t seq = static_cast<int64_t>(b) * a.key_stride;
  if constexpr (FMT == DSA_FMT_BF16) {
    const uint8_t* kd = static_cast<const uint8_t*>(a.key_data);
    const uint32_t st = sbase + P::kRing + stage * P::kStageBytes;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const int c = tid + kThreads * j;
      const int row = c >> 4, cr = c & 15;
      const int64_t kr = key_row(a, b, n_vis, r0 + row);
      const uint32_t dst = st + (cr >> 3) * (kTile * 128) + sw128_off(row, cr & 7);
      if (kr >= 0) {
        cp_async_16(dst, row_src(a, b, n_vis, kr, seq, kd, 256) + cr * 16);
      } else {
        st_shared_v4(dst, make_uint4(0, 0, 0, 0));
      }
    }
  } else {
    const uint8_t* kd = static_cast<const uint8_t*>(a.key_data);
    const uint32_t st = sbase + P::kRing + stage * P::kStageBytes;
#pragma unroll 4
    for (int j = 0; j < 8; ++j) {
      const int c = tid + kThreads * j;
      const int row = c >> 3, cr = c & 7;
      const int64_t kr = key_row(a, b, n_vis, r0 + row);
      const uint32_t dst = st + sw128_off(row, cr);
      if (kr >= 0) {
        cp_async_16(dst, row_src(a, b, n_vis, kr, seq, kd, 128) + cr * 16);
      } else {
        st_shared_v4(dst, make_uint4(0, 0, 0, 0));
      }
    }
    const int64_t kr = key_row(a, b, n_vis, r0 + tid);
    const uint32_t sdst = sbase + P::kScales + (stage * kTile + tid) * 4;
    if (kr >= 0) {
      const bool part = is_partial(a, n_vis, kr);
      cp_async_4(sdst, part ? a.partial_scales + static_cast<int64_t>(b) * 4
                            : a.key_scales + (seq + kr) * 4);
    } else {
      asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(sdst), "r"(127u * 0x01010101u) : "memory");
    }
  }
}

// Index query of query b -> B operand (16 rows x 128, K-major, swizzled).
template <int FMT>
__device__ __forceinline__ void load_query(const ScanArgs& a, uint32_t sbase, Misc* misc, int b) {
  using P = Plan<FMT>;
  const int tid = threadIdx.x;
  const uint16_t* q = a.q_idx + static_cast<int64_t>(b) * kIdxHeads * kIdxDim;
  if (tid < kIdxHeads) misc->w[tid] = a.w[static_cast<int64_t>(b) * kIdxHeads + tid];
  if constexpr (FMT == DSA_FMT_BF16) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = tid + kThreads * j;
      const int h = c >> 4, cr = c & 15;
      const uint4 v = *reinterpret_cast<const uint4*>(q + h * kIdxDim + cr * 8);
      st_shared_v4(sbase + P::kQ + (cr >> 3) * 2048 + sw128_off(h, cr & 7), v);
    }
    if (tid < kIdxHeads) misc->qinv[tid] = 1.0f;
  } else {
    // 8 threads per head, 16 elements each.
    const int h = tid >> 3, part = tid & 7;
    const uint4 v0 = *reinterpret_cast<const uint4*>(q + h * kIdxDim + part * 16);
    const uint4 v1 = *reinterpret_cast<const uint4*>(q + h * kIdxDim + part * 16 + 8);
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
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
    const uint32_t qb = sbase + P::kQ;
    const int c0 = 2 * part;  // f16 chunks c0, c0 + 1 (16 B each) of row h
    st_shared_v4(qb + (c0 >> 3) * 2048 + sw128_off(h, c0 & 7), make_uint4(hw[0], hw[1], hw[2], hw[3]));
    st_shared_v4(qb + ((c0 + 1) >> 3) * 2048 + sw128_off(h, (c0 + 1) & 7),
                 make_uint4(hw[4], hw[5], hw[6], hw[7]));
    if (part == 0) misc->qinv[h] = __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) scan_kernel(ScanArgs a, int64_t tpq, int64_t total) {
  using P = Plan<FMT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  Misc* misc = reinterpret_cast<Misc*>(gbase + P::kMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  // Contiguous share of the flattened (query, tile) space.
  const int64_t per = total / gridDim.x, rem = total % gridDim.x;
  const int64_t bx = blockIdx.x;
  const int64_t t_begin = bx * per + (bx < rem ? bx : rem);
  const int64_t t_end = t_begin + per + (bx < rem ? 1 : 0);

  if (tid == 0) {
    mbar_init(&misc->bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&misc->tmem_base, P::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  constexpr int kStages = P::kStages;
  for (int s = 0; s < kStages - 1; ++s) {
    if (t_begin + s < t_end) issue_tile_load<FMT>(a, sbase, s, t_begin + s, tpq);
    cp_async_commit();
  }

  uint32_t phase = 0;
  bool ok = true;
  int cur_b = -1;  // query whose index query sits in shared memory
  for (int64_t tile = t_begin; tile < t_end && ok; ++tile) {
    const int64_t it = tile - t_begin;
    const int64_t nxt = tile + kStages - 1;
    if (nxt < t_end) issue_tile_load<FMT>(a, sbase, static_cast<int>(nxt - t_begin) % kStages, nxt, tpq);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    const int stage = static_cast<int>(it % kStages);
    const int b = static_cast<int>(tile / tpq);
    const int64_t r0 = (tile % tpq) * kTile;

    // Every thread has finished the previous epilogue (which reads the query
    // data) and every thread's copies of this tile have landed.
    __syncthreads();
    if (b != cur_b) {
      load_query<FMT>(a, sbase, misc, b);
      cur_b = b;
    }

    uint32_t my_scales = 0;
    uint32_t a_base;
    if constexpr (FMT == DSA_FMT_BF16) {
      a_base = sbase + P::kRing + stage * P::kStageBytes;
    } else {
      const uint32_t rawt = sbase + P::kRing + stage * P::kStageBytes;
      const uint32_t op = sbase + P::kOp + static_cast<uint32_t>(it & 1) * P::kOpBytes;
      const int row = tid;
      asm volatile("ld.shared.u32 %0, [%1];\n"
                   : "=r"(my_scales)
                   : "r"(sbase + P::kScales + (stage * kTile + row) * 4));
#pragma unroll
      for (int cr = 0; cr < 8; ++cr) {
        const uint4 v = ld_shared_v4(rawt + sw128_off(row, cr));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>(wv[i] & 0xFFFF), __NV_E4M3);
          const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>(wv[i] >> 16), __NV_E4M3);
          h[2 * i] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
          h[2 * i + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
        }
        const int c0 = 2 * cr;
        st_shared_v4(op + (c0 >> 3) * (kTile * 128) + sw128_off(row, c0 & 7),
                     make_uint4(h[0], h[1], h[2], h[3]));
        st_shared_v4(op + ((c0 + 1) >> 3) * (kTile * 128) + sw128_off(row, (c0 + 1) & 7),
                     make_uint4(h[4], h[5], h[6], h[7]));
      }
      a_base = op;
    }
    fence_proxy_async_smem();
    __syncthreads();

    if (tid == 0) {
      tc_fence_after();
      const uint32_t qb = sbase + P::kQ;
      if constexpr (FMT == DSA_FMT_BF16) {
        constexpr uint32_t idesc = mma_idesc(kTile, kIdxHeads, true, false, false);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = sw128_desc(a_base + (k >> 2) * (kTile * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(qb + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024);
          mma_f16(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
      } else {
        constexpr uint32_t idesc = mma_idesc(kTile, kIdxHeads, false, false, false);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // group g = k / 2 -> accumulator columns 16 g
          const uint64_t ad = sw128_desc(a_base + (k >> 2) * (kTile * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(qb + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024);
          mma_f16(tmem + (k >> 1) * 16, ad, bd, idesc, (k & 1) ? 1u : 0u);
        }
      }
      mma_commit(&misc->bar);
    }
    ok = mbar_wait(&misc->bar, phase, a.status, SITE_SCAN);
    ok = __syncthreads_and(ok) != 0;  // one decision for the whole CTA
    phase ^= 1u;
    tc_fence_after();
    if (!ok) break;

    // Epilogue: thread tid owns TMEM lane tid = row r0 + tid.
    const uint32_t lane_addr = tmem_addr(tmem, static_cast<uint32_t>(warp * 32), 0);
    float dot[kIdxHeads];
    if constexpr (FMT == DSA_FMT_BF16) {
      tmem_ld16(lane_addr, dot);
    } else {
      float acc[16];
#pragma unroll
      for (int h = 0; h < kIdxHeads; ++h) dot[h] = 0.f;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        tmem_ld16(lane_addr + g * 16, acc);
        const uint32_t sc = (my_scales >> (8 * g)) & 0xFF;
        const float f = __uint_as_float(sc == 0 ? 0x00400000u : sc << 23);
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) dot[h] = fmaf(acc[h], f, dot[h]);
      }
#pragma unroll
      for (int h = 0; h < kIdxHeads; ++h) dot[h] *= misc->qinv[h];
    }
    tc_fence_before();
    const int64_t r = r0 + tid;
    if (r < a.n_rows) {
      int n_vis = visible_latents(a, b);
      if (n_vis > a.max_latents) n_vis = static_cast<int>(a.max_latents);
      float s = -INFINITY;
      if (key_row(a, b, n_vis, r) >= 0) {
        s = 0.f;
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) s = fmaf(misc->w[h], fmaxf(dot[h], 0.f), s);
      }
      a.scores[static_cast<int64_t>(b) * a.n_rows + r] = s;
    }
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, P::kTmemCols);
  }
}

template <int FMT>
cudaError_t launch_fmt(const ScanArgs& a, int num_sms, cudaStream_t s) {
  using P = Plan<FMT>;
  const int64_t tpq = (a.n_rows + kTile - 1) / kTile;
  const int64_t total = tpq * a.B;
  if (total == 0) return cudaSuccess;
  const int smem = P::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = (FMT == DSA_FMT_BF16) ? 1 : 2;
  const int64_t grid = std::min<int64_t>(total, static_cast<int64_t>(num_sms) * per_sm);
  scan_kernel<FMT><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(a, tpq, total);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, int num_sms, cudaStream_t s) {
  if (a.fmt == DSA_FMT_BF16) return launch_fmt<DSA_FMT_BF16>(a, num_sms, s);
  return launch_fmt<DSA_FMT_MXFP8>(a, num_sms, s);
}

}  // namespace dsa
