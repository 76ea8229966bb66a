// S5 - S7: attention over the gathered latents and the sliding window under one
// softmax (miles.radixark.com "DeepSeek-V4.1 Flash", §1 "Architecture": one
// 512-wide latent per position is both key and value for all 64 query heads;
// recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention":
// the 128-token window plus the selected latents).
//
// One CTA per query. Rows (selected latents, then window rows) stream through
// shared memory in tiles of 64 by cp.async into 128-byte-swizzled tiles. For
// each tile two tcgen05 MMAs run with fp32 accumulators in tensor memory:
//   S   = Q . KV^T  (M = 128 with the 64 heads in lanes 0..63, N = 64 rows, K = 512)
//   O^T += KV^T . P^T (four M = 128 slices of the 512 latent dims, N = 64 heads,
//                      K = 64 rows; the KV tile is read as an MN-major operand)
// The softmax runs in registers, one head per thread, online across tiles with
// the running maximum only moved when it grows by more than 2^8 (the stale
// maximum keeps every P value <= 256, exact enough in bf16 and fp32).
#include "kernels.h"

namespace dsa {

namespace {

constexpr int kThreads = 128;
constexpr int kRows = 64;  // KV rows per tile

// Shared-memory plan (offsets from a 1024-aligned base).
constexpr int kQ = 0;                        // 8 atoms x 64 heads x 128 B, + 8 KB read past the end
constexpr int kQBytes = 8 * kHeads * 128 + 8192;
constexpr int kKV = kQ + kQBytes;            // 2 buffers x 8 atoms x 64 rows x 128 B
constexpr int kKVBytes = 8 * kRows * 128;
constexpr int kP = kKV + 2 * kKVBytes;       // P: 64 heads x 64 rows bf16 (one atom)
constexpr int kIds = kP + kHeads * 128;      // compacted latent ids
constexpr int kMisc = kIds + kMaxKTokens * 4;
constexpr int kSmemBytes = kMisc + 1024 + 1024;
constexpr int kTmemCols = 512;               // S: cols [0, 64); O^T slice m: cols [64 + 64 m, 128 + 64 m)

struct Misc {
  uint64_t bar;
  uint32_t tmem_base;
  int n_sel;
  int rescale;
  int warp_cnt[kThreads / 32];
  float alpha[kHeads];
  float inv_l[kHeads];
};

__global__ void __launch_bounds__(kThreads, 1) attn_kernel(AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  Misc* misc = reinterpret_cast<Misc*>(gbase + kMisc);
  int32_t* ids = reinterpret_cast<int32_t*>(gbase + kIds);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;

  if (tid == 0) {
    mbar_init(&misc->bar, 1);
    misc->rescale = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&misc->tmem_base, kTmemCols);

  // Visible latents and this query's window rows.
  int n_vis;
  const uint16_t* win;
  int n_sw;
  if (a.prefill) {
    const int64_t P = a.ctx + b;
    n_vis = static_cast<int>((P + 1) / a.ratio);
    const int64_t first = P - a.window + 1 > 0 ? P - a.window + 1 : 0;
    const int64_t base_pos = a.ctx - a.window + 1;
    win = a.swa + (first - base_pos) * kLatent;
    n_sw = static_cast<int>(P - first + 1);
  } else {
    n_vis = a.n_latents[b];
    n_sw = a.swa_len[b];
    if (n_sw < 0 || n_sw > a.window) {
      if (tid == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, b);
      n_sw = n_sw < 0 ? 0 : a.window;
    }
    win = a.swa + static_cast<int64_t>(b) * a.window * kLatent;
  }
  if (n_vis > a.lat_stride) n_vis = static_cast<int>(a.lat_stride);

  // Compact the valid token ids (>= 0 and < n_vis) in order.
  {
    const int32_t* tk = a.token_ids + static_cast<int64_t>(b) * a.k_tokens;
    constexpr int kPer = kMaxKTokens / kThreads;  // 4
    int my[kPer];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid * kPer + j;
      int id = -1;
      if (i < a.k_tokens) {
        id = tk[i];
        if (id >= n_vis) {
          record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_ATTN, static_cast<uint32_t>(id));
          id = -1;
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
    __syncthreads();
    int before = incl - cnt;
    for (int w = 0; w < warp; ++w) before += misc->warp_cnt[w];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (my[j] >= 0) ids[before++] = my[j];
    }
    if (tid == kThreads - 1) misc->n_sel = before;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const int n_sel = misc->n_sel;
  const int n_rows = n_sel + n_sw;
  const int n_tiles = (n_rows + kRows - 1) / kRows;

  const uint16_t* qsrc = a.q + static_cast<int64_t>(b) * kHeads * kLatent;
  const uint16_t* lat = a.latents + (a.prefill ? 0 : static_cast<int64_t>(b) * a.lat_stride * kLatent);
  uint16_t* out = a.out + static_cast<int64_t>(b) * kHeads * kLatent;

  if (n_tiles == 0) {
    for (int i = tid; i < kHeads * kLatent / 8; i += kThreads) {
      reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
    }
    if (a.lse && tid < kHeads) a.lse[static_cast<int64_t>(b) * kHeads + tid] = -INFINITY;
  } else {
    // Q: 64 rows x 64 chunks of 16 B.
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
      const int c = tid + kThreads * j;
      const int h = c >> 6, cr = c & 63;
      cp_async_16(sbase + kQ + (cr >> 3) * (kHeads * 128) + sw128_off(h, cr & 7),
                  qsrc + h * kLatent + cr * 8);
    }
    auto load_tile = [&](int t, int buf) {
      const uint32_t dstb = sbase + kKV + buf * kKVBytes;
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int c = tid + kThreads * j;
        const int row = c >> 6, cr = c & 63;
        const int g = t * kRows + row;
        const uint32_t dst = dstb + (cr >> 3) * (kRows * 128) + sw128_off(row, cr & 7);
        if (g < n_sel) {
          cp_async_16(dst, lat + static_cast<int64_t>(ids[g]) * kLatent + cr * 8);
        } else if (g < n_rows) {
          cp_async_16(dst, win + static_cast<int64_t>(g - n_sel) * kLatent + cr * 8);
        } else {
          st_shared_v4(dst, make_uint4(0, 0, 0, 0));
        }
      }
    };
    load_tile(0, 0);
    cp_async_commit();

    float m_run = -INFINITY, l_run = 0.f;  // threads 0..63: head tid
    uint32_t phase = 0;
    bool ok = true;
    constexpr uint32_t idesc_s = mma_idesc(128, kRows, true, false, false);
    constexpr uint32_t idesc_o = mma_idesc(128, kHeads, true, true, false);
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int buf = t & 1;
      if (t + 1 < n_tiles) load_tile(t + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
      if (tid == 0) misc->rescale = 0;
      fence_proxy_async_smem();
      __syncthreads();
      const uint32_t kvb = sbase + kKV + buf * kKVBytes;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kLatent / 16; ++ks) {
          const uint64_t ad = sw128_desc(sbase + kQ + (ks >> 2) * (kHeads * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(kvb + (ks >> 2) * (kRows * 128) + (ks & 3) * 32, 16, 1024);
          mma_f16(tmem, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&misc->bar);
      }
      ok = __syncthreads_and(mbar_wait(&misc->bar, phase, a.status, SITE_ATTN)) != 0;
      phase ^= 1u;
      tc_fence_after();
      if (!ok) break;

      if (tid < kHeads) {
        const int valid = min(kRows, n_rows - t * kRows);
        float z[kRows];
#pragma unroll
        for (int c = 0; c < kRows / 16; ++c) {
          float v[16];
          tmem_ld16(tmem_addr(tmem, static_cast<uint32_t>(warp * 32), c * 16), v);
#pragma unroll
          for (int i = 0; i < 16; ++i) z[c * 16 + i] = (c * 16 + i < valid) ? v[i] * a.scale_log2 : -INFINITY;
        }
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < kRows; ++i) mt = fmaxf(mt, z[i]);
        float alpha = 1.f;
        if (t == 0) {
          m_run = mt;
        } else if (mt > m_run + 8.f) {
          alpha = exp2f(m_run - mt);
          m_run = mt;
          misc->rescale = 1;
        }
        float sum = 0.f;
        uint32_t pk[kRows / 2];
#pragma unroll
        for (int i = 0; i < kRows; i += 2) {
          const float p0 = exp2f(z[i] - m_run), p1 = exp2f(z[i + 1] - m_run);
          sum += p0 + p1;  // the denominator sums the fp32 probabilities
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(p0, p1);
          pk[i / 2] = *reinterpret_cast<const uint32_t*>(&p2);
        }
        l_run = l_run * alpha + sum;
        misc->alpha[tid] = alpha;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          st_shared_v4(sbase + kP + sw128_off(tid, c),
                       make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncthreads();
      if (misc->rescale) {
        tc_fence_after();
        const uint32_t la = tmem_addr(tmem, static_cast<uint32_t>(warp * 32), 0);
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v[16];
            const uint32_t addr = la + 64 + 64 * m + 16 * c;
            tmem_ld16(addr, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= misc->alpha[16 * c + i];
            tmem_st16(addr, v);
          }
        }
        tc_fence_before();
        __syncthreads();
      }
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks) {
            const uint64_t ad = sw128_desc(kvb + m * 2 * (kRows * 128) + ks * 16 * 128, kRows * 128, 1024);
            const uint64_t bd = sw128_desc(sbase + kP + ks * 32, 16, 1024);
            mma_f16(tmem + 64 + 64 * m, ad, bd, idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
          }
        }
        mma_commit(&misc->bar);
      }
      ok = __syncthreads_and(mbar_wait(&misc->bar, phase, a.status, SITE_ATTN)) != 0;
      phase ^= 1u;
      tc_fence_after();
    }

    if (tid < kHeads) {
      misc->inv_l[tid] = 1.f / l_run;
      if (a.lse) a.lse[static_cast<int64_t>(b) * kHeads + tid] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    }
    __syncthreads();
    if (ok) {
      const uint32_t la = tmem_addr(tmem, static_cast<uint32_t>(warp * 32), 0);
      for (int m = 0; m < 4; ++m) {
        const int d = m * 128 + tid;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
          tmem_ld16(la + 64 + 64 * m + 16 * c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = 16 * c + i;
            out[h * kLatent + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i] * misc->inv_l[h]));
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_kernel<<<a.B, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
