// S0: block keys of the candidate stage. Each block of 8 index keys is
// replaced by its mean (recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview,
// "Two-tier sparse attention": a candidate stage over "blocks of 8"; the mean
// is the block-key rule this library fixes), summed in fp32 in member order,
// divided by the member count in fp32 and stored in the keys' own format:
// bf16 round-to-nearest-even, or MXFP8 / MXFP4 by the OCP MX v1.0 conversion.
#include "kernels.h"

namespace dsa {

namespace {

// Lane l of a warp owns elements 4l .. 4l+3 of a 128-wide key row.
__device__ __forceinline__ void load4(int fmt, const void* key_data, const uint8_t* key_scales,
                                      int64_t row, int lane, float (&x)[4]) {
  if (fmt == DSA_FMT_BF16) {
    const uint16_t* k = static_cast<const uint16_t*>(key_data);
    const uint2 v = *reinterpret_cast<const uint2*>(k + row * 128 + lane * 4);
    x[0] = bf16_bits_to_float(v.x & 0xFFFF);
    x[1] = bf16_bits_to_float(v.x >> 16);
    x[2] = bf16_bits_to_float(v.y & 0xFFFF);
    x[3] = bf16_bits_to_float(v.y >> 16);
  } else if (fmt == DSA_FMT_MXFP4) {
    // bytes 2 lane, 2 lane + 1 of the 64-byte row: elements 4 lane .. 4 lane + 3
    const uint8_t* k = static_cast<const uint8_t*>(key_data);
    const uint32_t codes = *reinterpret_cast<const uint16_t*>(k + row * 64 + lane * 2);
    const int sc = key_scales[row * 4 + (lane >> 3)];
    const float f = __uint_as_float(sc == 0 ? 0x00400000u : static_cast<uint32_t>(sc) << 23);
    // e2m1 -> f16 -> f32 is exact, and so is the power-of-two scaling.
    const __half2_raw h01 = __nv_cvt_fp4x2_to_halfraw2(
        static_cast<__nv_fp4x2_storage_t>(codes & 0xFF), __NV_E2M1);
    const __half2_raw h23 = __nv_cvt_fp4x2_to_halfraw2(
        static_cast<__nv_fp4x2_storage_t>(codes >> 8), __NV_E2M1);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    x[0] = f01.x * f;
    x[1] = f01.y * f;
    x[2] = f23.x * f;
    x[3] = f23.y * f;
  } else {
    const uint8_t* k = static_cast<const uint8_t*>(key_data);
    const uint32_t codes = *reinterpret_cast<const uint32_t*>(k + row * 128 + lane * 4);
    const int sc = key_scales[row * 4 + (lane >> 3)];
    const float f = __uint_as_float(sc == 0 ? 0x00400000u : static_cast<uint32_t>(sc) << 23);
    // e4m3 -> f16 -> f32 is exact, and so is the power-of-two scaling.
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(codes & 0xFFFF), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(codes >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    x[0] = f01.x * f;
    x[1] = f01.y * f;
    x[2] = f23.x * f;
    x[3] = f23.y * f;
  }
}

// Mean of rows [row0, row0 + c), c in 1..8: fp32 sum in member order, then
// / c in fp32. The c loads are all issued before the first add, so the block
// costs one memory round trip rather than c.
__device__ __forceinline__ void block_mean(int fmt, const void* key_data, const uint8_t* key_scales,
                                           int64_t row0, int c, int lane, float (&acc)[4]) {
  float x[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < c) load4(fmt, key_data, key_scales, row0 + j, lane, x[j]);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] = x[0][e];
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    if (j < c) {
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], x[j][e]);
    }
  }
  const float cf = static_cast<float>(c);
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] = __fdiv_rn(acc[e], cf);
}

// Rounds a warp's 128 fp32 values to the key format. Returns the packed
// storage (bf16: 2 words; MXFP8: 1 word of codes, MXFP4: 16 bits of codes,
// + the group's scale byte) and, in `dec`, the stored values decoded back to
// fp32 (exact).
struct Stored {
  uint32_t w0, w1;
  uint8_t scale;
};
__device__ __forceinline__ Stored round_to_format(int fmt, const float (&v)[4], float (&dec)[4]) {
  Stored st{0, 0, 0};
  if (fmt == DSA_FMT_BF16) {
    uint16_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(v[e]));
      dec[e] = bf16_bits_to_float(h[e]);
    }
    st.w0 = h[0] | (static_cast<uint32_t>(h[1]) << 16);
    st.w1 = h[2] | (static_cast<uint32_t>(h[3]) << 16);
    return st;
  }
  // Group of 32 values = 8 lanes: X = floor(log2(amax)) - emax (8 for e4m3,
  // 2 for e2m1), clamped to [-127, 127]; an all-zero group takes X = 0.
  const int emax = fmt == DSA_FMT_MXFP4 ? 2 : 8;
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  int X;
  if (amax == 0.f) {
    X = 0;
  } else {
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
    X = (e == 0) ? -127 : max(-127, e - 127 - emax);
  }
  // v * 2^-X is exact (a power-of-two scaling); then the element format,
  // nearest-even, saturating (e4m3 to +-448, e2m1 to +-6).
  const int ex = 127 - X;  // biased exponent of 2^-X, in [2, 254]
  const float inv = __uint_as_float(ex == 0 ? 0x00400000u : static_cast<uint32_t>(ex) << 23);
  const float back = __uint_as_float(X + 127 == 0 ? 0x00400000u : static_cast<uint32_t>(X + 127) << 23);
  st.scale = static_cast<uint8_t>(X + 127);
  if (fmt == DSA_FMT_MXFP4) {
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const float2 pr = make_float2(v[e] * inv, v[e + 1] * inv);
      const __nv_fp4x2_storage_t q = __nv_cvt_float2_to_fp4x2(pr, __NV_E2M1, cudaRoundNearest);
      st.w0 |= static_cast<uint32_t>(q) << (8 * (e >> 1));
      const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(q, __NV_E2M1);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      dec[e] = f.x * back;
      dec[e + 1] = f.y * back;
    }
    return st;
  }
#pragma unroll
  for (int e = 0; e < 4; e += 2) {
    const float2 pr = make_float2(v[e] * inv, v[e + 1] * inv);
    const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
    st.w0 |= static_cast<uint32_t>(q) << (16 * (e >> 1));
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    dec[e] = f.x * back;
    dec[e + 1] = f.y * back;
  }
  return st;
}

// One warp per (sequence, block). The dependent kernel is released only once
// this kernel's own dependency wait has returned: a decode step's block scan
// reads the blocks this kernel does not write before its own wait, and those
// blocks must be final (every earlier kernel complete).
__global__ void __launch_bounds__(256) pool_kernel(PoolArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int n = a.n_latents[b];
  if (n < 0 || n > a.max_latents) {
    if (lane == 0 && warp == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_POOL, b);
    return;
  }
  const int nb = (n + 7) >> 3;
  int blk;
  if (a.tail_only) {
    if (warp != 0 || nb == 0) return;
    blk = nb - 1;
  } else {
    blk = warp;
    if (blk >= nb) return;
  }
  const int c = min(8, n - blk * 8);
  // The block's member rows (consecutive: a page holds whole blocks) and its
  // block-key row, contiguous or through the page table.
  int64_t row0 = static_cast<int64_t>(b) * a.key_stride + blk * 8;
  int64_t orow = static_cast<int64_t>(b) * a.out_stride + blk;
  if (a.key_pages.table) {
    row0 = paged_row(a.key_pages, b, static_cast<int64_t>(blk) * 8);
    orow = paged_row(a.out_pages, b, blk);
    if (row0 < 0 || orow < 0) {
      if (lane == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_POOL, b);
      return;
    }
  }
  if (!DSA_DCHECK(row0 >= 0 && row0 + c <= a.key_rows && orow >= 0 && orow < a.out_rows,
                  a.status, SITE_POOL, b)) {
    return;
  }
  float acc[4], dec[4];
  block_mean(a.fmt, a.key_data, a.key_scales, row0, c, lane, acc);
  const Stored st = round_to_format(a.fmt, acc, dec);
  if (a.fmt == DSA_FMT_BF16) {
    uint16_t* o = static_cast<uint16_t*>(a.out_data);
    *reinterpret_cast<uint2*>(o + orow * 128 + lane * 4) = make_uint2(st.w0, st.w1);
  } else {
    uint8_t* o = static_cast<uint8_t*>(a.out_data);
    if (a.fmt == DSA_FMT_MXFP4) {
      *reinterpret_cast<uint16_t*>(o + orow * 64 + lane * 2) = static_cast<uint16_t>(st.w0);
    } else {
      *reinterpret_cast<uint32_t*>(o + orow * 128 + lane * 4) = st.w0;
    }
    if ((lane & 7) == 0) a.out_scales[orow * 4 + (lane >> 3)] = st.scale;
  }
}

// One warp per prefill query (or multi-query decode query): pool its
// partially visible last block and score it.
__global__ void __launch_bounds__(256) prefill_partial_kernel(PartialArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= a.n_q) return;
  const int64_t P = query_pos(a.ctx, a.mq, a.n_tokens, b);
  if (P < 0) return;  // a sequence shorter than its queries (reported by the attention)
  const int n = static_cast<int>((P + 1) / a.ratio);
  const int c = n & 7;
  if (c == 0) return;
  const int blk = n >> 3;
  float acc[4], key[4];
  const int64_t row0 = static_cast<int64_t>(query_seq(a.mq, b)) * a.key_stride;
  if (!DSA_DCHECK(row0 + int64_t{blk} * 8 + c <= a.key_rows, nullptr, SITE_PREFILL, b)) return;
  block_mean(a.fmt, a.key_data, a.key_scales, row0 + static_cast<int64_t>(blk) * 8, c, lane, acc);
  round_to_format(a.fmt, acc, key);
  // dot_h = q_h . key: each lane's 4 products, then a fixed xor-tree sum.
  const uint16_t* q = a.q_idx + static_cast<int64_t>(b) * kIdxHeads * kIdxDim;
  float score = 0.f;
  for (int h = 0; h < kIdxHeads; ++h) {
    const uint2 qv = *reinterpret_cast<const uint2*>(q + h * kIdxDim + lane * 4);
    float d = bf16_bits_to_float(qv.x & 0xFFFF) * key[0];
    d = fmaf(bf16_bits_to_float(qv.x >> 16), key[1], d);
    d = fmaf(bf16_bits_to_float(qv.y & 0xFFFF), key[2], d);
    d = fmaf(bf16_bits_to_float(qv.y >> 16), key[3], d);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, off);
    score = fmaf(a.w[static_cast<int64_t>(b) * kIdxHeads + h], fmaxf(d, 0.f), score);
  }
  if (lane == 0) a.scores[static_cast<int64_t>(b) * a.n_rows + blk] = score;
}

// One warp per sequence: the compressed latent of its last ratio positions
// (softmax of the gate logits in fp32, lane i < ratio holding logit i; lane l
// sums dims [16 l, 16 l + 16) over the positions in order) and its index key.
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int n = a.n_tokens[b];
  const int n_lat = n >= 0 ? n / a.ratio : 0;
  if (lane == 0) a.n_lat_out[b] = n_lat;
  if (n <= 0 || n % a.ratio != 0) return;  // no latent completes at this step
  const int j = n_lat - 1;
  int64_t lrow = static_cast<int64_t>(b) * a.lat_stride + j;
  int64_t krow = static_cast<int64_t>(b) * a.key_stride + j;
  if (a.pages.table) lrow = krow = paged_row(a.pages, b, j);
  if (j >= a.max_latents || lrow < 0) {
    if (lane == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_POOL, b);
    return;
  }
  const float g = lane < a.ratio ? a.gate[static_cast<int64_t>(b) * a.ratio + lane] : -INFINITY;
  float m = g;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const float e = lane < a.ratio ? expf(g - m) : 0.f;
  float sum = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  const float wl = e / sum;
  float acc[16];
#pragma unroll
  for (int d = 0; d < 16; ++d) acc[d] = 0.f;
  for (int i = 0; i < a.ratio; ++i) {
    const float wi = __shfl_sync(0xFFFFFFFFu, wl, i);
    const uint4* src = reinterpret_cast<const uint4*>(
        a.kv + (static_cast<int64_t>(b) * a.ratio + i) * kLatent + 16 * lane);
    const uint4 x0 = src[0], x1 = src[1];
    const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[2 * k] = fmaf(wi, bf16_bits_to_float(xs[k] & 0xFFFF), acc[2 * k]);
      acc[2 * k + 1] = fmaf(wi, bf16_bits_to_float(xs[k] >> 16), acc[2 * k + 1]);
    }
  }
  uint32_t out[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
    out[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  uint4* dst = reinterpret_cast<uint4*>(a.latents + lrow * kLatent + 16 * lane);
  dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
  dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  // the index key row (and its scales)
  const int row_bytes = a.fmt == DSA_FMT_BF16 ? 256 : (a.fmt == DSA_FMT_MXFP8 ? 128 : 64);
  if (lane * 16 < row_bytes) {
    *reinterpret_cast<uint4*>(a.key_data + krow * row_bytes + lane * 16) =
        *reinterpret_cast<const uint4*>(a.new_key + static_cast<int64_t>(b) * row_bytes + lane * 16);
  }
  if (a.fmt != DSA_FMT_BF16 && lane < 4) {
    a.key_scales[krow * 4 + lane] = a.new_scales[static_cast<int64_t>(b) * 4 + lane];
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  const int grid = (a.B + 7) / 8;
  return launch_pdl(append_kernel, dim3(grid), dim3(256), 0, s, 1, a);
}

cudaError_t launch_pool(const PoolArgs& a, cudaStream_t s) {
  const int64_t nb_max = (a.max_latents + 7) / 8;
  const int warps = a.tail_only ? 1 : static_cast<int>(nb_max > 0 ? nb_max : 1);
  const int threads = a.tail_only ? 32 : 256;
  const int wpb = threads / 32;
  dim3 grid((warps + wpb - 1) / wpb, a.B);
  return launch_pdl(pool_kernel, grid, dim3(threads), 0, s, 1, a);
}

cudaError_t launch_prefill_partial(const PartialArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int grid = (a.n_q + warps_per_block - 1) / warps_per_block;
  return launch_pdl(prefill_partial_kernel, dim3(grid), dim3(32 * warps_per_block), 0, s, 1, a);
}

}  // namespace dsa
