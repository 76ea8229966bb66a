// S0: block keys of the candidate stage. Each block of 8 index keys is
// replaced by its mean (recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview,
// "Two-tier sparse attention": a candidate stage over "blocks of 8"; the mean
// is the block-key rule this library fixes), summed in fp32 in member order,
// divided by the member count in fp32 and stored in the keys' own format:
// bf16 round-to-nearest-even, or MXFP8 by the OCP MX v1.0 conversion.
#include "kernels.h"

namespace dsa {

namespace {

// One warp per (sequence, block): lane l owns elements 4l .. 4l+3.
__global__ void __launch_bounds__(256) pool_kernel(PoolArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  int n;
  if (a.prefill) {
    n = static_cast<int>((a.ctx + b + 1) / a.ratio);
    if ((n & 7) == 0) return;
  } else {
    n = a.n_latents[b];
  }
  if (n < 0 || n > a.max_latents) {
    if (lane == 0 && warp == 0) record_status(a.status, DSA_ERR_DEVICE_CHECK, SITE_POOL, b);
    return;
  }
  const int nb = (n + 7) >> 3;
  int blk;
  if (a.tail_only || a.prefill) {
    if (warp != 0 || nb == 0) return;
    blk = nb - 1;
  } else {
    blk = warp;
    if (blk >= nb) return;
  }
  const int first = blk * 8;
  const int c = min(8, n - first);
  float acc[4];
  const int64_t row0 = static_cast<int64_t>(b) * a.key_stride + first;
  if (a.fmt == DSA_FMT_BF16) {
    const uint16_t* k = static_cast<const uint16_t*>(a.key_data);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = 0.f;
    for (int j = 0; j < c; ++j) {
      const uint2 v = *reinterpret_cast<const uint2*>(k + (row0 + j) * 128 + lane * 4);
      const float x0 = bf16_bits_to_float(v.x & 0xFFFF), x1 = bf16_bits_to_float(v.x >> 16);
      const float x2 = bf16_bits_to_float(v.y & 0xFFFF), x3 = bf16_bits_to_float(v.y >> 16);
      if (j == 0) {
        acc[0] = x0; acc[1] = x1; acc[2] = x2; acc[3] = x3;
      } else {
        acc[0] = __fadd_rn(acc[0], x0); acc[1] = __fadd_rn(acc[1], x1);
        acc[2] = __fadd_rn(acc[2], x2); acc[3] = __fadd_rn(acc[3], x3);
      }
    }
  } else {
    const uint8_t* k = static_cast<const uint8_t*>(a.key_data);
    for (int j = 0; j < c; ++j) {
      const uint32_t codes = *reinterpret_cast<const uint32_t*>(k + (row0 + j) * 128 + lane * 4);
      const int sc = a.key_scales[(row0 + j) * 4 + (lane >> 3)];
      const float f = __uint_as_float(sc == 0 ? 0x00400000u : static_cast<uint32_t>(sc) << 23);
      // e4m3 -> f16 is exact; f16 -> f32 is exact; times 2^(sc-127) is exact.
      const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>(codes & 0xFFFF), __NV_E4M3);
      const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>(codes >> 16), __NV_E4M3);
      const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
      const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
      const float x0 = f01.x * f, x1 = f01.y * f, x2 = f23.x * f, x3 = f23.y * f;
      if (j == 0) {
        acc[0] = x0; acc[1] = x1; acc[2] = x2; acc[3] = x3;
      } else {
        acc[0] = __fadd_rn(acc[0], x0); acc[1] = __fadd_rn(acc[1], x1);
        acc[2] = __fadd_rn(acc[2], x2); acc[3] = __fadd_rn(acc[3], x3);
      }
    }
  }
  const float cf = static_cast<float>(c);
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] = __fdiv_rn(acc[e], cf);

  const int64_t orow = a.prefill ? b : static_cast<int64_t>(b) * a.out_stride + blk;
  if (a.fmt == DSA_FMT_BF16) {
    uint16_t* o = static_cast<uint16_t*>(a.out_data);
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[0])) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[1])))
                         << 16);
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2])) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[3])))
                         << 16);
    *reinterpret_cast<uint2*>(o + orow * 128 + lane * 4) = make_uint2(lo, hi);
  } else {
    // Group of 32 values = 8 lanes. X = floor(log2(amax)) - 8, clamped to
    // [-127, 127]; an all-zero group takes X = 0.
    float amax = fmaxf(fmaxf(fabsf(acc[0]), fabsf(acc[1])), fmaxf(fabsf(acc[2]), fabsf(acc[3])));
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    int X;
    if (amax == 0.f) {
      X = 0;
    } else {
      const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
      X = (e == 0) ? -127 : max(-127, e - 127 - 8);
    }
    // v * 2^-X is exact (a power-of-two scaling); then round to e4m3,
    // nearest-even, saturating to +-448.
    const int ex = 127 - X;  // biased exponent of 2^-X, in [0, 254]
    const float inv = __uint_as_float(ex == 0 ? 0x00400000u : static_cast<uint32_t>(ex) << 23);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const float2 pr = make_float2(acc[e] * inv, acc[e + 1] * inv);
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
      packed |= static_cast<uint32_t>(q) << (16 * (e >> 1));
    }
    uint8_t* o = static_cast<uint8_t*>(a.out_data);
    *reinterpret_cast<uint32_t*>(o + orow * 128 + lane * 4) = packed;
    if ((lane & 7) == 0) a.out_scales[orow * 4 + (lane >> 3)] = static_cast<uint8_t>(X + 127);
  }
}

}  // namespace

cudaError_t launch_pool(const PoolArgs& a, cudaStream_t s) {
  const int64_t nb_max = (a.max_latents + 7) / 8;
  const bool one = a.tail_only || a.prefill;
  const int warps = one ? 1 : static_cast<int>(nb_max > 0 ? nb_max : 1);
  const int threads = one ? 32 : 256;
  const int wpb = threads / 32;
  dim3 grid((warps + wpb - 1) / wpb, a.B);
  pool_kernel<<<grid, threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
