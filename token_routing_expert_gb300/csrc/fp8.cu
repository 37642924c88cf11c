// Rowwise FP8 (e4m3) quantisation for the experts' operands (page "Как устроен
// Olmo-core 3: обучение больших MoE-моделей", §"Rowwise FP8 и MXFP8": the
// experts run on pre-quantised weights and quantised activations).
// Each row gets one float32 scale, amax / 448 (448 = the largest e4m3 value;
// 1 for a zero row); an element's code is e4m3(x / scale) with the division
// correctly rounded in float32 and the conversion rounding to nearest-even,
// saturating at +-448.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) quantize_rowwise_e4m3_kernel(const uint4* __restrict__ x, long long rows,
                                                                     int vec, uint2* __restrict__ q,
                                                                     float* __restrict__ scale) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint4* row = x + r * vec;
  float amax = 0.f;
  for (int c = lane; c < vec; c += 32) {
    const uint4 v = row[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint2* out = q + r * vec;
  for (int c = lane; c < vec; c += 32) {
    const uint4 v = row[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 lo = make_float2(__fdiv_rn(bf16_lo(w[2 * h]), s), __fdiv_rn(bf16_hi(w[2 * h]), s));
      const float2 hi = make_float2(__fdiv_rn(bf16_lo(w[2 * h + 1]), s), __fdiv_rn(bf16_hi(w[2 * h + 1]), s));
      const uint32_t a = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
      const uint32_t b = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
      packed[h] = (a & 0xFFFFu) | (b << 16);
    }
    out[c] = make_uint2(packed[0], packed[1]);
  }
  if (lane == 0) scale[r] = s;
}

cudaError_t launch_quantize_rowwise_e4m3(const void* x, long long rows, int cols, void* q, float* scale,
                                         cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 8) return cudaErrorInvalidValue;
  const long long blocks = (rows + 7) / 8;
  launch_pdl(quantize_rowwise_e4m3_kernel, (unsigned)blocks, 256, 0, st, static_cast<const uint4*>(x), rows, cols / 8,
                                                                 static_cast<uint2*>(q), scale);
  return cudaGetLastError();
}

// MXFP8 (OCP microscaling) quantisation, §"Rowwise FP8 и MXFP8": each block of 32 consecutive
// values of a row shares the scale 2^(e - 127), e = floor(log2 amax) - 8 + 127 clamped to [0, 254]
// (e = 0 for an all-zero block), stored as the byte e (E8M0); a value's code is e4m3(v * 2^(127 - e)),
// the product exact in float32 (a power of two), rounded to nearest-even and saturating at +-448.
// A thread per block: 64 bytes of bf16 in, 32 code bytes and one scale byte out.
__global__ void __launch_bounds__(256) quantize_mx_e4m3_kernel(const uint4* __restrict__ x, long long rows, int nb,
                                                                uint4* __restrict__ q, uint8_t* __restrict__ scales,
                                                                int scale_ld) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= rows * nb) return;
  const long long r = b / nb;
  const int kb = (int)(b - r * nb);
  uint32_t w[16], out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = x[b * 4 + i];
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
  const uint32_t e = mx_quantize_block(w, out);
  q[b * 2] = make_uint4(out[0], out[1], out[2], out[3]);
  q[b * 2 + 1] = make_uint4(out[4], out[5], out[6], out[7]);
  scales[r * scale_ld + kb] = (uint8_t)e;
}

cudaError_t launch_quantize_mx_e4m3(const void* x, long long rows, int cols, void* q, void* scales, int scale_ld,
                                    cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 32 || scale_ld < cols / 32) return cudaErrorInvalidValue;
  const long long n = rows * (cols / 32);
  launch_pdl(quantize_mx_e4m3_kernel, (unsigned)((n + 255) / 256), 256, 0, st, static_cast<const uint4*>(x), rows,
             cols / 32, static_cast<uint4*>(q), static_cast<uint8_t*>(scales), scale_ld);
  return cudaGetLastError();
}

// dst[p] = src[gather_idx[p]] for e4m3 rows (row_bytes, a multiple of 16) and their scales;
// a padding slot (-1, capacity mode) gets a zero row and scale 1.
__global__ void __launch_bounds__(256) gather_rows_e4m3_kernel(const uint4* __restrict__ src,
                                                                const float* __restrict__ src_scale,
                                                                const int32_t* __restrict__ gather_idx, int R, int T,
                                                                int vec, uint4* __restrict__ dst,
                                                                float* __restrict__ dst_scale, int allow_padding,
                                                                int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= R) return;
  const int t = gather_idx[p];
  uint4* d = dst + p * vec;
  if (t < 0 || t >= T) {
    if (allow_padding && t == -1) {
      for (int c = lane; c < vec; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) dst_scale[p] = 1.0f;
    } else if (lane == 0) {
      set_status(status, MOE_ERR_BOUNDS);
    }
    return;
  }
  const uint4* s = src + (long long)t * vec;
  for (int c0 = lane; c0 < vec; c0 += 256) {   // eight 16-byte loads in flight per lane
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) v[i] = __ldg(s + c0 + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) d[c0 + 32 * i] = v[i];
  }
  if (lane == 0) dst_scale[p] = src_scale[t];
}

cudaError_t launch_gather_rows_e4m3(const void* src, const float* src_scale, const int32_t* gather_idx, int R, int T,
                                    int row_bytes, void* dst, float* dst_scale, int allow_padding, int* status,
                                    cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  if (row_bytes % 16) return cudaErrorInvalidValue;
  launch_pdl(gather_rows_e4m3_kernel, (R + 7) / 8, 256, 0, st, static_cast<const uint4*>(src), src_scale, gather_idx, R, T,
                                                       row_bytes / 16, static_cast<uint4*>(dst), dst_scale,
                                                       allow_padding, status);
  return cudaGetLastError();
}

// dst[p] = src[gather_idx[p]] for MXFP8 rows: the codes (vec 16-byte words) and the block scales
// (svec 32-bit words); a padding slot (-1, capacity mode) gets zero codes and scales 2^0 (byte 127).
__global__ void __launch_bounds__(256) gather_rows_mx_kernel(const uint4* __restrict__ src,
                                                             const uint32_t* __restrict__ src_scale,
                                                             const int32_t* __restrict__ gather_idx, int R, int T,
                                                             int vec, int svec, uint4* __restrict__ dst,
                                                             uint32_t* __restrict__ dst_scale, int allow_padding,
                                                             int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= R) return;
  const int t = gather_idx[p];
  uint4* d = dst + p * vec;
  uint32_t* ds = dst_scale + p * svec;
  if (t < 0 || t >= T) {
    if (allow_padding && t == -1) {
      for (int c = lane; c < vec; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
      for (int c = lane; c < svec; c += 32) ds[c] = 0x7F7F7F7Fu;
    } else if (lane == 0) {
      set_status(status, MOE_ERR_BOUNDS);
    }
    return;
  }
  const uint4* s = src + (long long)t * vec;
  for (int c0 = lane; c0 < vec; c0 += 256) {   // eight 16-byte loads in flight per lane
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) v[i] = __ldg(s + c0 + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) d[c0 + 32 * i] = v[i];
  }
  const uint32_t* ss = src_scale + (long long)t * svec;
  for (int c = lane; c < svec; c += 32) ds[c] = __ldg(ss + c);
}

cudaError_t launch_gather_rows_mx(const void* src, const void* src_scale, const int32_t* gather_idx, int R, int T,
                                  int row_bytes, int scale_ld, void* dst, void* dst_scale, int allow_padding,
                                  int* status, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  if (row_bytes % 16 || scale_ld % 4) return cudaErrorInvalidValue;
  launch_pdl(gather_rows_mx_kernel, (R + 7) / 8, 256, 0, st, static_cast<const uint4*>(src),
             static_cast<const uint32_t*>(src_scale), gather_idx, R, T, row_bytes / 16, scale_ld / 4,
             static_cast<uint4*>(dst), static_cast<uint32_t*>(dst_scale), allow_padding, status);
  return cudaGetLastError();
}

}  // namespace moe

extern "C" int moe_quantize_rowwise_fp8(const void* x, int64_t rows, int32_t cols, void* codes, float* scales,
                                        moe_stream_t stream) {
  if (rows < 0 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (cols % 16) return MOE_ERR_UNSUPPORTED;
  return moe::launch_quantize_rowwise_e4m3(x, rows, cols, codes, scales, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
