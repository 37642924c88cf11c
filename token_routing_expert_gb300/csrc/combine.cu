// Weighted combine, RMSNorm and split-K reduction (HBM-bound row kernels).
//
// combine:  z[t] = sum_j w[t, j] * y[scatter_idx[t*k + j]], y bf16 or fp32, fp32 accumulate,
//           bf16 store (page "Как устроен Olmo-core 3: обучение больших
//           MoE-моделей", §"Пересылка токенов между экспертами": restore the
//           original order by the saved indices).
// combine + RMSNorm (latent layer): the bf16-rounded z of the row is kept in
//           shared memory, then n = z / sqrt(mean(z^2) + eps) * gain in fp32,
//           stored bf16 (§"Латентная проекция экспертов": norm, then cast to
//           the up-projection's dtype).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRowWarps = 4;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Scales the bf16 row held in `zs` (vec 16-byte vectors) by inv * gain and stores it.
__device__ __forceinline__ void store_normalised(const uint4* zs, int vec, float inv, const uint4* gain,
                                                 uint4* dst, int lane) {
  for (int c = lane; c < vec; c += 32) {
    float f[8];
    unpack8(zs[c], f);
    if (gain) {
      float g[8];
      unpack8(gain[c], g);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = f[i] * inv * g[i];
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = f[i] * inv;
    }
    dst[c] = pack8(f);
  }
}

// Y32: the expert rows are fp32 (two 16-byte vectors per 8 values) instead of bf16.
template <bool RMS, bool Y32 = false>
__global__ void __launch_bounds__(32 * kRowWarps)
    combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ scatter_idx, const float* __restrict__ w,
                   int T, int k, int vec, int R, float eps, const uint4* __restrict__ gain, uint4* __restrict__ z,
                   int allow_dropped, int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  extern __shared__ uint4 zs_all[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const long long t = (long long)blockIdx.x * kRowWarps + warp;
  if (t >= T) return;
  // lane j < k holds assignment j's row and weight
  int my_p = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_p = scatter_idx[t * k + lane];
    my_w = w ? w[t * k + lane] : 1.0f;   // no weights: plain sum of the k rows
    if (my_p < 0 || my_p >= R) {
      if (!(allow_dropped && my_p == -1)) set_status(status, MOE_ERR_BOUNDS);  // -1: dropped, adds nothing
      my_p = 0;
      my_w = 0.f;
    }
  }
  uint4* zs = zs_all + (long long)warp * vec;
  uint4* dst = z + t * vec;
  float sumsq = 0.f;
  // every lane runs every iteration (the shuffles need the whole warp); loads are guarded.
  // The k rows are read eight at a time, all eight loads issued before the first is used,
  // and accumulated in ascending j.
  for (int c0 = 0; c0 < vec; c0 += 32) {
    const int c = c0 + lane;
    const bool active = c < vec;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (Y32) {
      // fp32 rows: four at a time (two 16-byte loads each), in ascending j
      for (int j0 = 0; j0 < k; j0 += 4) {
        uint4 v[4][2];
        float wj[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int p = __shfl_sync(0xffffffffu, my_p, (j0 + jj) & 31);
          wj[jj] = __shfl_sync(0xffffffffu, my_w, (j0 + jj) & 31);
          v[jj][0] = v[jj][1] = make_uint4(0u, 0u, 0u, 0u);
          if (active && j0 + jj < k) {
            const uint4* src = y + ((long long)p * vec + c) * 2;
            v[jj][0] = __ldcs(src);
            v[jj][1] = __ldcs(src + 1);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (j0 + jj >= k) break;
          const float f[8] = {__uint_as_float(v[jj][0].x), __uint_as_float(v[jj][0].y), __uint_as_float(v[jj][0].z),
                              __uint_as_float(v[jj][0].w), __uint_as_float(v[jj][1].x), __uint_as_float(v[jj][1].y),
                              __uint_as_float(v[jj][1].z), __uint_as_float(v[jj][1].w)};
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[jj], f[i], acc[i]);
        }
      }
    } else {
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 v[8];
        float wj[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int p = __shfl_sync(0xffffffffu, my_p, (j0 + jj) & 31);
          wj[jj] = __shfl_sync(0xffffffffu, my_w, (j0 + jj) & 31);
          v[jj] = make_uint4(0u, 0u, 0u, 0u);
          if (active && j0 + jj < k) v[jj] = __ldcs(y + (long long)p * vec + c);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj >= k) break;
          float f[8];
          unpack8(v[jj], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[jj], f[i], acc[i]);
        }
      }
    }
    if (!active) continue;
    const uint4 packed = pack8(acc);
    if (RMS) {
      zs[c] = packed;
      float f[8];
      unpack8(packed, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) sumsq = fmaf(f[i], f[i], sumsq);
    } else {
      dst[c] = packed;
    }
  }
  if (RMS) {
    sumsq = warp_sum_f(sumsq);
    const float inv = rsqrtf(sumsq / (float)(vec * 8) + eps);
    __syncwarp();
    store_normalised(zs, vec, inv, gain, dst, lane);
  }
}

__global__ void __launch_bounds__(32 * kRowWarps)
    rmsnorm_kernel(const uint4* __restrict__ z, int T, int vec, float eps, const uint4* __restrict__ gain,
                   uint4* __restrict__ out) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const uint4* row = z + t * vec;
  float sumsq = 0.f;
  for (int c = lane; c < vec; c += 32) {
    float f[8];
    unpack8(row[c], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) sumsq = fmaf(f[i], f[i], sumsq);
  }
  sumsq = warp_sum_f(sumsq);
  const float inv = rsqrtf(sumsq / (float)(vec * 8) + eps);
  store_normalised(row, vec, inv, gain, out + t * vec, lane);
}

__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4* __restrict__ part, int splits,
                                                             long long slice4, uint2* __restrict__ out) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < slice4;
       i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[(long long)s * slice4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    out[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  }
}

cudaError_t launch_combine(const void* y, const int32_t* scatter_idx, const float* w, int T, int k, int L, int R,
                           int rms, float eps, const void* gain, void* z, int allow_dropped, int* status,
                           cudaStream_t stream, int y_f32) {
  if (T <= 0) return cudaSuccess;
  const int vec = L / 8;
  const dim3 grid((T + kRowWarps - 1) / kRowWarps), block(32 * kRowWarps);
  if (y_f32) {
    if (rms) return cudaErrorInvalidValue;
    launch_pdl(combine_kernel<false, true>, grid, block, 0, stream, static_cast<const uint4*>(y), scatter_idx, w, T, k,
                                                      vec, R, eps, nullptr, static_cast<uint4*>(z), allow_dropped, status);
    return cudaGetLastError();
  }
  if (rms) {
    const size_t sm = (size_t)kRowWarps * vec * sizeof(uint4);
    if (sm > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(combine_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      if (e != cudaSuccess) return e;
    }
    launch_pdl(combine_kernel<true>, grid, block, sm, stream, static_cast<const uint4*>(y), scatter_idx, w, T, k, vec, R,
                                                      eps, static_cast<const uint4*>(gain), static_cast<uint4*>(z),
                                                      allow_dropped, status);
  } else {
    launch_pdl(combine_kernel<false>, grid, block, 0, stream, static_cast<const uint4*>(y), scatter_idx, w, T, k, vec, R,
                                                      eps, nullptr, static_cast<uint4*>(z), allow_dropped, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* z, int T, int L, float eps, const void* gain, void* out, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  launch_pdl(rmsnorm_kernel, (T + kRowWarps - 1) / kRowWarps, 32 * kRowWarps, 0, stream, 
      static_cast<const uint4*>(z), T, L / 8, eps, static_cast<const uint4*>(gain), static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_splitk_reduce_bf16(const float* partials, int splits, int64_t slice, void* out,
                                      cudaStream_t stream) {
  const long long slice4 = slice / 4;
  if (slice4 <= 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>((slice4 + 255) / 256, 4096);
  launch_pdl(splitk_reduce_kernel, blocks, 256, 0, stream, reinterpret_cast<const float4*>(partials), splits, slice4,
                                                   static_cast<uint2*>(out));
  return cudaGetLastError();
}

}  // namespace moe
