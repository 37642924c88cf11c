// Load-balancing counters: per-expert accumulation, the max / mean imbalance
// metric and the sign-based score-bias correction (page "Как устроен Olmo-core 3:
// обучение больших MoE-моделей", §"Счётчики и bias-корректировка").
// E <= 1024: one block, thread e owns expert e.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ long long block_sum_ll(long long v, long long* s_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_buf[warp] = v;
  __syncthreads();
  long long t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_buf[w];
  __syncthreads();
  return t;
}

__device__ long long block_max_ll(long long v, long long* s_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) s_buf[warp] = v;
  __syncthreads();
  long long t = s_buf[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = max(t, s_buf[w]);
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(1024) accumulate_counts_kernel(const int32_t* __restrict__ counts, int E,
                                                                  int64_t* __restrict__ accum) {
  const int e = threadIdx.x;
  if (e < E) accum[e] += counts[e];
}

// imbalance = max(counts) / mean(counts) = max * E / sum (NaN when the sum is zero)
template <typename C>
__global__ void __launch_bounds__(1024) load_imbalance_kernel(const C* __restrict__ counts, int E,
                                                               float* __restrict__ out) {
  __shared__ long long s_buf[32];
  const int e = threadIdx.x;
  const long long c = e < E ? (long long)counts[e] : 0;
  const long long sum = block_sum_ll(c, s_buf);
  const long long mx = block_max_ll(e < E ? c : LLONG_MIN, s_buf);
  if (e == 0) *out = sum > 0 ? (float)((double)mx * (double)E / (double)sum) : nanf("");
}

// score_bias[e] += gamma * sign(mean - accum[e]); the sign is taken exactly as
// sign(sum - E * accum[e]); then accum is zeroed.
__global__ void __launch_bounds__(1024) score_bias_update_kernel(int64_t* __restrict__ accum, int E, float gamma,
                                                                  float* __restrict__ score_bias) {
  __shared__ long long s_buf[32];
  const int e = threadIdx.x;
  const long long a = e < E ? accum[e] : 0;
  const long long sum = block_sum_ll(a, s_buf);
  if (e < E) {
    const long long d = sum - (long long)E * a;
    const float sgn = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
    score_bias[e] = score_bias[e] + gamma * sgn;
    accum[e] = 0;
  }
}

cudaError_t launch_accumulate_counts(const int32_t* counts, int E, int64_t* accum, cudaStream_t st) {
  accumulate_counts_kernel<<<1, 1024, 0, st>>>(counts, E, accum);
  return cudaGetLastError();
}

cudaError_t launch_load_imbalance(const void* counts, int is64, int E, float* out, cudaStream_t st) {
  if (is64) load_imbalance_kernel<int64_t><<<1, 1024, 0, st>>>(static_cast<const int64_t*>(counts), E, out);
  else load_imbalance_kernel<int32_t><<<1, 1024, 0, st>>>(static_cast<const int32_t*>(counts), E, out);
  return cudaGetLastError();
}

cudaError_t launch_score_bias_update(int64_t* accum, int E, float gamma, float* score_bias, cudaStream_t st) {
  score_bias_update_kernel<<<1, 1024, 0, st>>>(accum, E, gamma, score_bias);
  return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_accumulate_counts(const int32_t* counts, int32_t num_experts, int64_t* accum, moe_stream_t stream) {
  if (!counts || !accum || num_experts < 1) return MOE_ERR_INVALID_ARG;
  if (num_experts > 1024) return MOE_ERR_UNSUPPORTED;
  return launch_accumulate_counts(counts, num_experts, accum, (cudaStream_t)stream) == cudaSuccess ? MOE_OK
                                                                                                   : MOE_ERR_CUDA;
}

int moe_load_imbalance(const void* counts, int32_t counts_are_int64, int32_t num_experts, float* imbalance,
                       moe_stream_t stream) {
  if (!counts || !imbalance || num_experts < 1) return MOE_ERR_INVALID_ARG;
  if (num_experts > 1024) return MOE_ERR_UNSUPPORTED;
  return launch_load_imbalance(counts, counts_are_int64, num_experts, imbalance, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_score_bias_update(int64_t* accum, int32_t num_experts, float bias_gamma, float* score_bias,
                          moe_stream_t stream) {
  if (!accum || !score_bias || num_experts < 1 || !std::isfinite(bias_gamma)) return MOE_ERR_INVALID_ARG;
  if (num_experts > 1024) return MOE_ERR_UNSUPPORTED;
  return launch_score_bias_update(accum, num_experts, bias_gamma, score_bias, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

}  // extern "C"
