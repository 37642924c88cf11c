// Router post-processing: one warp per token over fp32 logits.
//
// Sums split-K partial logits (fixed order), adds the router bias, computes
// the gating scores, selects the top-k by (score or logit) + score_bias with
// equal keys resolved to the lower expert index, forms the unbiased weights,
// then applies the p-norm and the scalings.
// Page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"Маршрутизация: как роутер выбирает экспертов" and
// §"Разрешение равенства логитов и квантизация".
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {

struct TopkParams {
  const float* logits;
  int n_partials;
  long long partial_stride;
  const float* b_router;
  const float* score_bias;
  int T, E, k, gating;
  float sig_eps, p_norm;
  int restore;
  float ews;
  int orig_k;
  float* logits_out;
  int32_t* idx;
  float* w;
  int* status;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// true when (ka, ea) ranks before (kb, eb): larger key, or equal key and lower index
__device__ __forceinline__ bool ranks_before(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

template <int NI>
__global__ void __launch_bounds__(256) topk_kernel(const TopkParams p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int E = p.E;
  const long long row = (long long)t * E;

  float lg[NI], key[NI], src[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    float v = 0.f;
    if (e < E) {
      for (int s = 0; s < p.n_partials; ++s) v += p.logits[(long long)s * p.partial_stride + row + e];
      if (p.b_router) v += p.b_router[e];
      if (p.logits_out) p.logits_out[row + e] = v;
    }
    lg[i] = v;
  }

  if (p.gating == MOE_GATING_SIGMOID) {
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] = 1.0f / (1.0f + expf(-lg[i])) + p.sig_eps;
  } else if (p.gating == MOE_GATING_SOFTMAX) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) m = fmaxf(m, lg[i]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      src[i] = (lane + 32 * i < E) ? expf(lg[i] - m) : 0.f;
      s += src[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] *= inv;
  } else {  // topk_softmax: select on logits, weights from the selected logits
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] = lg[i];
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    float kv = src[i];
    if (p.score_bias && e < E) kv += p.score_bias[e];
    key[i] = (e < E && kv == kv) ? kv : -INFINITY;   // NaN never outranks a number
  }

  uint32_t removed = 0;
  int my_e = 0;
  float my_w = 0.f;
  for (int j = 0; j < p.k; ++j) {
    float bk = -INFINITY, bw = 0.f;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((removed >> i) & 1u) && ranks_before(key[i], e, bk, be)) {
        bk = key[i];
        be = e;
        bw = src[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float ow = __shfl_xor_sync(0xffffffffu, bw, o);
      if (ranks_before(ok, oe, bk, be)) {
        bk = ok;
        be = oe;
        bw = ow;
      }
    }
    if (be == INT_MAX) {  // fewer than k experts (cannot happen for a validated config)
      set_status(p.status, MOE_ERR_BOUNDS);
      be = 0;
    }
    if ((be & 31) == lane) removed |= 1u << (be >> 5);
    if (lane == j) {
      my_e = be;
      my_w = bw;
    }
  }

  const bool mine = lane < p.k;
  float w = my_w;
  if (p.gating == MOE_GATING_TOPK_SOFTMAX) {
    const float m = warp_max(mine ? my_w : -FLT_MAX);
    const float ex = mine ? expf(my_w - m) : 0.f;
    w = ex / warp_sum(ex);
  }
  if (p.p_norm > 0.f) {
    float nrm;
    if (p.p_norm == 1.0f) {
      nrm = warp_sum(mine ? fabsf(w) : 0.f);
    } else if (p.p_norm == 2.0f) {
      nrm = sqrtf(warp_sum(mine ? w * w : 0.f));
    } else {
      nrm = powf(warp_sum(mine ? powf(fabsf(w), p.p_norm) : 0.f), 1.0f / p.p_norm);
    }
    w = w / nrm;
  }
  if (p.restore) w *= (float)p.k;
  if (p.ews != 0.f) w *= p.ews;
  if (p.orig_k > 0 && p.orig_k != p.k) w *= sqrtf((float)p.orig_k / (float)p.k);
  if (mine) {
    p.idx[(long long)t * p.k + lane] = my_e;
    p.w[(long long)t * p.k + lane] = w;
  }
}

cudaError_t launch_topk(const float* logits, int n_partials, int64_t partial_stride, const float* b_router,
                        const float* score_bias, int T, int E, int k, int gating, float sig_eps, float p_norm,
                        int restore, float ews, int orig_k, float* logits_out, int32_t* idx, float* w,
                        int* status, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  TopkParams p{logits, n_partials, partial_stride, b_router, score_bias, T, E, k, gating, sig_eps, p_norm,
               restore, ews, orig_k, logits_out, idx, w, status};
  const int warps = 8;
  dim3 grid((T + warps - 1) / warps), block(32 * warps);
  const int ni = (E + 31) / 32;
  if (ni <= 1) topk_kernel<1><<<grid, block, 0, stream>>>(p);
  else if (ni <= 2) topk_kernel<2><<<grid, block, 0, stream>>>(p);
  else if (ni <= 4) topk_kernel<4><<<grid, block, 0, stream>>>(p);
  else if (ni <= 8) topk_kernel<8><<<grid, block, 0, stream>>>(p);
  else if (ni <= 16) topk_kernel<16><<<grid, block, 0, stream>>>(p);
  else if (ni <= 32) topk_kernel<32><<<grid, block, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace moe
