// Router post-processing: one warp per token over fp32 logits.
//
// Adds the router bias, computes the gating scores, selects the top-k by
// (score or logit) + score_bias with equal keys resolved to the lower expert
// index, forms the unbiased weights, then applies the p-norm and the scalings.
// Selection: tau = k-th largest per-lane maximum bounds the k-th key from
// below, the keys >= tau (usually about k of them) are compacted with ballots
// and ordered by one warp bitonic sort; more than 32 candidates (many equal
// keys) fall back to k rounds of warp arg-max over all keys.  Split-K partial
// logits are summed as they are loaded, in slice order.
// Page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"Маршрутизация: как роутер выбирает экспертов" and
// §"Разрешение равенства логитов и квантизация".
#include <algorithm>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {

struct TopkParams {
  const float* logits;         // n_partials slices, partial_stride floats apart (split-K), summed in order
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

constexpr int kTopkWarps = 8;
constexpr int kCand = 32;  // candidates one warp sorts in registers

// One compare-exchange step of a warp bitonic sort in rank order (best first).
__device__ __forceinline__ void bitonic_step(float& k, int& e, float& w, int lane, int size, int stride) {
  const float ok = __shfl_xor_sync(0xffffffffu, k, stride);
  const int oe = __shfl_xor_sync(0xffffffffu, e, stride);
  const float ow = __shfl_xor_sync(0xffffffffu, w, stride);
  const bool lower = (lane & stride) == 0;
  const bool first_half_best = ((lane & size) == 0);   // this block sorts best-first
  const bool other_first = ranks_before(ok, oe, k, e);
  // the lower lane of a best-first block keeps the better element, the upper one the worse
  const bool take = (lower == first_half_best) ? other_first : (!other_first && !(ok == k && oe == e));
  if (take) {
    k = ok;
    e = oe;
    w = ow;
  }
}

template <int NI>
__global__ void __launch_bounds__(32 * kTopkWarps) topk_kernel(const TopkParams p) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  __shared__ float s_key[kTopkWarps][kCand];
  __shared__ int s_e[kTopkWarps][kCand];
  __shared__ float s_w[kTopkWarps][kCand];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= p.T) return;
  const int E = p.E;
  const long long row = (long long)t * E;

  // all NI loads of a lane are independent and issue back to back; split-K partial slices are
  // added in slice order
  float lg[NI], key[NI], src[NI];
  const float* lrow = p.logits + row;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? __ldg(lrow + e) : 0.f;
  }
  for (int sl = 1; sl < p.n_partials; ++sl) {
    const float* prow = lrow + sl * p.partial_stride;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (e < E) lg[i] += __ldg(prow + e);
    }
  }
  if (p.b_router) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (e < E) lg[i] += __ldg(p.b_router + e);
    }
  }
  if (p.logits_out) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      if (e < E) p.logits_out[row + e] = lg[i];
    }
  }

  // scores (fast exp / reciprocal: a few ulp, far below the selection's fp32 noise)
  if (p.gating == MOE_GATING_SIGMOID) {
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] = __fdividef(1.0f, 1.0f + __expf(-lg[i])) + p.sig_eps;
  } else if (p.gating == MOE_GATING_SOFTMAX) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < E) m = fmaxf(m, lg[i]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      src[i] = (lane + 32 * i < E) ? __expf(lg[i] - m) : 0.f;
      s += src[i];
    }
    s = warp_sum(s);
    const float inv = __fdividef(1.0f, s);
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] *= inv;
  } else {  // topk_softmax: select on logits, weights from the selected logits
#pragma unroll
    for (int i = 0; i < NI; ++i) src[i] = lg[i];
  }
  float lane_max = -INFINITY;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    float kv = src[i];
    if (p.score_bias && e < E) kv += __ldg(p.score_bias + e);
    key[i] = (e < E && kv == kv) ? kv : -INFINITY;   // NaN never outranks a number
    lane_max = fmaxf(lane_max, key[i]);
  }

  // tau = k-th largest lane maximum.  At least k keys are >= tau, so every key of
  // the top k is >= tau: the candidates {key >= tau} contain the answer exactly.
  float tau;
  {
    float v = lane_max;
    int dummy_e = lane;
    float dummy_w = 0.f;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) bitonic_step(v, dummy_e, dummy_w, lane, size, stride);
    tau = __shfl_sync(0xffffffffu, v, p.k - 1);
  }

  // compact the candidates of the warp into shared memory, in (slot, lane) order
  const unsigned lt = (1u << lane) - 1u;
  int n_cand = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    const bool c = e < E && key[i] >= tau;
    const unsigned b = __ballot_sync(0xffffffffu, c);
    if (c) {
      const int pos = n_cand + __popc(b & lt);
      if (pos < kCand) {
        s_key[warp][pos] = key[i];
        s_e[warp][pos] = e;
        s_w[warp][pos] = src[i];
      }
    }
    n_cand += __popc(b);
  }
  __syncwarp();

  int my_e = 0;
  float my_w = 0.f;
  if (n_cand <= kCand) {
    // one candidate per lane, then a warp bitonic sort: lanes 0..k-1 hold the answer
    float ck = -INFINITY, cw = 0.f;
    int ce = INT_MAX;
    if (lane < n_cand) {
      ck = s_key[warp][lane];
      ce = s_e[warp][lane];
      cw = s_w[warp][lane];
    }
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) bitonic_step(ck, ce, cw, lane, size, stride);
    my_e = ce;
    my_w = cw;
  } else {
    // many equal keys at the threshold: k rounds of warp arg-max over all keys
    uint32_t removed = 0;
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
      if ((be & 31) == lane) removed |= 1u << (be >> 5);
      if (lane == j) {
        my_e = be;
        my_w = bw;
      }
    }
  }
  const bool mine = lane < p.k;
  if (mine && (my_e < 0 || my_e >= E)) {  // fewer than k experts (cannot happen for a validated config)
    set_status(p.status, MOE_ERR_BOUNDS);
    my_e = 0;
  }

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

// logits[t, e] = sum over s of partials[s, t, e], in a fixed order (split-K router GEMM).
__global__ void __launch_bounds__(256) sum_partials_kernel(const float4* __restrict__ part, int splits,
                                                            long long n4, float4* __restrict__ out) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[(long long)s * n4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    out[i] = a;
  }
}

cudaError_t launch_sum_slices_f32(const float* part, int splits, long long n, float* out, cudaStream_t st) {
  const long long n4 = n / 4;
  if (n4 <= 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>((n4 + 255) / 256, 2048);
  launch_pdl(sum_partials_kernel, blocks, 256, 0, st, reinterpret_cast<const float4*>(part), splits, n4,
                                              reinterpret_cast<float4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int n_partials, int64_t partial_stride, const float* b_router,
                        const float* score_bias, int T, int E, int k, int gating, float sig_eps, float p_norm,
                        int restore, float ews, int orig_k, float* logits_out, int32_t* idx, float* w,
                        int* status, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  // split-K: up to kTopkFusedSlices slices the kernel adds them itself as it loads; more (few
  // tokens, a deep split) are first summed by a grid-wide kernel into the slice after the last
  // one, which the caller's buffer then holds
  if (n_partials > kTopkFusedSlices) {
    float* sum = const_cast<float*>(logits) + (int64_t)n_partials * partial_stride;
    const long long n4 = partial_stride / 4;
    const int blocks = (int)std::min<long long>((n4 + 255) / 256, 2048);
    launch_pdl(sum_partials_kernel, blocks, 256, 0, stream, reinterpret_cast<const float4*>(logits), n_partials, n4,
               reinterpret_cast<float4*>(sum));
    logits = sum;
    n_partials = 1;
  }
  TopkParams p{logits, std::max(1, n_partials), (long long)partial_stride, b_router, score_bias, T, E, k, gating,
               sig_eps, p_norm, restore, ews, orig_k, logits_out, idx, w, status};
  dim3 grid((T + kTopkWarps - 1) / kTopkWarps), block(32 * kTopkWarps);
  const int ni = (E + 31) / 32;
  if (ni <= 1) launch_pdl(topk_kernel<1>, grid, block, 0, stream, p);
  else if (ni <= 2) launch_pdl(topk_kernel<2>, grid, block, 0, stream, p);
  else if (ni <= 4) launch_pdl(topk_kernel<4>, grid, block, 0, stream, p);
  else if (ni <= 8) launch_pdl(topk_kernel<8>, grid, block, 0, stream, p);
  else if (ni <= 16) launch_pdl(topk_kernel<16>, grid, block, 0, stream, p);
  else if (ni <= 28) launch_pdl(topk_kernel<28>, grid, block, 0, stream, p);
  else if (ni <= 32) launch_pdl(topk_kernel<32>, grid, block, 0, stream, p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace moe
