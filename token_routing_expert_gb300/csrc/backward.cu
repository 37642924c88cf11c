// Backward of the grouped SwiGLU experts and of the weighted combine (training).
//
// Page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"SwiGLU с квантизацией": the SwiGLU backward splits the last dimension into
// up and gate, computes the sigmoid, gate * sigmoid, its derivative and the two
// gradients in float32 and concatenates them back in the input dtype.
//
// Row kernels here are HBM-bound; the contractions run on the tcgen05 GEMM:
//   UG  = Xp W_up_gate^T            (recomputed pre-activations, bf16)
//   dH  = dY W_out                  (B = per-expert transpose of W_out)
//   dXp = dUG W_up_gate             (B = per-expert transpose of W_up_gate)
//   dW_out[e]     = dY_e^T H_e      (K-grouped over the expert's rows)
//   dW_up_gate[e] = dUG_e^T Xp_e    (K-grouped)
// The K-grouped GEMMs read K-major copies dY^T, H^T, dUG^T, Xp^T whose
// expert row ranges start on 64-column boundaries, zero-padded.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// out[e] = in[e]^T for in (E, A, B) -> out (E, B, A), bf16; A, B multiples of 32.
__global__ void __launch_bounds__(256) transpose_experts_kernel(const uint16_t* __restrict__ in, int A, int B,
                                                                 uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[32][33];
  const long long e = blockIdx.z;
  const int b0 = blockIdx.x * 32, a0 = blockIdx.y * 32;
  const uint16_t* src = in + e * (long long)A * B;
  uint16_t* dst = out + e * (long long)A * B;
  for (int i = threadIdx.y; i < 32; i += 8) tile[i][threadIdx.x] = src[(long long)(a0 + i) * B + b0 + threadIdx.x];
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) dst[(long long)(b0 + i) * A + a0 + threadIdx.x] = tile[threadIdx.x][i];
}

cudaError_t launch_transpose_experts(const void* in, int E, int A, int B, void* out, cudaStream_t st) {
  if ((A % 32) || (B % 32)) return cudaErrorInvalidValue;
  dim3 grid(B / 32, A / 32, E), block(32, 8);
  transpose_experts_kernel<<<grid, block, 0, st>>>(static_cast<const uint16_t*>(in), A, B,
                                                   static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

// XT[c][col] for col in [0, 64 * k_off[E]): expert e's columns start at 64 * k_off[e];
// its r-th column is row off[e] + r of X (rows x C) while r < off[e+1] - off[e], zero after.
__global__ void __launch_bounds__(256) group_transpose_kernel(const uint16_t* __restrict__ X, int C,
                                                               const int32_t* __restrict__ off,
                                                               const int32_t* __restrict__ k_off, int E,
                                                               long long ld_out, uint16_t* __restrict__ XT) {
  __shared__ uint16_t tile[32][33];
  __shared__ int s_src[32];
  const long long col0 = (long long)blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  if (col0 >= 64ll * k_off[E]) return;
  if (threadIdx.y == 0) {
    const long long col = col0 + threadIdx.x;
    // expert of this column: last e with 64 * k_off[e] <= col
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (64ll * k_off[mid] <= col) lo = mid; else hi = mid - 1;
    }
    const long long r = col - 64ll * k_off[lo];
    s_src[threadIdx.x] = r < (long long)(off[lo + 1] - off[lo]) ? off[lo] + (int)r : -1;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int src = s_src[i];
    tile[i][threadIdx.x] = src >= 0 ? X[(long long)src * C + c0 + threadIdx.x] : (uint16_t)0;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) XT[(long long)(c0 + i) * ld_out + col0 + threadIdx.x] = tile[threadIdx.x][i];
}

cudaError_t launch_group_transpose(const void* X, int C, const int32_t* off, const int32_t* k_off, int E,
                                   long long max_cols, long long ld_out, void* XT, cudaStream_t st) {
  if (C % 32) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((max_cols + 31) / 32), C / 32), block(32, 8);
  group_transpose_kernel<<<grid, block, 0, st>>>(static_cast<const uint16_t*>(X), C, off, k_off, E, ld_out,
                                                 static_cast<uint16_t*>(XT));
  return cudaGetLastError();
}

// From UG = [u | g] (rows x 2h) and dH (rows x h): H = silu(g) u, dU = dH silu(g),
// dG = dH u silu'(g), silu'(g) = s (1 + g (1 - s)), s = sigmoid(g); fp32, stored bf16.
__global__ void __launch_bounds__(256) swiglu_backward_kernel(const uint4* __restrict__ UG, const uint4* __restrict__ dH,
                                                               long long rows, int h8, uint4* __restrict__ dUG,
                                                               uint4* __restrict__ H) {
  const long long n = rows * h8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long p = i / h8;
    const int c = (int)(i - p * h8);
    const uint4 uv = UG[p * 2 * h8 + c], gv = UG[p * 2 * h8 + h8 + c], dv = dH[p * h8 + c];
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
    uint32_t du[4], dg[4], hh[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float u[2] = {bf16_lo(uw[q]), bf16_hi(uw[q])}, g[2] = {bf16_lo(gw[q]), bf16_hi(gw[q])};
      float d[2] = {bf16_lo(dw[q]), bf16_hi(dw[q])}, ru[2], rg[2], rh[2];
#pragma unroll
      for (int z = 0; z < 2; ++z) {
        const float s = 1.0f / (1.0f + expf(-g[z]));
        const float si = g[z] * s;
        rh[z] = si * u[z];
        ru[z] = d[z] * si;
        rg[z] = d[z] * u[z] * (s * (1.0f + g[z] * (1.0f - s)));
      }
      du[q] = pack_bf16x2(ru[0], ru[1]);
      dg[q] = pack_bf16x2(rg[0], rg[1]);
      hh[q] = pack_bf16x2(rh[0], rh[1]);
    }
    dUG[p * 2 * h8 + c] = make_uint4(du[0], du[1], du[2], du[3]);
    dUG[p * 2 * h8 + h8 + c] = make_uint4(dg[0], dg[1], dg[2], dg[3]);
    H[p * h8 + c] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
  }
}

cudaError_t launch_swiglu_backward(const void* UG, const void* dH, long long rows, int h, void* dUG, void* H,
                                   cudaStream_t st) {
  const long long n = rows * (h / 8);
  if (n <= 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>((n + 255) / 256, 8192);
  swiglu_backward_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(UG), static_cast<const uint4*>(dH), rows,
                                                 h / 8, static_cast<uint4*>(dUG), static_cast<uint4*>(H));
  return cudaGetLastError();
}

// Warp per token: dy[p] = w[t, j] dz[t] (bf16) and dw[t, j] = <dz[t], y[p]> (fp32) for each
// assignment with a row p (p = -1: dropped, dw = 0).
__global__ void __launch_bounds__(128) combine_backward_kernel(const uint4* __restrict__ dz, const uint4* __restrict__ y,
                                                                const int32_t* __restrict__ scatter_idx,
                                                                const float* __restrict__ w, int T, int k, int vec,
                                                                int rows, uint4* __restrict__ dy,
                                                                float* __restrict__ dw, int* status) {
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const uint4* dzr = dz + t * vec;
  for (int j = 0; j < k; ++j) {
    const int p = scatter_idx[t * k + j];
    const float wj = w[t * k + j];
    if (p < 0 || p >= rows) {
      if (p != -1 && lane == 0) set_status(status, MOE_ERR_BOUNDS);
      if (lane == 0) dw[t * k + j] = 0.f;
      continue;
    }
    float dot = 0.f;
    for (int c = lane; c < vec; c += 32) {
      const uint4 a = dzr[c], b = y[(long long)p * vec + c];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a0 = bf16_lo(aw[q]), a1 = bf16_hi(aw[q]);
        dot = fmaf(a0, bf16_lo(bw[q]), dot);
        dot = fmaf(a1, bf16_hi(bw[q]), dot);
        o[q] = pack_bf16x2(wj * a0, wj * a1);
      }
      dy[(long long)p * vec + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) dw[t * k + j] = dot;
  }
}

cudaError_t launch_combine_backward(const void* dz, const void* y, const int32_t* scatter_idx, const float* w, int T,
                                    int k, int L, int rows, void* dy, float* dw, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  combine_backward_kernel<<<(T + 3) / 4, 128, 0, st>>>(static_cast<const uint4*>(dz), static_cast<const uint4*>(y),
                                                       scatter_idx, w, T, k, L / 8, rows, static_cast<uint4*>(dy), dw,
                                                       status);
  return cudaGetLastError();
}

// Rows p whose gather index is -1 (capacity padding) are set to zero.
__global__ void __launch_bounds__(256) zero_padding_rows_kernel(const int32_t* __restrict__ gather_idx, int rows,
                                                                 int vec, uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= rows || gather_idx[p] != -1) return;
  for (int c = lane; c < vec; c += 32) dst[p * vec + c] = make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t launch_zero_padding_rows(const int32_t* gather_idx, int rows, int cols, void* dst, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  zero_padding_rows_kernel<<<(rows + 7) / 8, 256, 0, st>>>(gather_idx, rows, cols / 8, static_cast<uint4*>(dst));
  return cudaGetLastError();
}

}  // namespace moe
