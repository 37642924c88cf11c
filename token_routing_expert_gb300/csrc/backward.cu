// Backward of the grouped SwiGLU experts and of the weighted combine (training).
//
// Page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"SwiGLU с квантизацией": the SwiGLU backward splits the last dimension into
// up and gate, computes the sigmoid, gate * sigmoid, its derivative and the two
// gradients in float32 and concatenates them back in the input dtype.
//
// Row kernels here are HBM-bound; the contractions run on the tcgen05 GEMM, which reads every
// operand as stored (weights and activations as MN-major operands where the contraction runs
// along their rows), so nothing is transposed:
//   UG  = Xp W_up_gate^T            (pre-activations: the forward's, kept, or recomputed; bf16)
//   dH  = dY W_out                  (W_out as an MN-major B; dY read at the dense rows; the SwiGLU
//                                    backward runs in this GEMM's epilogue: dUG and H out, dH is
//                                    never stored)
//   dXp = dUG W_up_gate             (W_up_gate as an MN-major B)
//   dW_out[e]     = dY_e^T H_e      (K-grouped over the expert's rows, MN-major A and B; dY dense)
//   dW_up_gate[e] = dUG_e^T Xp_e    (K-grouped)
// The activations live in a padded row layout (each expert from a 64-row boundary, zero rows
// between), so that every 64-row k-tile of the K-grouped GEMMs belongs to one expert.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// Padded row layout of the experts backward: expert e's rows start at row poff[e] = 64 k_off[e]
// and are followed by zero rows up to the next multiple of 64, so every 64-row k-tile of the
// weight-gradient GEMMs belongs to one expert and they read the activations as stored.
// ---------------------------------------------------------------------------

// One block of 1024 threads: k_off = prefix of ceil(count / 64), poff = 64 k_off, and the tile
// table of the M-grouped GEMMs over the padded groups (prefix of ceil(64 ceil(count / 64) / rpt)).
__global__ void __launch_bounds__(1024) pad_offsets_kernel(const int32_t* __restrict__ off, int E, int rows_per_tile,
                                                           int32_t* __restrict__ k_off, int32_t* __restrict__ poff,
                                                           int32_t* __restrict__ tile_off) {
  __shared__ int s_warp[32], s_warp2[32];
  const int e = threadIdx.x;
  const int cnt = e < E ? off[e + 1] - off[e] : 0;
  const int kt = (cnt + 63) / 64;
  const int excl = block_exclusive_scan(kt, s_warp);
  const int tiles = (64 * kt + rows_per_tile - 1) / rows_per_tile;
  const int texcl = block_exclusive_scan(tiles, s_warp2);
  if (e < E) {
    k_off[e] = excl;
    poff[e] = 64 * excl;
    tile_off[e] = texcl;
    if (e == E - 1) {
      k_off[E] = excl + kt;
      poff[E] = 64 * (excl + kt);
      tile_off[E] = texcl + tiles;
    }
  }
}

// dst row pr (a warp each, pr < 64 k_off[E]) of expert e = the group whose 64-row tiles hold it,
// r = pr - poff[e]: for r < count, source row gather[off[e] + r] (gather NULL: off[e] + r; -1: a
// zero row); a zero row past the expert's count.
__global__ void __launch_bounds__(256) pad_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ gather,
                                                       const int32_t* __restrict__ off,
                                                       const int32_t* __restrict__ k_off, int E, int src_rows,
                                                       int vec, long long max_rows, uint4* __restrict__ dst,
                                                       int* status) {
  const int lane = threadIdx.x & 31;
  const long long pr = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (pr >= max_rows || pr >= 64ll * k_off[E]) return;
  const int kt = (int)(pr / 64);
  int lo = 0, hi = E - 1;   // last e with k_off[e] <= kt (an expert with rows owns the tile)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (k_off[mid] <= kt) lo = mid; else hi = mid - 1;
  }
  const int r = (int)(pr - 64ll * k_off[lo]);
  int srow = -1;
  if (r < off[lo + 1] - off[lo]) {
    srow = gather ? gather[off[lo] + r] : off[lo] + r;
    if (srow < -1 || srow >= src_rows) {
      if (lane == 0) set_status(status, MOE_ERR_BOUNDS);
      srow = -1;
    }
  }
  uint4* d = dst + pr * vec;
  if (srow < 0) {
    for (int c = lane; c < vec; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* sr = src + (long long)srow * vec;
  for (int c0 = lane; c0 < vec; c0 += 256) {   // eight 16-byte loads in flight per lane
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) v[i] = __ldg(sr + c0 + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) d[c0 + 32 * i] = v[i];
  }
}

// A scatter index into the dense row order, moved to the padded one (-1 stays -1).
__global__ void __launch_bounds__(256) pad_scatter_kernel(const int32_t* __restrict__ scatter, int R,
                                                          const int32_t* __restrict__ off,
                                                          const int32_t* __restrict__ poff, int E,
                                                          int32_t* __restrict__ out) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= R) return;
  const int p = scatter[f];
  if (p < 0) {
    out[f] = p;
    return;
  }
  int lo = 0, hi = E - 1;   // last e with off[e] <= p: the expert that owns row p (never an empty one)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= p) lo = mid; else hi = mid - 1;
  }
  out[f] = p - off[lo] + poff[lo];
}

cudaError_t launch_pad_offsets(const int32_t* off, int E, int rows_per_tile, int32_t* k_off, int32_t* poff,
                               int32_t* tile_off, cudaStream_t st) {
  if (E > 1024) return cudaErrorInvalidValue;
  pad_offsets_kernel<<<1, 1024, 0, st>>>(off, E, rows_per_tile, k_off, poff, tile_off);
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(const void* src, const int32_t* gather, const int32_t* off, const int32_t* k_off, int E,
                            int src_rows, int cols, long long max_rows, void* dst, int* status, cudaStream_t st) {
  if (max_rows <= 0) return cudaSuccess;
  if (cols % 8) return cudaErrorInvalidValue;
  pad_rows_kernel<<<(unsigned)((max_rows + 7) / 8), 256, 0, st>>>(static_cast<const uint4*>(src), gather, off, k_off, E,
                                                                   src_rows, cols / 8, max_rows,
                                                                   static_cast<uint4*>(dst), status);
  return cudaGetLastError();
}

cudaError_t launch_pad_scatter(const int32_t* scatter, int R, const int32_t* off, const int32_t* poff, int E,
                               int32_t* out, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  pad_scatter_kernel<<<(R + 255) / 256, 256, 0, st>>>(scatter, R, off, poff, E, out);
  return cudaGetLastError();
}

// Warp per token: dy[p] = w[t, j] dz[t] (bf16) and dw[t, j] = <dz[t], y[p]> (fp32) for each
// assignment with a row p (p = -1: dropped, dw = 0).  The token's dz row is held in registers,
// 256 16-byte chunks (eight per lane) at a time, and each y row's chunks are loaded together.
__global__ void __launch_bounds__(128) combine_backward_kernel(const uint4* __restrict__ dz, const uint4* __restrict__ y,
                                                                const int32_t* __restrict__ scatter_idx,
                                                                const float* __restrict__ w, int T, int k, int vec,
                                                                int rows, uint4* __restrict__ dy,
                                                                float* __restrict__ dw, int* status) {
  __shared__ float s_dot[4][32];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const long long t = (long long)blockIdx.x * (blockDim.x >> 5) + wi;
  if (t >= T) return;
  // lane j (< k) holds assignment j's row and weight; broadcast by shuffles
  int my_p = -1;
  float my_w = 0.f;
  if (lane < k) {
    my_p = scatter_idx[t * k + lane];
    my_w = w[t * k + lane];
    if (my_p < -1 || my_p >= rows) {
      set_status(status, MOE_ERR_BOUNDS);
      my_p = -1;
    }
  }
  s_dot[wi][lane] = 0.f;
  __syncwarp();
  const uint4* dzr = dz + t * vec;
  for (int base = 0; base < vec; base += 256) {   // every lane runs every iteration (shuffles below)
    const int c0 = base + lane;
    uint4 a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec) a[i] = dzr[c0 + 32 * i];
    for (int j = 0; j < k; ++j) {
      const int p = __shfl_sync(0xffffffffu, my_p, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      if (p < 0) continue;   // warp-uniform
      const uint4* yr = y + (long long)p * vec;
      uint4* dyr = dy + (long long)p * vec;
      uint4 b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + 32 * i < vec) b[i] = yr[c0 + 32 * i];
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c0 + 32 * i < vec) {
          const uint32_t aw[4] = {a[i].x, a[i].y, a[i].z, a[i].w}, bw[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float a0 = bf16_lo(aw[q]), a1 = bf16_hi(aw[q]);
            dot = fmaf(a0, bf16_lo(bw[q]), dot);
            dot = fmaf(a1, bf16_hi(bw[q]), dot);
            o[q] = pack_bf16x2(wj * a0, wj * a1);
          }
          dyr[c0 + 32 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (lane == 0) s_dot[wi][j] += dot;
    }
  }
  __syncwarp();
  if (lane < k) dw[t * k + lane] = my_p < 0 ? 0.f : s_dot[wi][lane];
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

namespace moe {

// ---------------------------------------------------------------------------
// Router backward (for a fixed choice of experts; score_bias gets no gradient)
// ---------------------------------------------------------------------------
struct RouterBwdParams {
  const float* logits;   // (T, E) with the router bias
  const int32_t* idx;    // (T, k)
  const float* dw;       // (T, k)
  int T, E, k, gating;
  float sig_eps, p_norm, scale;
  float* dlogits;        // (T, E) fp32 out
  uint16_t* dl_bf16;     // (T, Epad) bf16 out, zero padded
  int Epad;
};

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int NI>
__global__ void __launch_bounds__(256) router_backward_kernel(const RouterBwdParams p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int E = p.E, k = p.k;
  const float* lrow = p.logits + (long long)t * E;
  const bool mine = lane < k;
  const int my_e = mine ? p.idx[(long long)t * k + lane] : 0;
  const float my_lg = mine ? lrow[my_e] : 0.f;
  // raw weight of the chosen expert (before normalisation and scaling)
  float s_all[NI];
  float w_raw = 0.f, sig = 0.f;
  if (p.gating == MOE_GATING_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int e = lane + 32 * i;
      s_all[i] = e < E ? lrow[e] : -INFINITY;
      m = fmaxf(m, s_all[i]);
    }
    m = wmax(m);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      s_all[i] = (lane + 32 * i < E) ? expf(s_all[i] - m) : 0.f;
      sum += s_all[i];
    }
    sum = wsum(sum);
#pragma unroll
    for (int i = 0; i < NI; ++i) s_all[i] /= sum;
    w_raw = mine ? expf(my_lg - m) / sum : 0.f;
  } else if (p.gating == MOE_GATING_TOPK_SOFTMAX) {
    const float m = wmax(mine ? my_lg : -INFINITY);
    const float ex = mine ? expf(my_lg - m) : 0.f;
    w_raw = ex / wsum(ex);
  } else {
    sig = 1.0f / (1.0f + expf(-my_lg));
    w_raw = mine ? sig + p.sig_eps : 0.f;
  }
  // undo the scalings, then the p-norm
  const float d_norm = mine ? p.dw[(long long)t * k + lane] * p.scale : 0.f;
  float d_raw = d_norm;
  if (p.p_norm > 0.f) {
    const float pp = p.p_norm;
    const float n = powf(wsum(mine ? powf(fabsf(w_raw), pp) : 0.f), 1.0f / pp);
    const float dot = wsum(d_norm * w_raw);
    const float dn_dw = mine ? copysignf(powf(fabsf(w_raw), pp - 1.f), w_raw) * powf(n, 1.f - pp) : 0.f;
    d_raw = d_norm / n - dot / (n * n) * dn_dw;
  }
  // gradient with respect to the selected scores / logits
  float d_sel = 0.f;
  if (p.gating == MOE_GATING_TOPK_SOFTMAX) {
    d_sel = w_raw * (d_raw - wsum(d_raw * w_raw));
  } else if (p.gating == MOE_GATING_SIGMOID) {
    d_sel = d_raw * sig * (1.f - sig);
  } else {
    d_sel = d_raw;   // gradient of the full softmax's score at the chosen expert
  }
  float dsoft_dot = 0.f;
  float row[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    float v = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_e, j);
      const float dj = __shfl_sync(0xffffffffu, d_sel, j);
      if (ej == e) v += dj;
    }
    row[i] = v;
    if (p.gating == MOE_GATING_SOFTMAX && e < E) dsoft_dot += v * s_all[i];
  }
  if (p.gating == MOE_GATING_SOFTMAX) {
    dsoft_dot = wsum(dsoft_dot);
#pragma unroll
    for (int i = 0; i < NI; ++i) row[i] = s_all[i] * (row[i] - dsoft_dot);
  }
  float* drow = p.dlogits + (long long)t * E;
  uint16_t* brow = p.dl_bf16 + (long long)t * p.Epad;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E) drow[e] = row[i];
  }
  for (int e = lane; e < p.Epad; e += 32) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i == e) v = row[i];
    __nv_bfloat16 b = __float2bfloat16_rn(e < E ? v : 0.f);
    brow[e] = *reinterpret_cast<uint16_t*>(&b);
  }
}

cudaError_t launch_router_backward(const float* logits, const int32_t* idx, const float* dw, int T, int E, int k,
                                   int gating, float sig_eps, float p_norm, float scale, float* dlogits,
                                   void* dl_bf16, int Epad, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  RouterBwdParams p{logits, idx, dw, T, E, k, gating, sig_eps, p_norm, scale, dlogits,
                    static_cast<uint16_t*>(dl_bf16), Epad};
  const dim3 grid((T + 7) / 8), block(256);
  const int ni = (E + 31) / 32;
  if (ni <= 1) router_backward_kernel<1><<<grid, block, 0, st>>>(p);
  else if (ni <= 2) router_backward_kernel<2><<<grid, block, 0, st>>>(p);
  else if (ni <= 4) router_backward_kernel<4><<<grid, block, 0, st>>>(p);
  else if (ni <= 8) router_backward_kernel<8><<<grid, block, 0, st>>>(p);
  else if (ni <= 16) router_backward_kernel<16><<<grid, block, 0, st>>>(p);
  else if (ni <= 28) router_backward_kernel<28><<<grid, block, 0, st>>>(p);
  else if (ni <= 32) router_backward_kernel<32><<<grid, block, 0, st>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}


// db[e] = sum over t of d[t, e]: 32 columns per block, 8 row groups reduced in shared memory.
__global__ void __launch_bounds__(256) column_sum_kernel(const float* __restrict__ d, int T, int E,
                                                          float* __restrict__ out) {
  __shared__ float part[8][33];
  const int e = blockIdx.x * 32 + threadIdx.x;
  float s = 0.f;
  if (e < E)
    for (int t = threadIdx.y; t < T; t += 8) s += d[(long long)t * E + e];
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && e < E) {
    float tot = 0.f;
    for (int i = 0; i < 8; ++i) tot += part[i][threadIdx.x];
    out[e] = tot;
  }
}

cudaError_t launch_column_sum(const float* d, int T, int E, float* out, cudaStream_t st) {
  column_sum_kernel<<<(E + 31) / 32, dim3(32, 8), 0, st>>>(d, T, E, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward of the latent up-projection's input norm (page "Как устроен Olmo-core 3",
// §"Латентная проекция экспертов": bias-free RMSNorm of the experts' combined output, then the
// up-projection).  n = z r gamma, r = 1 / sqrt(mean(z^2) + eps):
//   dz = r gamma dn - z r^3 mean(z gamma dn)        (fp32, stored bf16)
//   dgamma = sum over tokens of dn z r               (fp32, fixed summation order)
// ---------------------------------------------------------------------------

// Warp per row: both row sums in one pass, dz in a second (the row is re-read from L1 / L2);
// r_out[t] = r for the gain's gradient.
__global__ void __launch_bounds__(256) rmsnorm_backward_kernel(const uint4* __restrict__ z,
                                                                const uint4* __restrict__ dn,
                                                                const uint4* __restrict__ gamma, int T, int vec,
                                                                float eps, uint4* __restrict__ dz,
                                                                float* __restrict__ r_out) {
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const uint4* zr = z + t * vec;
  const uint4* dr = dn + t * vec;
  const uint32_t one2 = 0x3F803F80u;   // two bf16 ones: the gain without a weight
  float ss = 0.f, dot = 0.f;
  for (int c = lane; c < vec; c += 32) {
    const uint4 a = zr[c], b = dr[c];
    const uint4 gv = gamma ? gamma[c] : make_uint4(one2, one2, one2, one2);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float z0 = bf16_lo(aw[q]), z1 = bf16_hi(aw[q]);
      const float g0 = bf16_lo(gw[q]), g1 = bf16_hi(gw[q]);
      ss = fmaf(z0, z0, fmaf(z1, z1, ss));
      dot = fmaf(z0 * g0, bf16_lo(bw[q]), fmaf(z1 * g1, bf16_hi(bw[q]), dot));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
  }
  const float n = (float)(8 * vec);
  const float r = rsqrtf(ss / n + eps);
  const float k3 = r * r * r * (dot / n);
  for (int c = lane; c < vec; c += 32) {
    const uint4 a = zr[c], b = dr[c];
    const uint4 gv = gamma ? gamma[c] : make_uint4(one2, one2, one2, one2);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float g0 = bf16_lo(gw[q]), g1 = bf16_hi(gw[q]);
      o[q] = pack_bf16x2(r * g0 * bf16_lo(bw[q]) - bf16_lo(aw[q]) * k3, r * g1 * bf16_hi(bw[q]) - bf16_hi(aw[q]) * k3);
    }
    dz[t * vec + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) r_out[t] = r;
}

// part[s][l] = sum over the rows of slab s of dn[t][l] z[t][l] r[t] (a thread per column).
__global__ void __launch_bounds__(256) rms_gain_grad_kernel(const __nv_bfloat16* __restrict__ z,
                                                             const __nv_bfloat16* __restrict__ dn,
                                                             const float* __restrict__ r, int T, int L, int slab,
                                                             float* __restrict__ part) {
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= L) return;
  const int t0 = blockIdx.y * slab, t1 = min(T, t0 + slab);
  float acc = 0.f;
  for (int t = t0; t < t1; ++t)
    acc = fmaf(__bfloat162float(dn[(long long)t * L + l]) * __bfloat162float(z[(long long)t * L + l]), r[t], acc);
  part[(long long)blockIdx.y * L + l] = acc;
}

cudaError_t launch_rmsnorm_backward(const void* z, const void* dn, const void* gamma, int T, int L, float eps,
                                    void* dz, float* r, float* gain_part, int slab, float* dgamma, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (L % 8) return cudaErrorInvalidValue;
  rmsnorm_backward_kernel<<<(T + 7) / 8, 256, 0, st>>>(static_cast<const uint4*>(z), static_cast<const uint4*>(dn),
                                                       static_cast<const uint4*>(gamma), T, L / 8, eps,
                                                       static_cast<uint4*>(dz), r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !dgamma) return e;
  const int nslab = (T + slab - 1) / slab;
  rms_gain_grad_kernel<<<dim3((L + 255) / 256, nslab), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(z), static_cast<const __nv_bfloat16*>(dn), r, T, L, slab, gain_part);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_column_sum(gain_part, nslab, L, dgamma, st);
}

// out = a + b for bf16 tensors (fp32 add, rounded to bf16), n8 16-byte vectors.
__global__ void __launch_bounds__(256) add_bf16_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b,
                                                        long long n8, uint4* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const uint4 x = a[i], y = b[i];
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(bf16_lo(xw[q]) + bf16_lo(yw[q]), bf16_hi(xw[q]) + bf16_hi(yw[q]));
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_add_bf16(const void* a, const void* b, long long n, void* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  const long long n8 = n / 8;
  const int blocks = (int)std::min<long long>((n8 + 255) / 256, (long long)num_sms() * 8);
  add_bf16_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(a), static_cast<const uint4*>(b), n8,
                                          static_cast<uint4*>(out));
  return cudaGetLastError();
}

// out = sum over s of part[s] (fp32), slices of n4 float4.
cudaError_t launch_sum_slices_f32(const float* part, int splits, long long n, float* out, cudaStream_t st);

}  // namespace moe
