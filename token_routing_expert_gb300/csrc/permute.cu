// Token permutation: histogram, scan and stable placement of the assignments.
//
// Assignment f = t*k + j of expert idx[f] goes to row
//   offsets[e] + #{f' < f : idx[f'] == e}
// (page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"Пересылка токенов между экспертами": indices sorted by expert, bins =
// cumulative sum of the per-expert counts).  Up to 16,384 assignments it is one launch on one
// 8-CTA cluster (histograms exchanged through distributed shared memory); beyond, three passes
// over chunks of assignments (256 to 4096 per block): per-chunk histograms; per-expert scan over
// chunks plus the exclusive scan over experts; placement, where each warp walks its slice of the
// chunk in order and ranks equal experts with __match_any_sync (the cluster kernel places the
// same way).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kMaxChunk = 4096;
constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;

int permute_blocks(int R, int chunk) { return (R + chunk - 1) / chunk; }

// Assignments per block: about 76 blocks (the scan walks one histogram per block,
// so more blocks cost more than they gain), 256 to 4096, a multiple of 256 (each
// of the 8 warps walks chunk / 8 assignments).
int permute_chunk(int R) {
  int c = (R / 76 + 255) / 256 * 256;
  return c < 256 ? 256 : (c > kMaxChunk ? kMaxChunk : c);
}

__global__ void __launch_bounds__(kPermThreads) perm_count_kernel(const int32_t* __restrict__ idx, int R, int E,
                                                                   int chunk, int32_t* __restrict__ blk,
                                                                   int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  extern __shared__ int32_t hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * chunk;
  const int end = min(R, base + chunk);
  for (int r = base + threadIdx.x; r < end; r += blockDim.x) {
    const int e = idx[r];
    if (e < 0 || e >= E) set_status(status, MOE_ERR_BOUNDS);
    else atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) blk[(long long)blockIdx.x * E + i] = hist[i];
}


// One block of 1024 threads.  G = 1024 / E (rounded down to a power of two, at most 32)
// threads share expert e: thread g of the group takes a contiguous run of the per-chunk
// histograms, and a shuffle scan across the group's lanes turns them into each chunk's
// exclusive prefix within the expert.  Then an exclusive scan over the experts' totals gives
// the offsets; the placement adds offsets[e] to the chunk prefixes itself.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ blk, int nblk, int E,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets, int rows_per_tile,
                                                          int32_t* __restrict__ tile_off) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  __shared__ int s_warp[32];
  __shared__ int s_tot[1024];
  int G = 1;
  while (G < 32 && E * G * 2 <= 1024) G <<= 1;
  const int t = threadIdx.x;
  const int e = t / G, g = t % G;
  const int per = (nblk + G - 1) / G;
  const int b0 = min(nblk, g * per), b1 = min(nblk, b0 + per);
  // pass 1: the total of this thread's chunks (loads issued eight at a time, no stores between)
  int run = 0;
  if (e < E) {
    for (int b = b0; b < b1; b += 8) {
      int c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = b + i < b1 ? blk[(long long)(b + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) run += c[i];
    }
  }
  // the group's G lanes are consecutive (G divides 32): inclusive scan of the run totals
  int incl = run;
  for (int o = 1; o < G; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o, G);
    if (g >= o) incl += y;
  }
  // pass 2: each chunk's exclusive prefix within the expert (the group's earlier chunks first)
  if (e < E) {
    int acc = incl - run;
    for (int b = b0; b < b1; b += 8) {
      int c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = b + i < b1 ? blk[(long long)(b + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (b + i < b1) blk[(long long)(b + i) * E + e] = acc;
        acc += c[i];
      }
    }
  }
  if (e < E && g == G - 1) s_tot[e] = incl;
  __syncthreads();
  const int tot = t < E ? s_tot[t] : 0;
  const int excl = block_exclusive_scan(tot, s_warp);
  if (t < E) {
    counts[t] = tot;
    offsets[t] = excl;
    if (t == E - 1) offsets[E] = excl + tot;
  }
  if (tile_off) {   // the grouped GEMMs' tile table as well (what tile_table_kernel computes)
    __syncthreads();   // s_warp is reused
    const int tiles = t < E ? (tot + rows_per_tile - 1) / rows_per_tile : 0;
    const int texcl = block_exclusive_scan(tiles, s_warp);
    if (t < E) {
      tile_off[t] = texcl;
      if (t == E - 1) tile_off[E] = texcl + tiles;
    }
  }
}

__global__ void __launch_bounds__(kPermThreads) perm_place_kernel(const int32_t* __restrict__ idx, int R, int E,
                                                                   int k, int chunk, const int32_t* __restrict__ blk,
                                                                   const int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ gather_idx,
                                                                   int32_t* __restrict__ scatter_idx) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  extern __shared__ int32_t wh[];  // [kPermWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * chunk;
  const int end = min(R, base + chunk);
  const int sub = chunk / kPermWarps;
  const int s0 = base + warp * sub;
  const int s1 = min(end, s0 + sub);
  int32_t* mine = wh + warp * E;

  // pass 1: this warp's per-expert counts
  for (int r0 = s0; r0 < s1; r0 += 32) {
    const int r = r0 + lane;
    const int e = r < s1 ? idx[r] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
  }
  __syncthreads();
  // bases: expert e's offset, plus its rows in earlier chunks, plus the counts of earlier warps
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = offsets[e] + blk[(long long)blockIdx.x * E + e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = wh[w * E + e];
      wh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: stable placement
  const unsigned lt = (1u << lane) - 1u;
  for (int r0 = s0; r0 < s1; r0 += 32) {
    const int r = r0 + lane;
    const int e = r < s1 ? idx[r] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    int pos = 0;
    if (valid) pos = mine[e] + __popc(grp & lt);
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
    __syncwarp();
    if (valid) {
      gather_idx[pos] = r / k;
      scatter_idx[r] = pos;
    }
  }
}

// ---------------------------------------------------------------------------
// The same permutation in one launch, for up to kClusterCtas x kClusterChunk assignments: one
// cluster of kClusterCtas CTAs, each owning a contiguous chunk.  The CTAs count their chunks into
// shared memory, meet at a cluster barrier, read each other's histograms through distributed
// shared memory (every CTA computes the expert offsets and its own chunk's prefix; CTA 0 writes
// counts, offsets and the tile table), meet again so that no CTA leaves while another still
// reads its histogram, and place their assignments as perm_place_kernel does.
// ---------------------------------------------------------------------------
constexpr int kClusterCtas = 8;
constexpr int kClusterThreads = 1024;
constexpr int kClusterWarps = kClusterThreads / 32;
// Each of a CTA's 32 warps walks its slice serially, so the single cluster only pays off while the
// slices are short: decode-sized batches (R = 512: 10.8 vs 13.7 us per layer's permutation);
// at R = 65,536 the three-kernel path, 76 blocks wide, was 10 us faster.
constexpr int kClusterChunk = 2048;

__device__ __forceinline__ int ld_shared_cluster_i32(uint32_t cluster_addr) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(kClusterThreads) perm_cluster_kernel(const int32_t* __restrict__ idx, int R, int E,
                                                                        int k, int chunk, int32_t* __restrict__ counts,
                                                                        int32_t* __restrict__ offsets,
                                                                        int rows_per_tile,
                                                                        int32_t* __restrict__ tile_off,
                                                                        int32_t* __restrict__ gather_idx,
                                                                        int32_t* __restrict__ scatter_idx,
                                                                        int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  extern __shared__ int32_t sm[];
  int32_t* wh = sm;                          // [kClusterWarps][E]: per-warp counts, then bases
  int32_t* hist = wh + kClusterWarps * E;    // [E]: this chunk's histogram (read by the other CTAs)
  __shared__ int s_warp[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  for (int i = threadIdx.x; i < kClusterWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int base = (int)rank * chunk;
  const int end = min(R, base + chunk);
  const int sub = (chunk + kClusterWarps - 1) / kClusterWarps;
  const int s0 = min(end, base + warp * sub);
  const int s1 = min(end, s0 + sub);
  int32_t* mine = wh + warp * E;

  // this warp's per-expert counts
  for (int r0 = s0; r0 < s1; r0 += 32) {
    const int r = r0 + lane;
    const int e = r < s1 ? idx[r] : -1;
    const bool valid = e >= 0 && e < E;
    if (r < s1 && !valid) set_status(status, MOE_ERR_BOUNDS);
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < kClusterWarps; ++w) c += wh[w * E + e];
    hist[e] = c;
  }
  cluster_sync_all();   // every CTA's histogram is complete

  // expert totals and this chunk's prefix within each expert, from all CTAs' histograms
  // (E <= 1024: a thread per expert)
  const uint32_t hist_addr = smem_u32(hist);
  const int e = threadIdx.x;
  int tot = 0, pre = 0;
  if (e < E) {
    for (int c = 0; c < kClusterCtas; ++c) {
      const int h = ld_shared_cluster_i32(map_to_cta(hist_addr + 4u * (uint32_t)e, (uint32_t)c));
      if (c < (int)rank) pre += h;
      tot += h;
    }
  }
  const int excl = block_exclusive_scan(tot, s_warp);
  if (e < E) {
    // per-warp bases: expert e's offset, its rows in earlier chunks, then the earlier warps' counts
    int run = excl + pre;
    for (int w = 0; w < kClusterWarps; ++w) {
      const int c = wh[w * E + e];
      wh[w * E + e] = run;
      run += c;
    }
    if (rank == 0) {
      counts[e] = tot;
      offsets[e] = excl;
      if (e == E - 1) offsets[E] = excl + tot;
    }
  }
  if (tile_off) {
    __syncthreads();   // s_warp is reused
    const int tiles = e < E ? (tot + rows_per_tile - 1) / rows_per_tile : 0;
    const int texcl = block_exclusive_scan(tiles, s_warp);
    if (rank == 0 && e < E) {
      tile_off[e] = texcl;
      if (e == E - 1) tile_off[E] = texcl + tiles;
    }
  }
  __syncthreads();   // the bases in wh are complete
  cluster_sync_all();   // no CTA leaves while another still reads its histogram

  // stable placement
  const unsigned lt = (1u << lane) - 1u;
  for (int r0 = s0; r0 < s1; r0 += 32) {
    const int r = r0 + lane;
    const int e = r < s1 ? idx[r] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    int pos = 0;
    if (valid) pos = mine[e] + __popc(grp & lt);
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
    __syncwarp();
    if (valid) {
      gather_idx[pos] = r / k;
      scatter_idx[r] = pos;
    }
  }
}

bool permute_fits_cluster(int R, int E) { return R > 0 && R <= kClusterCtas * kClusterChunk && E <= 1024; }

cudaError_t launch_permute_cluster(const int32_t* idx, int R, int E, int32_t* counts, int32_t* offsets,
                                   int32_t* gather_idx, int32_t* scatter_idx, int k, int* status,
                                   cudaStream_t stream, int rows_per_tile, int32_t* tile_off) {
  if (!permute_fits_cluster(R, E)) return cudaErrorInvalidValue;
  const int chunk = (R + kClusterCtas - 1) / kClusterCtas;
  const size_t smem = (size_t)(kClusterWarps + 1) * E * sizeof(int32_t);
  static std::atomic<int> ready[kMaxDeviceSlots];
  const int dev = device_slot();
  if (dev < 0 || !ready[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(perm_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((kClusterWarps + 1) * 1024 * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    if (dev >= 0) ready[dev].store(1);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterCtas);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kClusterCtas;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, perm_cluster_kernel, idx, R, E, k, chunk, counts, offsets, rows_per_tile, tile_off,
                            gather_idx, scatter_idx, status);
}

cudaError_t launch_permute(const int32_t* idx, int R, int E, int32_t* counts, int32_t* offsets,
                           int32_t* gather_idx, int32_t* scatter_idx, int k, int chunk, int32_t* blk, int* status,
                           cudaStream_t stream, int rows_per_tile, int32_t* tile_off) {
  if (chunk < 256 || chunk > kMaxChunk || chunk % 256) return cudaErrorInvalidValue;
  if (permute_fits_cluster(R, E))   // one launch: the whole permutation on one cluster
    return launch_permute_cluster(idx, R, E, counts, offsets, gather_idx, scatter_idx, k, status, stream,
                                  rows_per_tile, tile_off);
  const int nb = permute_blocks(R, chunk);
  if (nb > 0) {
    launch_pdl(perm_count_kernel, nb, kPermThreads, E * sizeof(int32_t), stream, idx, R, E, chunk, blk, status);
  }
  launch_pdl(perm_scan_kernel, 1, 1024, 0, stream, blk, nb, E, counts, offsets, rows_per_tile, tile_off);
  if (nb > 0) {
    const size_t sm = (size_t)kPermWarps * E * sizeof(int32_t);
    launch_pdl(perm_place_kernel, nb, kPermThreads, sm, stream, idx, R, E, k, chunk, blk, offsets, gather_idx, scatter_idx);
  }
  return cudaGetLastError();
}

// tile_off[e] = sum over e' < e of ceil(count[e'] / rows_per_tile); tile_off[E] = total tiles.
__global__ void __launch_bounds__(1024) tile_table_kernel(const int32_t* __restrict__ offsets, int E, int rows_per_tile,
                                                           int32_t* __restrict__ tile_off) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  const int tiles = e < E ? (offsets[e + 1] - offsets[e] + rows_per_tile - 1) / rows_per_tile : 0;
  const int excl = block_exclusive_scan(tiles, s_warp);
  if (e < E) {
    tile_off[e] = excl;
    if (e == E - 1) tile_off[E] = excl + tiles;
  }
}

cudaError_t launch_tile_table(const int32_t* offsets, int E, int rows_per_tile, int32_t* tile_off,
                              cudaStream_t stream) {
  launch_pdl(tile_table_kernel, 1, 1024, 0, stream, offsets, E, rows_per_tile, tile_off);
  return cudaGetLastError();
}

// dst[p, :] = src[gather_idx[p], :] for p < R; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                           const int32_t* __restrict__ gather_idx, int R, int T,
                                                           int vec_per_row, uint4* __restrict__ dst,
                                                           int allow_padding, int* status) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= R) return;
  const int t = gather_idx[p];
  if (t < 0 || t >= T) {
    if (allow_padding && t == -1) {  // a padding slot of a capacity-limited expert: a zero row
      uint4* d = dst + p * vec_per_row;
      for (int c = lane; c < vec_per_row; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
    } else if (lane == 0) {
      set_status(status, MOE_ERR_BOUNDS);
    }
    return;
  }
  const uint4* s = src + (long long)t * vec_per_row;
  uint4* d = dst + p * vec_per_row;
  // eight 16-byte loads in flight per lane before the stores
  for (int c0 = lane; c0 < vec_per_row; c0 += 256) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + 32 * i < vec_per_row) v[i] = __ldg(s + c0 + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i)   // streaming stores: keep the source rows, not the copy, in L2
      if (c0 + 32 * i < vec_per_row) __stcs(d + c0 + 32 * i, v[i]);
  }
}

cudaError_t launch_gather_rows(const void* src, const int32_t* gather_idx, int R, int T, int cols, void* dst,
                               int allow_padding, int* status, cudaStream_t stream) {
  if (R <= 0) return cudaSuccess;
  const int warps = 8;
  launch_pdl(gather_rows_kernel, (R + warps - 1) / warps, 32 * warps, 0, stream, 
      static_cast<const uint4*>(src), gather_idx, R, T, cols / 8, static_cast<uint4*>(dst), allow_padding, status);
  return cudaGetLastError();
}

// Capacity slots (page "Как устроен Olmo-core 3: обучение больших MoE-моделей",
// §"Ёмкость эксперта и переполнение"): expert e owns slots [e*cap, (e+1)*cap);
// its r-th assignment in the stable order goes to slot e*cap + r if r < cap,
// otherwise it is dropped (-1); unused slots are padding (-1).
__global__ void __launch_bounds__(256) capacity_remap_kernel(const int32_t* __restrict__ idx, int R, int E, int cap,
                                                              const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ off_dense,
                                                              const int32_t* __restrict__ gather_dense,
                                                              const int32_t* __restrict__ scatter_dense,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ gather_idx,
                                                              int32_t* __restrict__ scatter_idx) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  const long long slots = (long long)E * cap;
  const long long n = max(max(slots, (long long)R), (long long)E + 1);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    if (i <= E) offsets[i] = (int32_t)(i * cap);
    if (i < slots) {
      const int e = (int)(i / cap);
      const int r = (int)(i - (long long)e * cap);
      gather_idx[i] = r < counts[e] ? gather_dense[off_dense[e] + r] : -1;
    }
    if (i < R) {
      const int e = idx[i];
      int slot = -1;
      if (e >= 0 && e < E) {
        const int r = scatter_dense[i] - off_dense[e];
        if (r < cap) slot = e * cap + r;
      }
      scatter_idx[i] = slot;
    }
  }
}

cudaError_t launch_capacity_remap(const int32_t* idx, int R, int E, int cap, const int32_t* counts,
                                  const int32_t* off_dense, const int32_t* gather_dense,
                                  const int32_t* scatter_dense, int32_t* offsets, int32_t* gather_idx,
                                  int32_t* scatter_idx, cudaStream_t stream) {
  const long long n = std::max(std::max((long long)E * cap, (long long)R), (long long)E + 1);
  const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
  launch_pdl(capacity_remap_kernel, blocks, 256, 0, stream, idx, R, E, cap, counts, off_dense, gather_dense, scatter_dense,
                                                    offsets, gather_idx, scatter_idx);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// moe_permute_noalloc: the same permutation with its scratch in static device memory
// ---------------------------------------------------------------------------

// Per-chunk expert histograms of moe_permute_noalloc.  Every GPU that loads the
// library reserves this array until the process exits.
constexpr int64_t kNoAllocScratchInts = int64_t(1) << 19;  // 2 MiB
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

namespace {
constexpr int kMaxScratchDevices = 64;
std::atomic<int32_t*> g_permute_scratch_addr[kMaxScratchDevices];
}  // namespace

// Device address of g_permute_scratch on the current device, looked up once per
// device (the host-side symbol is only a stand-in, never a device address).  Two
// host threads that make a device's first call at once both look it up and store
// the same address.
static int scratch_address(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_NO_DEVICE;
  int32_t* p = g_permute_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    p = static_cast<int32_t*>(ptr);
    g_permute_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_permute_noalloc(const moe_config_t* cfg, const int32_t* idx, int64_t T, int32_t* counts,
                                   int32_t* offsets, int32_t* gather_idx, int32_t* scatter_idx,
                                   moe_stream_t stream) {
  int s = moe_validate_config(cfg);
  if (s != MOE_OK) return s;
  if (cfg->capacity_factor > 0.f) return MOE_ERR_UNSUPPORTED;  // capacity slots need the workspace path
  if (T < 0 || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!idx || !gather_idx || !scatter_idx)) return MOE_ERR_INVALID_ARG;
  if (T * cfg->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  const int R = (int)(T * cfg->top_k);
  const int64_t E = cfg->num_experts;
  // the histograms need one int per (chunk, expert): with the largest chunks, beyond the
  // static array, refuse; otherwise take moe_permute's own chunk size when its histograms fit
  // (more, smaller chunks spread the passes over more SMs; the result does not depend on it)
  const int64_t need = (int64_t)std::max(1, moe::permute_blocks(R, moe::kMaxChunk)) * E;
  if (need > moe::kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
  int chunk = moe::permute_chunk(R);
  if ((int64_t)std::max(1, moe::permute_blocks(R, chunk)) * E > moe::kNoAllocScratchInts) chunk = moe::kMaxChunk;
  int32_t* scratch = nullptr;
  s = moe::scratch_address(&scratch);
  if (s != MOE_OK) return s;
  int* status = moe::device_status();
  if (!status) return MOE_ERR_NO_DEVICE;
  // every histogram entry the scan reads is written by this call first: nothing to clear
  return moe::launch_permute(idx, R, cfg->num_experts, counts, offsets, gather_idx, scatter_idx, cfg->top_k,
                             chunk, scratch, status, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
