// Persistent, warp-specialised tcgen05 GEMM for sm_103a, dense or grouped.
//
// One CTA per SM walks a static round-robin list of 128 x BN output tiles.
//   warp 0 (one lane)  : TMA producer, STAGES-deep ring of (A, B) k-tiles
//   warp 1 (one lane)  : UMMA issuer (M=128, N=BN, K=16 per instruction),
//                        accumulates into one of two TMEM accumulators
//   warps 2..9         : epilogue, TMEM -> registers -> global, two warps per
//                        TMEM lane quadrant (alternate 32-column chunks), overlapping
//                        the next tile's mainloop through the second accumulator
// Grouped mode: the row ranges of the groups and their tile prefix sums are
// read on the device, so no host synchronisation is needed to schedule them.
// Epilogues: fp32 (router logits, split-K partials), bf16, and SwiGLU, where
// the B tile holds BN/2 "up" rows and BN/2 "gate" rows of the same expert and
// the epilogue writes silu(gate) * up as bf16.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int BM = 128;
constexpr int BK = 64;                 // 64 bf16 = 128 bytes: one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kMaxGroups = 1024;
constexpr int kEpiWarps = 8;                   // two warps per TMEM lane quadrant, each half the columns
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kEpiStageBytes = kEpiWarps * 2048;   // a 32 x 32 bf16 block per epilogue warp
// Gathered-A kernels add 4 warps that copy the A rows from their source rows (cp.async) and
// one warp whose lane 0 hands each landed stage on to the MMA (see gather_a_relay).
constexpr int kGatherWarps = 4;
constexpr int kGatherThread0 = 32 * (2 + kEpiWarps);
constexpr int kRelayWarp = 2 + kEpiWarps + kGatherWarps;
constexpr int kThreadsGA = 32 * (kRelayWarp + 1);

struct GemmParams {
  int M, N, K;
  int num_groups;          // 0 = dense
  const int* group_off;
  const int* tile_off;
  int b_rows_per_group;
  int b_gate_offset;
  int n_tiles;
  int splits;
  int kt_per_split;
  int kt_total;
  void* out;
  long long ldo;
  long long split_stride;
  int k_groups;            // > 0: K-grouped (group g contracts k-tiles [k_off[g], k_off[g+1]))
  const int* k_off;        // device (k_groups+1) k-tile offsets
  const float* a_scale;    // e4m3 operands: scale of each A row
  const float* b_scale;    // e4m3 operands: scale of each B row
  const int* a_gather;     // non-null: A row r is row a_gather[r] of a_src (-1: a zero row)
  const uint8_t* a_src;    //   source rows (a_src_rows x K), a_ld_bytes apart
  long long a_ld_bytes;
  int a_src_rows;
  int b_mn;                // 1: B is MN-major, group g's K rows [g * b_rows_per_group, ...) x N columns
  int a_mn;                // 1 (K-grouped, 1 CTA): A is MN-major, K rows x M columns
  const int* a_off;        // non-null: group g's A rows start at A row a_off[g] (see a_row_shift)
  void* preact;            // SwiGLU: also store [u | g] (bf16) here, preact_ld elements per row;
                           // SwiGLU backward: read [u | g] from here
  long long preact_ld;
  int preact_dense;        // SwiGLU backward: [u | g] rows at A's rows (shifted by a_off), else the output's
  void* out2;              // SwiGLU backward: H
  long long ldo2;
  const int* b_gather;     // K-grouped, gathered B: group g's K row r is row b_gather[b_goff[g] + r] of b_src
  const uint8_t* b_src;    //   (r < the group's count; zeros past it), b_ld_bytes apart
  const int* b_goff;
  long long b_ld_bytes;
  int b_src_rows;
  const uint8_t* mx_a_scale;   // MXFP8 operands: E8M0 block scales of A's rows (mx_a_ld bytes apart)
  long long mx_a_ld;
  long long mx_a_rows;
  const uint8_t* mx_b_scale;   //   and of B's rows
  long long mx_b_ld;
  long long mx_b_rows;
  uint8_t* mx_out_codes;       // MXFP8 SwiGLU: H leaves as MXFP8 codes (ldo bytes per row) and block
  uint8_t* mx_out_scale;       //   scales (mx_out_ld bytes per row) instead of bf16
  long long mx_out_ld;
  int a_keep;                  // gathered A: its source rows are read with an evict_last L2 policy
  RouterEpilogue router;       // EPI_ROUTER
  int* status;
};

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (196 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int ACC_STRIDE = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE < 32 ? 32 : 2 * ACC_STRIDE;
  // ring | barriers (full, empty, tmem_full x2, tmem_empty x2, gathered) | tmem holder | abort | group tables
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 3 * STAGES + 4;
  static constexpr int HOLDER_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int ABORT_OFF = HOLDER_OFF + 4;
  static constexpr int TABLE_OFF = (ABORT_OFF + 4 + 15) & ~15;
  static constexpr int EPI_OFF = (TABLE_OFF + 3 * (kMaxGroups + 1) * 4 + 127) & ~127;  // epilogue staging
  static constexpr int SMEM_BYTES = EPI_OFF + kEpiStageBytes + 1024;                  // + alignment slack
  static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte alignment");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=128, whole 32-column epilogue chunks");
};

struct TileCoord {
  int row0;     // first row of A / C
  int rows;     // valid rows (<= BM)
  int group;
  int nt;       // n tile
  int split;
  int kt0, kt1; // k-tile range
};

template <int ROWS = BM>
__device__ __forceinline__ TileCoord decode_tile(int t, const GemmParams& p, const int* s_toff,
                                                 const int* s_goff) {
  TileCoord c;
  if (p.k_groups > 0) {
    // K-grouped: tile t = ((g * mtiles) + mt) * n_tiles + nt; the group's output is the g-th "split" slice
    const int mtiles = (p.M + ROWS - 1) / ROWS;
    c.nt = t % p.n_tiles;
    const int rest = t / p.n_tiles;
    const int mt = rest % mtiles;
    c.group = rest / mtiles;
    c.split = c.group;
    c.row0 = mt * ROWS;
    c.rows = min(ROWS, p.M - c.row0);
    c.kt0 = s_goff[c.group];
    c.kt1 = s_goff[c.group + 1];
    return c;
  }
  c.split = t % p.splits;
  const int rest = t / p.splits;
  c.nt = rest % p.n_tiles;
  const int mt = rest / p.n_tiles;
  int row_base = 0, row_end = p.M, mt_local = mt;
  c.group = 0;
  if (p.num_groups > 0) {
    // last group g with tile_off[g] <= mt (it is non-empty because mt < tile_off[G])
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_toff[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    c.group = lo;
    mt_local = mt - s_toff[lo];
    row_base = s_goff[lo];
    row_end = s_goff[lo + 1];
  }
  c.row0 = row_base + mt_local * ROWS;
  c.rows = min(ROWS, row_end - c.row0);
  c.kt0 = c.split * p.kt_per_split;
  c.kt1 = min(p.kt_total, c.kt0 + p.kt_per_split);
  return c;
}

// With a_off, the A rows of group g are read from a_off[g] on instead of the output's own rows:
// M-grouped, output row r of group g multiplies A row r - group_off[g] + a_off[g]; K-grouped
// (MN-major A), the group's K rows start at A row a_off[g] instead of 64 k_off[g].  The rows a
// tile reads past the group's end are A's next rows (zeros past A's last row); the caller makes
// the other operand zero there.
__device__ __forceinline__ int a_row_shift(const GemmParams& p, const TileCoord& c, const int* s_goff,
                                           const int* s_aoff) {
  if (!p.a_off) return 0;
  return s_aoff[c.group] - (p.k_groups > 0 ? BK * s_goff[c.group] : s_goff[c.group]);
}

// Stores a warp's block of 32 rows x 64 bytes (thread i holds row i as 16 words: 32 bf16 or 16
// fp32) through a 2 KB shared buffer, so that each global store instruction writes 8 rows x 64
// contiguous bytes instead of 32 rows x 16 bytes.  The 16-byte slots are XOR-swizzled by row:
// both the row-wise writes and the column-wise reads hit 8 distinct bank groups per quarter warp.
// out0: the block's first byte in its first row; ld_bytes: the row pitch in bytes; valid: how
// many of the 32 rows exist.
__device__ __forceinline__ void store_block_64b(uint4* stg, const uint32_t (&packed)[16], char* out0,
                                                long long ld_bytes, int valid, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    stg[lane * 4 + (i ^ ((lane >> 1) & 3))] =
        make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
  __syncwarp();
  const int q = lane & 3;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int r = s * 8 + (lane >> 2);
    const uint4 v = stg[r * 4 + (q ^ ((r >> 1) & 3))];
    if (r < valid) *reinterpret_cast<uint4*>(out0 + r * ld_bytes + q * 16) = v;
  }
  __syncwarp();
}

__device__ __forceinline__ void store_block_bf16(uint4* stg, const uint32_t (&packed)[16], __nv_bfloat16* out0,
                                                 long long ldo, int valid, int lane) {
  store_block_64b(stg, packed, reinterpret_cast<char*>(out0), ldo * 2, valid, lane);
}

// SwiGLU backward epilogue: the [u | g] pre-activations of a warp's 32 rows, 32 columns (64 bytes
// of u and 64 of g per row) at a time.  swb_issue starts the loads, 8 rows x 64 contiguous bytes
// per instruction, into pv[0..3] (u) and pv[4..7] (g), zeros for rows whose bit in `live` is
// clear; swb_take later hands thread i row i as 16 words, through the warp's swizzled 2 KB buffer
// (the converse of store_block_64b).  A chunk's loads are issued while the previous chunk is
// computed, the first one before the accumulator is ready.
struct SwbRows {
  const char* pre;   // [u | g] of the warp's first row
  uint32_t live;     // bit r: row r of the warp's 32 is a real row (else padding: zeros)
  int valid;         // rows of the 32 inside the tile
  long long wrow0;   // output row of the warp's first row
};

__device__ __forceinline__ SwbRows swb_rows(const GemmParams& p, int row0, int rows, int row_in_tile, int ash,
                                            int live_end) {
  const int lane = row_in_tile & 31;
  SwbRows r;
  r.valid = min(max(rows - (row_in_tile - lane), 0), 32);
  r.wrow0 = (long long)row0 + (row_in_tile - lane);
  r.live = __ballot_sync(0xffffffffu, lane < r.valid && r.wrow0 + lane + ash < (long long)live_end);
  r.pre = reinterpret_cast<const char*>(p.preact) + (p.preact_dense ? r.wrow0 + ash : r.wrow0) * p.preact_ld * 2;
  return r;
}

__device__ __forceinline__ void swb_issue(uint4 (&pv)[8], const SwbRows& r, const GemmParams& p, int col0, int lane) {
  const int q = lane & 3;
  const long long ld = p.preact_ld * 2;
  const char* a0 = r.pre + (long long)col0 * 2;
  const char* b0 = r.pre + (long long)(p.N + col0) * 2;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int row = s * 8 + (lane >> 2);
    const bool live = (r.live >> row) & 1u;
    pv[s] = live ? __ldcs(reinterpret_cast<const uint4*>(a0 + row * ld + q * 16)) : make_uint4(0u, 0u, 0u, 0u);
    pv[4 + s] = live ? __ldcs(reinterpret_cast<const uint4*>(b0 + row * ld + q * 16)) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void swb_take(uint4* stg, const uint4 (&pv)[8], uint32_t (&a)[16], uint32_t (&b)[16],
                                         int lane) {
  const int q = lane & 3;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = s * 8 + (lane >> 2);
      stg[r * 4 + (q ^ ((r >> 1) & 3))] = pv[4 * pass + s];
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = stg[lane * 4 + (i ^ ((lane >> 1) & 3))];
      uint32_t* d = pass ? b : a;
      d[4 * i] = v.x;
      d[4 * i + 1] = v.y;
      d[4 * i + 2] = v.z;
      d[4 * i + 3] = v.w;
    }
    __syncwarp();
  }
}

// The first chunk's loads of a tile (called before the accumulator wait).
template <int BN>
__device__ __forceinline__ void swb_issue_first(uint4 (&pv)[8], const GemmParams& p, int row0, int rows,
                                                int row_in_tile, int nt, int half, int ash, int live_end) {
  const SwbRows r = swb_rows(p, row0, rows, row_in_tile, ash, live_end);
  const int col0 = nt * BN + half * 32;
  if (r.valid > 0 && col0 < p.N) swb_issue(pv, r, p, col0, row_in_tile & 31);
}

// Epilogue of one tile for the 32 rows a warp owns: TMEM -> registers -> global.
// row_in_tile: this thread's row of the 128-row accumulator; rows: valid rows from row0.
// e4m3 operands: the accumulator is scaled by the A row's scale and each column's B-row
// scale; cs / cs_gate point at the B-row scales of this tile's first column.
// With 8 epilogue warps two share a lane quadrant and `half` (0 or 1) picks every other
// 32-column chunk.
// SwiGLU backward: ash = the tile group's A row shift, live_end = the group's end among A's rows;
// rows whose A row is past it are padding and get zeros.
// Router epilogue (EPI_ROUTER): the tile holds every logit of its 128 rows.  The four warps of half
// 0 take one row per thread; half 1 has nothing to do.  A thread streams its row's columns from
// TMEM (twice for softmax gating: the row maximum and the sum of exponentials first), adds the
// router bias, stores the logits if asked, forms score and selection key as the top-k kernel does,
// and keeps the kRouterFusedK best (key descending, lower expert index first on equal keys) in
// registers: columns arrive in ascending expert order, and a candidate goes to the first place
// whose key it strictly exceeds, the entries below moving down.  The first k entries are the
// choice; weights, the p-norm and the scalings follow as in the top-k kernel, summed over the k
// entries in order.
template <int BN>
__device__ __forceinline__ void router_epilogue(uint32_t tbase, int row0, int rows, int row_in_tile,
                                                const GemmParams& p, int half) {
  if (half != 0) return;
  constexpr int KM = kRouterFusedK;
  const RouterEpilogue& r = p.router;
  const bool live = row_in_tile < rows;
  const long long t = (long long)row0 + row_in_tile;
  const int E = p.N;
  float m = -FLT_MAX, inv = 1.f;
  if (r.gating == MOE_GATING_SOFTMAX) {
    float ssum = 0.f;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = cc * 32 + i;
          if (e >= E) continue;
          const float l = __uint_as_float(v[i]) + (r.b_router ? __ldg(r.b_router + e) : 0.f);
          if (pass == 0)
            m = fmaxf(m, l);
          else
            ssum += __expf(l - m);
        }
      }
    }
    inv = __fdividef(1.0f, ssum);
  }
  float tk[KM], ts[KM];
  int te[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    tk[j] = -INFINITY;
    ts[j] = 0.f;
    te[j] = INT_MAX;
  }
#pragma unroll 1
  for (int cc = 0; cc < BN / 32; ++cc) {
    uint32_t v[32];
    __syncwarp();
    tmem_ld_32x32b_x32(tbase + cc * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = cc * 32 + i;
      if (e >= E) continue;
      const float l = __uint_as_float(v[i]) + (r.b_router ? __ldg(r.b_router + e) : 0.f);
      if (r.logits && live) r.logits[t * E + e] = l;
      float sc = l;   // topk_softmax selects on the logits and weights the selected ones
      if (r.gating == MOE_GATING_SIGMOID)
        sc = __fdividef(1.0f, 1.0f + __expf(-l)) + r.sig_eps;
      else if (r.gating == MOE_GATING_SOFTMAX)
        sc = __expf(l - m) * inv;
      float kv = sc;
      if (r.score_bias) kv += __ldg(r.score_bias + e);
      if (!(kv == kv)) kv = -INFINITY;   // NaN never outranks a number
      if (kv > tk[KM - 1]) {
        // the candidate takes the first place whose key it strictly exceeds; from there on every
        // entry moves down one place (the list stays in order, equal keys keep their order)
        float ck = kv, cs = sc;
        int ce = e;
        bool moving = false;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (moving || ck > tk[j]) {
            const float tk0 = tk[j], ts0 = ts[j];
            const int te0 = te[j];
            tk[j] = ck; ts[j] = cs; te[j] = ce;
            ck = tk0; cs = ts0; ce = te0;
            moving = true;
          }
        }
      }
    }
  }
  if (!live) return;
  const int k = r.k;
  float w[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) w[j] = ts[j];
  if (r.gating == MOE_GATING_TOPK_SOFTMAX) {
    float mx = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) mx = fmaxf(mx, w[j]);
    float se = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      w[j] = j < k ? expf(w[j] - mx) : 0.f;
      se += w[j];
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) w[j] = w[j] / se;
  }
  if (r.p_norm > 0.f) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) acc += r.p_norm == 1.0f ? fabsf(w[j]) : r.p_norm == 2.0f ? w[j] * w[j] : powf(fabsf(w[j]), r.p_norm);
    const float nrm = r.p_norm == 1.0f ? acc : r.p_norm == 2.0f ? sqrtf(acc) : powf(acc, 1.0f / r.p_norm);
#pragma unroll
    for (int j = 0; j < KM; ++j) w[j] = w[j] / nrm;
  }
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    if (j >= k) break;
    float wj = w[j];
    if (r.restore) wj *= (float)k;
    if (r.ews != 0.f) wj *= r.ews;
    if (r.orig_k > 0 && r.orig_k != k) wj *= sqrtf((float)r.orig_k / (float)k);
    int ej = te[j];
    if (ej < 0 || ej >= E) {   // fewer than k experts (cannot happen for a validated config)
      set_status(p.status, MOE_ERR_BOUNDS);
      ej = 0;
    }
    r.idx[t * k + j] = ej;
    r.w[t * k + j] = wj;
  }
}

template <int BN, int EPI, bool F8 = false>
__device__ __forceinline__ void store_tile(uint32_t tbase, int row0, int rows, int row_in_tile, int nt, int split,
                                           const GemmParams& p, int half, uint4* stg, bool zero = false,
                                           const float* cs = nullptr, const float* cs_gate = nullptr, int ash = 0,
                                           int live_end = 0, uint4* pv_in = nullptr) {
  if constexpr (EPI == EPI_ROUTER) {
    router_epilogue<BN>(tbase, row0, rows, row_in_tile, p, half);
    return;
  }
  const bool row_ok = row_in_tile < rows;
  const long long row = (long long)row0 + row_in_tile;
  float rs = 1.0f;
  if (F8 && row_ok) {
    if (p.a_gather) {   // gathered A: the scale belongs to the source row
      const int src = p.a_gather[row];
      rs = src >= 0 ? p.a_scale[src] : 1.0f;
    } else {
      rs = p.a_scale[row];
    }
  }
  const int lane = row_in_tile & 31;
  const int valid = min(max(rows - (row_in_tile - lane), 0), 32);   // rows of this warp's 32 that exist
  const long long wrow0 = (long long)row0 + (row_in_tile - lane);
  if (EPI == EPI_SWIGLU_BWD) {
    // dH chunk (rounded to bf16) with the [u | g] of the same rows and columns; pv_in holds the
    // loads of the warp's first chunk, issued before the accumulator wait
    uint4(&pv)[8] = *reinterpret_cast<uint4(*)[8]>(pv_in);
    const SwbRows sr = swb_rows(p, row0, rows, row_in_tile, ash, live_end);
    const bool me = (sr.live >> lane) & 1u;
    __nv_bfloat16* dug = reinterpret_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo;
    __nv_bfloat16* hout = reinterpret_cast<__nv_bfloat16*>(p.out2) + wrow0 * p.ldo2;
#pragma unroll 1
    for (int cc = half; cc < BN / 32; cc += kEpiWarps / 4) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld_32x32b_x32(tbase + cc * 32, v);
      tmem_ld_wait();
      const int col0 = nt * BN + cc * 32;
      if (valid == 0 || col0 >= p.N) continue;   // warp-uniform
      uint32_t uw[16], gw[16];
      swb_take(stg, pv, uw, gw, lane);
      const int ncol = col0 + 32 * (kEpiWarps / 4);
      if (cc + kEpiWarps / 4 < BN / 32 && ncol < p.N) swb_issue(pv, sr, p, ncol, lane);
      uint32_t pu[16], pg[16], ph[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t dpk = me ? pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])) : 0u;
        float du0, dg0, h0, du1, dg1, h1;
        swiglu_bwd_elem(bf16_lo(uw[i]), bf16_lo(gw[i]), bf16_lo(dpk), du0, dg0, h0);
        swiglu_bwd_elem(bf16_hi(uw[i]), bf16_hi(gw[i]), bf16_hi(dpk), du1, dg1, h1);
        pu[i] = pack_bf16x2(du0, du1);
        pg[i] = pack_bf16x2(dg0, dg1);
        ph[i] = pack_bf16x2(h0, h1);
      }
      store_block_bf16(stg, pu, dug + col0, p.ldo, valid, lane);
      store_block_bf16(stg, pg, dug + p.N + col0, p.ldo, valid, lane);
      store_block_bf16(stg, ph, hout + col0, p.ldo2, valid, lane);
    }
  } else if (EPI == EPI_SWIGLU) {
    constexpr int HALF = BN / 2;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int cc = half; cc < HALF / 32; cc += kEpiWarps / 4) {
      uint32_t u[32], g[32];
      __syncwarp();
      tmem_ld_32x32b_x32(tbase + cc * 32, u);
      tmem_ld_32x32b_x32(tbase + HALF + cc * 32, g);
      tmem_ld_wait();
      const int col0 = nt * HALF + cc * 32;
      if (valid > 0 && col0 < p.N) {
        if (F8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            u[i] = __float_as_uint(__uint_as_float(u[i]) * rs * __ldg(cs + cc * 32 + i));
            g[i] = __float_as_uint(__uint_as_float(g[i]) * rs * __ldg(cs_gate + cc * 32 + i));
          }
        }
        if (p.preact) {   // the pre-activations [u | g] in bf16, kept for the backward
          __nv_bfloat16* pre = reinterpret_cast<__nv_bfloat16*>(p.preact) + wrow0 * p.preact_ld + col0;
          uint32_t pu[16], pg[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pu[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            pg[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
          }
          store_block_bf16(stg, pu, pre, p.preact_ld, valid, lane);
          store_block_bf16(stg, pg, pre + p.N, p.preact_ld, valid, lane);
        }
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
          const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
          // silu(g) = g / (1 + e^-g); the approximate division returns 0 when e^-g overflows
          const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
          const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
          packed[i] = pack_bf16x2(h0, h1);
        }
        store_block_bf16(stg, packed, out + wrow0 * p.ldo + col0, p.ldo, valid, lane);
      }
    }
  } else {
#pragma unroll 1
    for (int cc = half; cc < BN / 32; cc += kEpiWarps / 4) {
      uint32_t v[32];
      __syncwarp();
      if (zero) {  // empty contraction (a K-grouped group without rows): the product is zero
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      } else {
        tmem_ld_32x32b_x32(tbase + cc * 32, v);
        tmem_ld_wait();
      }
      const int col0 = nt * BN + cc * 32;
      if (valid == 0 || col0 >= p.N) continue;   // warp-uniform
      if (F8) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * rs * __ldg(cs + cc * 32 + i));
      }
      if (EPI == EPI_F32) {
        float* base = reinterpret_cast<float*>(p.out) + (long long)split * p.split_stride;
        if (col0 + 32 <= p.N && (p.ldo & 3) == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0) {
          // two 16-column halves, each a 32 x 64-byte block staged for row-contiguous stores
          char* out0 = reinterpret_cast<char*>(base + wrow0 * p.ldo + col0);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t words[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) words[i] = v[16 * hf + i];
            store_block_64b(stg, words, out0 + 64 * hf, p.ldo * 4, valid, lane);
          }
        } else if (row_ok) {
          float* out = base + row * p.ldo + col0;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) out[i] = __uint_as_float(v[i]);
        }
      } else {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        store_block_bf16(stg, packed, reinterpret_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo + col0, p.ldo, valid,
                         lane);
      }
    }
  }
}

// Producer of a gathered A operand (4 warps).  For every k-tile it copies the CTA's 128
// rows of the tile, row r from source row a_gather[row0 + r], into the stage's A region in the
// 128-byte-swizzled layout a TMA load writes (16-byte chunk c of row r at c ^ (r mod 8)).
// Thread t moves chunk (t & 7) of rows (t >> 3) + 16 j, so a warp instruction reads four whole
// 128-byte lines.  Rows past the tile's valid rows and -1 rows are zero-filled without reads.
// Each thread's copies for a stage end with a no-wait arrive on the CTA's gathered-rows barrier
// of that stage (128 arrivals); gather_a_relay takes it from there.
template <int ROWS, int NST, bool PAIR>
__device__ __forceinline__ void gather_a_load_rows(const GemmParams& p, const TileCoord& c, int t, int rank,
                                                   int (&tok)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 128 * rank + (t >> 3) + 16 * j;   // row of the tile
    tok[j] = r < c.rows ? __ldg(p.a_gather + c.row0 + r) : -1;
  }
}

template <int ROWS, int NST, bool PAIR>
__device__ __forceinline__ void gather_a_producer(const GemmParams& p, const int* s_toff, const int* s_goff,
                                                  int t_first, int t_step, int total_tiles, int rank, uint8_t* smem,
                                                  int stage_bytes, uint64_t* empty_bar, uint64_t* gath_bar,
                                                  volatile int* abort_flag) {
  const int t = threadIdx.x - kGatherThread0;
  const int lane = t & 31;
  const int chunk = t & 7;
  const uint64_t keep = l2_policy_evict_last();
  uint32_t stage = 0, phase = 0;
  bool ok = true;
  // the source rows of the next tile are loaded while the current one is copied
  int nxt[8];
  if (t_first < total_tiles)
    gather_a_load_rows<ROWS, NST, PAIR>(p, decode_tile<ROWS>(t_first, p, s_toff, s_goff), t, rank, nxt);
  for (int tile = t_first; tile < total_tiles && ok; tile += t_step) {
    const TileCoord c = decode_tile<ROWS>(tile, p, s_toff, s_goff);
    int tok[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int src = nxt[j];
      if (src < -1 || src >= p.a_src_rows) {
        set_status(p.status, MOE_ERR_BOUNDS);
        src = -1;
      }
      tok[j] = src;
    }
    if (tile + t_step < total_tiles)
      gather_a_load_rows<ROWS, NST, PAIR>(p, decode_tile<ROWS>(tile + t_step, p, s_toff, s_goff), t, rank, nxt);
    for (int kt = c.kt0; kt < c.kt1; ++kt) {
      int free_slot = 1;
      if (lane == 0)
        free_slot = (PAIR ? mbar_wait_cluster(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)
                          : mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status))
                        ? 1
                        : 0;
      if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
        ok = false;
        break;
      }
      const uint32_t sa = smem_u32(smem + stage * stage_bytes);
      const uint8_t* kb = p.a_src + (long long)kt * 128 + chunk * 16;
      // the copies of a stage, with or without the keep policy (two loops: no per-copy test)
      if (p.a_keep) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = (t >> 3) + 16 * j;
          const int src = tok[j];
          cp_async_16_hint(sa + r * 128 + ((chunk ^ (r & 7)) << 4),
                           kb + (long long)(src < 0 ? 0 : src) * p.a_ld_bytes, src < 0 ? 0u : 16u, keep);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = (t >> 3) + 16 * j;
          const int src = tok[j];
          cp_async_16(sa + r * 128 + ((chunk ^ (r & 7)) << 4), kb + (long long)(src < 0 ? 0 : src) * p.a_ld_bytes,
                      src < 0 ? 0u : 16u);
        }
      }
      cp_async_arrive_noinc(&gath_bar[stage]);
      if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1u; }
    }
  }
  cp_async_wait_all();   // every copy lands before the CTA's shared memory can go away
}

// One thread per CTA: for every stage, in order, waits until the CTA's gathered rows have
// landed, fences them into the async proxy (the tensor core reads shared memory through it)
// and arrives on the stage's full barrier, which on a CTA pair is CTA 0's.  It issues no
// copies itself, so neither the fence nor the arrive waits on copies of later stages.
template <int ROWS, int NST, bool PAIR>
__device__ __forceinline__ void gather_a_relay(const GemmParams& p, const int* s_toff, const int* s_goff, int t_first,
                                               int t_step, int total_tiles, uint64_t* gath_bar, uint64_t* full_bar,
                                               volatile int* abort_flag) {
  uint32_t stage = 0, phase = 0;
  for (int tile = t_first; tile < total_tiles; tile += t_step) {
    const TileCoord c = decode_tile<ROWS>(tile, p, s_toff, s_goff);
    for (int kt = c.kt0; kt < c.kt1; ++kt) {
      if (!(PAIR ? mbar_wait_cluster(&gath_bar[stage], phase, abort_flag, p.status)
                 : mbar_wait(&gath_bar[stage], phase, abort_flag, p.status)))
        return;
      fence_proxy_async_smem();
      // CTA 1's rows stay in its own shared memory and its own tensor core reads them, so the
      // arrive on CTA 0's barrier keeps the default CTA-scope release: a cluster-scope release
      // cost ~0.5 us per stage here and halved the GEMM's speed
      if (PAIR)
        mbar_arrive_cluster(map_to_cta(smem_u32(&full_bar[stage]), 0));
      else
        mbar_arrive(&full_bar[stage]);
      if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1u; }
    }
  }
}

template <int BN, int EPI, bool F8 = false, bool GA = false>
__global__ void __launch_bounds__(GA ? kThreadsGA : kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* gath_bar = tempty_bar + 2;   // gathered A only
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::HOLDER_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::ABORT_OFF);
  int* s_toff = reinterpret_cast<int*>(smem + C::TABLE_OFF);
  int* s_goff = s_toff + (kMaxGroups + 1);
  int* s_aoff = s_goff + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Group tables into shared memory.
  int total_tiles;
  if (p.num_groups > 0) {
    for (int i = threadIdx.x; i <= p.num_groups; i += blockDim.x) {
      s_toff[i] = p.tile_off[i];
      s_goff[i] = p.group_off[i];
    }
  } else if (p.k_groups > 0) {
    for (int i = threadIdx.x; i <= p.k_groups; i += blockDim.x) s_goff[i] = p.k_off[i];
  }
  if (p.a_off)
    for (int i = threadIdx.x; i <= max(p.num_groups, p.k_groups); i += blockDim.x) s_aoff[i] = p.a_off[i];
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], GA ? 2 : 1);   // producer arrive (+ the gathered rows' relay)
      mbar_init(&empty_bar[s], 1);
      if (GA) mbar_init(&gath_bar[s], 32 * kGatherWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], kEpiWarps * 32);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    if (!GA) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  {
    const int mtiles = p.num_groups > 0 ? s_toff[p.num_groups] : (p.M + BM - 1) / BM;
    total_tiles = mtiles * p.n_tiles * (p.k_groups > 0 ? p.k_groups : p.splits);
  }

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const TileCoord c = decode_tile(t, p, s_toff, s_goff);
        const int ash = a_row_shift(p, c, s_goff, s_aoff);
        const int brow = c.group * p.b_rows_per_group + c.nt * (EPI == EPI_SWIGLU ? BN / 2 : BN);
        bool ok = true;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], GA ? C::B_BYTES : C::STAGE_BYTES);
          const int kx = kt * (F8 ? 2 * BK : BK);   // 128 bytes of K per k-tile: 64 bf16 or 128 e4m3
          if (p.a_mn) {   // MN-major A: 64 K rows x 128 M columns as two 64-column blocks (8 KB each)
            tma_load_2d(sa, &tmA, &full_bar[stage], c.row0, kt * BK + ash);
            tma_load_2d(sa + 8192, &tmA, &full_bar[stage], c.row0 + 64, kt * BK + ash);
          } else if (!GA) {
            tma_load_2d(sa, &tmA, &full_bar[stage], kx, c.row0 + ash);
          }
          if (EPI == EPI_SWIGLU) {
            tma_load_2d(sb, &tmB, &full_bar[stage], kx, brow);
            tma_load_2d(sb + C::B_BYTES / 2, &tmB, &full_bar[stage], kx, brow + p.b_gate_offset);
          } else if (p.b_mn) {   // MN-major B: 64 K rows x BN columns, as BN / 64 blocks of 64 columns (8 KB)
            for (int b = 0; b < BN / 64; ++b)
              tma_load_2d(sb + b * 8192, &tmB, &full_bar[stage], c.nt * BN + 64 * b,
                          c.group * p.b_rows_per_group + kt * BK);
          } else {
            tma_load_2d(sb, &tmB, &full_bar[stage], kx, brow);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- UMMA issuer ----------------
      constexpr uint32_t idesc = F8 ? umma_idesc_e4m3_f32(BM, BN) : umma_idesc_bf16_f32(BM, BN);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const TileCoord c = decode_tile(t, p, s_toff, s_goff);
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1u) ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::ACC_STRIDE);
        bool ok = true;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          // a K-major operand advances 32 bytes per MMA inside its swizzled rows, an MN-major one by
          // two 8-row K groups (2048 bytes)
          const uint64_t a_desc = p.a_mn ? umma_sdesc_mn_sw128(sa, 8192) : umma_sdesc_sw128(sa);
          const uint64_t b_desc = p.b_mn ? umma_sdesc_mn_sw128(sa + C::A_BYTES, 8192) : umma_sdesc_sw128(sa + C::A_BYTES);
          const uint64_t a_step = p.a_mn ? 2048 / 16 : 2;
          const uint64_t b_step = p.b_mn ? 2048 / 16 : 2;
          // bits 15 / 16 of the instruction descriptor: A / B is MN-major
          const uint32_t id = idesc | (p.a_mn ? (1u << 15) : 0u) | (p.b_mn ? (1u << 16) : 0u);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // one MMA takes 32 bytes of K (16 bf16 or 32 e4m3)
            if (F8)
              umma_e4m3(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, id, (kt > c.kt0 || kk > 0) ? 1u : 0u);
            else
              umma_bf16(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, id, (kt > c.kt0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);
      }
    }
  } else if (warp < 2 + kEpiWarps) {
    // ---------------- epilogue: warps 2..9 ----------------
    const int quad = warp & 3;                    // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;             // which alternate column chunks
    const int row_in_tile = quad * 32 + lane;
    uint4* stg = reinterpret_cast<uint4*>(smem + C::EPI_OFF) + (warp - 2) * 128;
    int it = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const TileCoord c = decode_tile(t, p, s_toff, s_goff);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int ash = 0, live_end = 0;
      uint4 pv[8];
      if (EPI == EPI_SWIGLU_BWD) {
        ash = a_row_shift(p, c, s_goff, s_aoff);
        live_end = s_aoff[c.group + 1];
        swb_issue_first<BN>(pv, p, c.row0, c.rows, row_in_tile, c.nt, half, ash, live_end);
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull_bar[acc], use & 1u, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * C::ACC_STRIDE);
      const float* cs = nullptr;
      const float* cs_gate = nullptr;
      if (F8) {
        const int brow = c.group * p.b_rows_per_group + c.nt * (EPI == EPI_SWIGLU ? BN / 2 : BN);
        cs = p.b_scale + brow;
        cs_gate = cs + p.b_gate_offset;
      }
      store_tile<BN, EPI, F8>(tbase, c.row0, c.rows, row_in_tile, c.nt, c.split, p, half, stg, c.kt1 <= c.kt0, cs,
                              cs_gate, ash, live_end, pv);
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
  } else if constexpr (GA) {
    if (warp < kRelayWarp) {
      // ---------------- gathered A rows: warps 10..13 ----------------
      gather_a_producer<BM, C::STAGES, false>(p, s_toff, s_goff, blockIdx.x, gridDim.x, total_tiles, 0, smem,
                                              C::STAGE_BYTES, empty_bar, gath_bar, abort_flag);
    } else if (lane == 0) {
      gather_a_relay<BM, C::STAGES, false>(p, s_toff, s_goff, blockIdx.x, gridDim.x, total_tiles, gath_bar, full_bar,
                                           abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let copies and MMAs already in flight land before the CTA's shared memory and TMEM go away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) { }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// MXFP8 operands (OCP microscaling): A and B are e4m3 codes, and every 32 consecutive K values
// of a row share one power-of-two scale 2^(s - 127), s an unsigned byte (E8M0).  The tensor core
// applies the scales itself (tcgen05.mma ... kind::mxf8f6f4.block_scale): each MMA (K = 32) reads
// one scale per A row and one per B row from tensor memory.
//
// One CTA, 128 x 256 tiles, a single accumulator (TMEM columns 0..255), the 4-stage ring of
// GemmCfg<256> (16 KB of A codes + 32 KB of B codes per stage).  Stage s, MMA j of the stage's
// four, takes its A scales from TMEM columns 256 + 64 s + 16 j .. +3 and its B scales from the
// 8 columns after 256 + 64 s + 16 j + 8:
//   A row m:  lane m, column (m / 32), byte 0;
//   B row n:  column (n / 32), byte 0, lane (n % 32) of every lane quadrant (the quadrant of
//             the accumulator row being computed is the one read).
// Four scale-writer warps (one per lane quadrant) copy a stage's scales from global memory into
// those columns with tcgen05.st once the stage's previous MMAs have finished (the empty barrier),
// then arrive on the stage's scale barrier, which the MMA issuer waits on beside the TMA barrier.
// Warps: 0 TMA producer, 1 MMA issuer, 2..9 epilogue, 10..13 scale writers.
// ---------------------------------------------------------------------------
constexpr int kMxScaleWarp0 = 2 + kEpiWarps;
constexpr int kThreadsMX = 32 * (kMxScaleWarp0 + 4);

__device__ __forceinline__ uint32_t mx_col_a(int stage, int j) { return 256u + 64u * stage + 16u * j; }

__device__ __forceinline__ uint32_t uint4_word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// The 16-byte words of block scales for k-tiles [4 g, 4 g + 4) of the tile: this lane's A row
// (row 32 quad + lane of the tile) and B rows 32 i + lane, i = 0..7 (SwiGLU: rows 0..127 of the
// tile are the up rows, 128..255 the gate rows); rows past an operand read 2^0 (byte 127), their
// products are never stored.
template <int EPI>
__device__ __forceinline__ void mx_load_scales(const GemmParams& p, const TileCoord& c, int quad, int lane, int g,
                                               uint4& a, uint4 (&b)[8]) {
  constexpr int b_tile_rows = EPI == EPI_SWIGLU ? 128 : 256;
  const uint4 one = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const long long arow = (long long)c.row0 + quad * 32 + lane;
  a = arow < p.mx_a_rows ? __ldg(reinterpret_cast<const uint4*>(p.mx_a_scale + arow * p.mx_a_ld) + g) : one;
  const long long base = (long long)c.group * p.b_rows_per_group + (long long)c.nt * b_tile_rows;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = 32 * i + lane;
    const long long brow = base + (EPI == EPI_SWIGLU && i >= 4 ? p.b_gate_offset + n - 128 : n);
    b[i] = brow < p.mx_b_rows ? __ldg(reinterpret_cast<const uint4*>(p.mx_b_scale + brow * p.mx_b_ld) + g) : one;
  }
}

// MXFP8 epilogue of one tile for the 32 rows a warp owns.  The warp reads its whole share of
// the accumulator (every other 32-column chunk) into registers, already converted (SwiGLU: 64 h
// values, bf16 out: 128 values, packed in bf16 pairs), and releases the accumulator before its
// global stores, so the next tile's MMAs run while this tile is written out.  With mx_out_codes
// (SwiGLU), each thread's 32 h values of a chunk, rounded to bf16, are one MXFP8 block of its row:
// they leave as 32 e4m3 codes and a scale byte, the next GEMM's A operand.
template <int EPI>
__device__ __forceinline__ void mx_store_tile(uint32_t tbase, const TileCoord& c, int row_in_tile,
                                              const GemmParams& p, int half, uint4* stg, uint64_t* tempty) {
  constexpr int CHUNKS = EPI == EPI_SWIGLU ? 2 : 4;   // 32-column output chunks of this warp
  const int lane = row_in_tile & 31;
  const int valid = min(max(c.rows - (row_in_tile - lane), 0), 32);
  const long long wrow0 = (long long)c.row0 + (row_in_tile - lane);
  uint32_t packed[CHUNKS][16];
  __syncwarp();
#pragma unroll
  for (int q = 0; q < CHUNKS; ++q) {
    const int cc = half + 2 * q;
    if (EPI == EPI_SWIGLU) {   // u in columns [0, 128), g in [128, 256)
      uint32_t u[32], g[32];
      tmem_ld_32x32b_x32(tbase + cc * 32, u);
      tmem_ld_32x32b_x32(tbase + 128 + cc * 32, g);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
        // silu(g) = g / (1 + e^-g); the approximate division returns 0 when e^-g overflows
        const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(u[2 * i]);
        const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(u[2 * i + 1]);
        packed[q][i] = pack_bf16x2(h0, h1);
      }
    } else {   // 16 columns at a time: fewer live registers beside the 64 packed words
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tbase + cc * 32 + 16 * h, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          packed[q][8 * h + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      }
    }
  }
  tc_fence_before();
  mbar_arrive(tempty);
  constexpr int out_cols = EPI == EPI_SWIGLU ? 128 : 256;   // output columns per tile
  if (EPI == EPI_SWIGLU && p.mx_out_codes) {
    const long long row = wrow0 + lane;
#pragma unroll
    for (int q = 0; q < CHUNKS; ++q) {
      const int col0 = c.nt * out_cols + (half + 2 * q) * 32;
      if (lane < valid && col0 < p.N) {
        uint32_t codes[8];
        const uint32_t e = mx_quantize_block(packed[q], codes);
        uint4* dst = reinterpret_cast<uint4*>(p.mx_out_codes + row * p.ldo + col0);
        dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        p.mx_out_scale[row * p.mx_out_ld + col0 / 32] = (uint8_t)e;
      }
    }
    return;
  }
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo;
#pragma unroll
  for (int q = 0; q < CHUNKS; ++q) {
    const int col0 = c.nt * out_cols + (half + 2 * q) * 32;
    if (valid > 0 && col0 < p.N) store_block_bf16(stg, packed[q], out + col0, p.ldo, valid, lane);
  }
}

template <int EPI>
__global__ void __launch_bounds__(kThreadsMX, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  pdl_wait();
  pdl_trigger();
  using C = GemmCfg<256>;
  static_assert(C::STAGES == 4, "the scale columns of TMEM hold four stages");
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* sfull_bar = tempty_bar + 2;   // the stage's scales are in TMEM
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::HOLDER_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::ABORT_OFF);
  int* s_toff = reinterpret_cast<int*>(smem + C::TABLE_OFF);
  int* s_goff = s_toff + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (p.num_groups > 0)
    for (int i = threadIdx.x; i <= p.num_groups; i += blockDim.x) {
      s_toff[i] = p.tile_off[i];
      s_goff[i] = p.group_off[i];
    }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&sfull_bar[s], 4);   // one arrive per scale-writer warp
    }
    mbar_init(&tfull_bar[0], 1);
    mbar_init(&tempty_bar[0], kEpiWarps * 32);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int mtiles = p.num_groups > 0 ? s_toff[p.num_groups] : (p.M + BM - 1) / BM;
  const int total_tiles = mtiles * p.n_tiles;
  constexpr int b_tile_rows = EPI == EPI_SWIGLU ? BN / 2 : BN;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const TileCoord c = decode_tile(t, p, s_toff, s_goff);
        const int brow = c.group * p.b_rows_per_group + c.nt * b_tile_rows;
        bool ok = true;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
          const int kx = kt * 128;   // 128 e4m3 of K per k-tile
          tma_load_2d(sa, &tmA, &full_bar[stage], kx, c.row0);
          if (EPI == EPI_SWIGLU) {
            tma_load_2d(sb, &tmB, &full_bar[stage], kx, brow);
            tma_load_2d(sb + C::B_BYTES / 2, &tmB, &full_bar[stage], kx, brow + p.b_gate_offset);
          } else {
            tma_load_2d(sb, &tmB, &full_bar[stage], kx, brow);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- UMMA issuer ----------------
      constexpr uint32_t idesc = umma_idesc_mx_e4m3(BM, BN);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const TileCoord c = decode_tile(t, p, s_toff, s_goff);
        if (!mbar_wait(&tempty_bar[0], ((uint32_t)it & 1u) ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        bool ok = true;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.status) ||
              !mbar_wait(&sfull_bar[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t a_desc = umma_sdesc_sw128(sa);
          const uint64_t b_desc = umma_sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // one MMA takes 32 e4m3 of K: 32 bytes further along the swizzled rows
            const uint32_t ca = tmem_base + mx_col_a(stage, j);
            umma_mx_e4m3(tmem_base, a_desc + 2 * j, b_desc + 2 * j, idesc, ca, ca + 8,
                         (kt > c.kt0 || j > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[0]);
      }
    }
  } else if (warp < kMxScaleWarp0) {
    // ---------------- epilogue: warps 2..9 ----------------
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quad * 32 + lane;
    uint4* stg = reinterpret_cast<uint4*>(smem + C::EPI_OFF) + (warp - 2) * 128;
    int it = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      const TileCoord c = decode_tile(t, p, s_toff, s_goff);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull_bar[0], (uint32_t)it & 1u, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      mx_store_tile<EPI>(tmem_base + ((uint32_t)(quad * 32) << 16), c, row_in_tile, p, half, stg, &tempty_bar[0]);
    }
  } else {
    // ---------------- scale writers: warps 10..13, one per lane quadrant ----------------
    // A row's scales for four k-tiles are one aligned 16-byte word; the words of the next group of
    // four k-tiles are loaded while this group's are written, so an L2 round trip is paid once per
    // four k-tiles and overlaps the MMAs instead of once per k-tile in series with them
    const int quad = warp & 3;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    const int groups = (p.kt_total + 3) / 4;
    uint32_t stage = 0, phase = 0;
    int t = blockIdx.x, g = 0;
    TileCoord c{};
    uint4 ca{}, cb[8]{};
    if (t < total_tiles) {
      c = decode_tile(t, p, s_toff, s_goff);
      mx_load_scales<EPI>(p, c, quad, lane, 0, ca, cb);
    }
    bool ok = true;
    while (ok && t < total_tiles) {
      int tn = t, gn = g + 1;
      if (gn == groups) { tn = t + gridDim.x; gn = 0; }
      TileCoord cn = c;
      uint4 na{}, nb[8]{};
      if (tn < total_tiles) {
        if (tn != t) cn = decode_tile(tn, p, s_toff, s_goff);
        mx_load_scales<EPI>(p, cn, quad, lane, gn, na, nb);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (!ok || 4 * g + kk >= c.kt1) break;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        const uint32_t wa = uint4_word(ca, kk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t col = mx_col_a(stage, j);
          tmem_st_32x32b_x1(lane_base + col + quad, (wa >> (8 * j)) & 0xFFu);
          uint32_t v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = (uint4_word(cb[i], kk) >> (8 * j)) & 0xFFu;
          tmem_st_32x32b_x8(lane_base + col + 8, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull_bar[stage]);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      ca = na;
#pragma unroll
      for (int i = 0; i < 8; ++i) cb[i] = nb[i];
      c = cn;
      t = tn;
      g = gn;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) { }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}


// ---------------------------------------------------------------------------
// CTA-pair variant: a cluster of two CTAs computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2.  CTA r stages A rows [128r, 128r+128) of the tile
// and B rows [128r, 128r+128) of the 256-row B tile (for SwiGLU: CTA 0 the 128
// "up" rows, CTA 1 the 128 "gate" rows), so a stage is 32 KB per CTA and the
// ring is 6 deep.  Only CTA 0 issues MMAs; both CTAs' TMA loads complete on
// CTA 0's full barrier; MMA completion is multicast to both CTAs' empty and
// accumulator-full barriers; both epilogues release the accumulator on CTA 0.
// ---------------------------------------------------------------------------
constexpr int BM2 = 256;

// Wide-tile epilogue for one 256-column accumulator with bf16 out (bf16 operands): the warp takes
// its whole share of the accumulator (4 chunks of 32 columns) into registers as packed bf16,
// releases the accumulator, and only then stores, so the next tile's MMAs into this accumulator
// start while the stores drain.  Releasing after the stores, as the 256-column tiles do, left
// grouped GEMM 2 slower on wide tiles than on 256-column ones.
__device__ __forceinline__ void drain_wide_bf16(uint32_t tb, int row0, int rows, int row_in_tile, int nt,
                                                const GemmParams& p, int half, uint4* stg, uint64_t* tempty) {
  const int lane = row_in_tile & 31;
  const int valid = min(max(rows - (row_in_tile - lane), 0), 32);
  const long long wrow0 = (long long)row0 + (row_in_tile - lane);
  uint32_t pk[4][16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tb + (half + 2 * i) * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 16; ++q) pk[i][q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(tempty), 0));
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int col0 = nt * 256 + (half + 2 * i) * 32;
    if (valid > 0 && col0 < p.N) store_block_bf16(stg, pk[i], out + col0, p.ldo, valid, lane);
  }
}

// SwiGLU backward: 4 stages, and a ring of [u | g] boxes for the epilogue (2 slots for each
// half of the epilogue warps, 16 KB each: 128 rows x 32 columns of u and of g), with a full and
// an empty barrier per slot.
// W2 (wide tiles, bf16 out): a tile spans two adjacent 256-column n-tiles that share each k-tile
// of A; a stage holds A and both n-tiles' B halves (48 KB, 4 stages), and the two accumulators
// (TMEM columns 0-255 and 256-511) hold the tile's two n-tiles instead of alternating between tiles.
template <int EPI, bool W2 = false>
struct PairCfgT {
  static constexpr bool SWB = EPI == EPI_SWIGLU_BWD;
  static_assert(!(W2 && SWB), "wide tiles: forward epilogues only");
  static constexpr int BN = 256;                            // columns of one accumulator
  static constexpr int NB = W2 ? 2 : 1;                     // n-tiles per tile
  static constexpr int A_BYTES = 128 * BK * 2;
  static constexpr int B_BYTES = NB * (BN / 2) * BK * 2;
  static constexpr int B_PART = (BN / 2) * BK * 2;          // one n-tile's B half
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = W2 ? 4 : (SWB ? 4 : 6);
  static constexpr int ACC_STRIDE = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr int PRE_SLOTS = 2;                       // per half of the epilogue warps
  static constexpr int PRE_SLOT_BYTES = 2 * 128 * 64;       // u box + g box
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 3 * STAGES + 4 + (SWB ? 2 * 2 * PRE_SLOTS : 0);
  static constexpr int HOLDER_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int ABORT_OFF = HOLDER_OFF + 4;
  static constexpr int TABLE_OFF = (ABORT_OFF + 4 + 15) & ~15;
  static constexpr int EPI_OFF = (TABLE_OFF + 3 * (kMaxGroups + 1) * 4 + 127) & ~127;
  static constexpr int PRE_OFF = (EPI_OFF + kEpiStageBytes + 1023) & ~1023;
  static constexpr int SMEM_BYTES = PRE_OFF + (SWB ? 2 * PRE_SLOTS * PRE_SLOT_BYTES : 0) + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Producer of a gathered, MN-major B operand of the K-grouped pair GEMM (4 warps of each CTA):
// for every k-tile the group's 64 K rows, row r from source row b_gather[b_goff[g] + local row]
// (zeros past the group's count), this CTA's 128 of the tile's 256 N columns as two 64-column
// blocks, in the 128-byte-swizzled layout a TMA load of 64 x 64 boxes writes.  Thread t moves
// chunk (t & 7) of rows (t >> 3) + 16 j of both blocks; the next k-tile's source rows are loaded
// while the current one is copied.  Arrivals and the relay work as for a gathered A.
template <int NST>
__device__ __forceinline__ void gather_b_mn_producer(const GemmParams& p, const int* s_toff, const int* s_goff,
                                                     int t_first, int t_step, int total_tiles, int rank,
                                                     uint8_t* smem, int stage_bytes, int a_bytes, uint64_t* empty_bar,
                                                     uint64_t* gath_bar, volatile int* abort_flag) {
  const int t = threadIdx.x - kGatherThread0;
  const int lane = t & 31;
  const int chunk = t & 7;
  uint32_t stage = 0, phase = 0;
  bool ok = true;
  for (int tile = t_first; tile < total_tiles && ok; tile += t_step) {
    const TileCoord c = decode_tile<BM2>(tile, p, s_toff, s_goff);
    const int goff = __ldg(p.b_goff + c.group);
    const int cnt = __ldg(p.b_goff + c.group + 1) - goff;
    const int col0 = c.nt * 256 + 128 * rank;   // this CTA's first N column
    // loads only: the values are checked one k-tile later, so the loads' latency is not waited on
    auto rows_of = [&](int kt, int (&raw)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rl = (kt - c.kt0) * 64 + (t >> 3) + 16 * j;
        raw[j] = rl < cnt ? __ldg(p.b_gather + goff + rl) : -1;
      }
    };
    int nxt[4];
    if (c.kt0 < c.kt1) rows_of(c.kt0, nxt);
    for (int kt = c.kt0; kt < c.kt1; ++kt) {
      int tok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int src = nxt[j];
        if (src < -1 || src >= p.b_src_rows) {
          set_status(p.status, MOE_ERR_BOUNDS);
          src = -1;
        }
        tok[j] = src;
      }
      if (kt + 1 < c.kt1) rows_of(kt + 1, nxt);
      int free_slot = 1;
      if (lane == 0) free_slot = mbar_wait_cluster(&empty_bar[stage], phase ^ 1u, abort_flag, p.status) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
        ok = false;
        break;
      }
      const uint32_t sb = smem_u32(smem + stage * stage_bytes + a_bytes);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int col = col0 + 64 * b + 8 * chunk;
        const bool col_ok = col < p.N;
        const uint8_t* cb = p.b_src + (long long)col * 2;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = (t >> 3) + 16 * j;
          const int src = col_ok ? tok[j] : -1;
          cp_async_16(sb + b * 8192 + r * 128 + ((chunk ^ (r & 7)) << 4),
                      cb + (long long)(src < 0 ? 0 : src) * p.b_ld_bytes, src < 0 ? 0u : 16u);
        }
      }
      cp_async_arrive_noinc(&gath_bar[stage]);
      if (++stage == (uint32_t)NST) { stage = 0; phase ^= 1u; }
    }
  }
  cp_async_wait_all();   // every copy lands before the CTA's shared memory can go away
}

// SwiGLU backward on CTA pairs: the [u | g] pre-activations reach the epilogue through TMA boxes
// (128 rows x 32 columns of u and of g, 64-byte swizzle) in a 2-slot ring per half of the
// epilogue warps.  The half's first warp issues chunk j + 2 once all four warps have taken
// chunk j; the first two chunks of a tile are issued before its accumulator wait.  Chunk j of a
// half covers columns (half + 2 j) * 32 of the tile; rows come from preact at the CTA's output
// rows, shifted like A's when preact_dense.
template <class C>
__device__ __forceinline__ void swb_pre_issue(const GemmParams& p, const CUtensorMap* tmP, uint8_t* smem,
                                              uint64_t* pre_full, uint64_t* pre_empty, int half, uint32_t& issued,
                                              const TileCoord& c, int rank, int ash, int j, volatile int* abort_flag) {
  const int col0 = c.nt * C::BN + (half + 2 * j) * 32;
  if (col0 >= p.N) return;
  const uint32_t n = issued++;
  const int slot = half * C::PRE_SLOTS + (int)(n % C::PRE_SLOTS);
  const uint32_t ph = (n / C::PRE_SLOTS) & 1u;
  if (!mbar_wait(&pre_empty[slot], ph ^ 1u, abort_flag, p.status)) return;
  uint8_t* dst = smem + C::PRE_OFF + slot * C::PRE_SLOT_BYTES;
  const int drow = c.row0 + 128 * rank + (p.preact_dense ? ash : 0);
  mbar_arrive_expect_tx(&pre_full[slot], C::PRE_SLOT_BYTES);
  tma_load_2d(dst, tmP, &pre_full[slot], col0, drow);
  tma_load_2d(dst + C::PRE_SLOT_BYTES / 2, tmP, &pre_full[slot], p.N + col0, drow);
}

template <class C>
__device__ __forceinline__ void swb_pair_tile(uint32_t tbase, const TileCoord& c, int rank, int row_in_tile,
                                              const GemmParams& p, int half, uint4* stg, uint8_t* smem,
                                              const CUtensorMap* tmP, uint64_t* pre_full, uint64_t* pre_empty,
                                              bool pre_issuer, uint32_t& issued, uint32_t& used, int ash,
                                              int live_end, volatile int* abort_flag) {
  const int lane = row_in_tile & 31;
  const int crows = c.rows - 128 * rank;
  const long long wrow0 = (long long)c.row0 + 128 * rank + (row_in_tile - lane);
  const int valid = min(max(crows - (row_in_tile - lane), 0), 32);
  const bool me = lane < valid && wrow0 + lane + ash < (long long)live_end;
  __nv_bfloat16* dug = reinterpret_cast<__nv_bfloat16*>(p.out) + wrow0 * p.ldo;
  __nv_bfloat16* hout = reinterpret_cast<__nv_bfloat16*>(p.out2) + wrow0 * p.ldo2;
  const int sw = (row_in_tile >> 1) & 3;   // the 64-byte swizzle of this row's 16-byte chunks
#pragma unroll 1
  for (int j = 0; j < C::BN / 64; ++j) {
    const int cc = half + 2 * j;
    uint32_t v[32];
    __syncwarp();
    tmem_ld_32x32b_x32(tbase + cc * 32, v);
    tmem_ld_wait();
    const int col0 = c.nt * C::BN + cc * 32;
    if (crows <= 0 || col0 >= p.N) continue;   // the same for the whole half: no chunk was issued
    const uint32_t n = used++;
    const int slot = half * C::PRE_SLOTS + (int)(n % C::PRE_SLOTS);
    mbar_wait(&pre_full[slot], (n / C::PRE_SLOTS) & 1u, abort_flag, p.status);
    const uint8_t* su = smem + C::PRE_OFF + slot * C::PRE_SLOT_BYTES + row_in_tile * 64;
    uint32_t uw[16], gw[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 a = *reinterpret_cast<const uint4*>(su + ((q ^ sw) << 4));
      const uint4 b = *reinterpret_cast<const uint4*>(su + C::PRE_SLOT_BYTES / 2 + ((q ^ sw) << 4));
      uw[4 * q] = a.x; uw[4 * q + 1] = a.y; uw[4 * q + 2] = a.z; uw[4 * q + 3] = a.w;
      gw[4 * q] = b.x; gw[4 * q + 1] = b.y; gw[4 * q + 2] = b.z; gw[4 * q + 3] = b.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pre_empty[slot]);
    if (pre_issuer && j + C::PRE_SLOTS < C::BN / 64)
      swb_pre_issue<C>(p, tmP, smem, pre_full, pre_empty, half, issued, c, rank, ash, j + C::PRE_SLOTS, abort_flag);
    if (valid == 0) continue;
    uint32_t pu[16], pg[16], ph[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // a padding row (its A row belongs to the next expert, or is past A) gets zeros
      const uint32_t dpk = me ? pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])) : 0u;
      const uint32_t u2 = me ? uw[i] : 0u, g2 = me ? gw[i] : 0u;
      float du0, dg0, h0, du1, dg1, h1;
      swiglu_bwd_elem(bf16_lo(u2), bf16_lo(g2), bf16_lo(dpk), du0, dg0, h0);
      swiglu_bwd_elem(bf16_hi(u2), bf16_hi(g2), bf16_hi(dpk), du1, dg1, h1);
      pu[i] = pack_bf16x2(du0, du1);
      pg[i] = pack_bf16x2(dg0, dg1);
      ph[i] = pack_bf16x2(h0, h1);
    }
    store_block_bf16(stg, pu, dug + col0, p.ldo, valid, lane);
    store_block_bf16(stg, pg, dug + p.N + col0, p.ldo, valid, lane);
    store_block_bf16(stg, ph, hout + col0, p.ldo2, valid, lane);
  }
}

// GB: the B operand of a K-grouped fp32 GEMM is gathered by the kernel (gather_b_mn_producer).
// W2: wide tiles (PairCfgT); p.n_tiles counts tiles of two n-tiles, tile nt covering n-tiles 2 nt
// and 2 nt + 1.
template <int EPI, bool F8 = false, bool GA = false, bool GB = false, bool W2 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GA || GB ? kThreadsGA : kThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmP, const GemmParams p) {
  pdl_wait();   // the previous kernel on the stream is done (programmatic launch, see launch_pdl)
  pdl_trigger();
  using C = PairCfgT<EPI, W2>;
  static_assert(!W2 || (EPI == EPI_BF16 && !F8 && !GA && !GB), "wide tiles: bf16 out, TMA-loaded operands");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* gath_bar = tempty_bar + 2;   // gathered A only
  uint64_t* pre_full = tempty_bar + 2;   // SwiGLU backward only: [half][slot]
  uint64_t* pre_empty = pre_full + 2 * C::PRE_SLOTS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::HOLDER_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::ABORT_OFF);
  int* s_toff = reinterpret_cast<int*>(smem + C::TABLE_OFF);
  int* s_goff = s_toff + (kMaxGroups + 1);
  int* s_aoff = s_goff + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (p.num_groups > 0) {
    for (int i = threadIdx.x; i <= p.num_groups; i += blockDim.x) {
      s_toff[i] = p.tile_off[i];
      s_goff[i] = p.group_off[i];
    }
  } else if (p.k_groups > 0) {
    for (int i = threadIdx.x; i <= p.k_groups; i += blockDim.x) s_goff[i] = p.k_off[i];
  }
  if (p.a_off)
    for (int i = threadIdx.x; i <= max(p.num_groups, p.k_groups); i += blockDim.x) s_aoff[i] = p.a_off[i];
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      // CTA 0 only: its producer's arrive + both CTAs' bytes (+ both CTAs' gathered-rows relays)
      mbar_init(&full_bar[s], GA || GB ? 3 : 1);
      if (GA || GB) mbar_init(&gath_bar[s], 32 * kGatherWarps);
      mbar_init(&empty_bar[s], 1);    // one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);    // one multicast commit per tile
      mbar_init(&tempty_bar[a], 2 * kEpiWarps);   // CTA 0 only: one lane of each epilogue warp of both CTAs
    }
    if constexpr (C::SWB) {
      for (int i = 0; i < 2 * C::PRE_SLOTS; ++i) {
        mbar_init(&pre_full[i], 1);                 // the half's issuing thread (+ the boxes' bytes)
        mbar_init(&pre_empty[i], kEpiWarps / 2);    // one lane of each warp of the half
      }
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    if (!GA) tma_prefetch_desc(&tmA);
    if (!GB) tma_prefetch_desc(&tmB);
    if constexpr (C::SWB) tma_prefetch_desc(&tmP);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int mtiles = p.num_groups > 0 ? s_toff[p.num_groups] : (p.M + BM2 - 1) / BM2;
  const int total_tiles = mtiles * p.n_tiles * (p.k_groups > 0 ? p.k_groups : 1);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = pair; t < total_tiles && ok; t += npairs) {
        const TileCoord c = decode_tile<BM2>(t, p, s_toff, s_goff);
        const int arow = c.row0 + 128 * (int)rank;
        const int ash = a_row_shift(p, c, s_goff, s_aoff);
        // B rows of the tile's first n-tile (a wide tile's second n-tile starts 256 rows later)
        const int nt0 = W2 ? 2 * c.nt : c.nt;
        const int brow = EPI == EPI_SWIGLU
                             ? c.group * p.b_rows_per_group + nt0 * 128 + (rank ? p.b_gate_offset : 0)
                             : c.group * p.b_rows_per_group + nt0 * C::BN + 128 * (int)rank;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait_cluster(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          const uint32_t full0 = map_to_cta(smem_u32(&full_bar[stage]), 0);
          const int kx = kt * (F8 ? 2 * BK : BK);
          // a group's last tile with <= 128 rows has none in CTA 1: CTA 1 skips its A rows
          // (its accumulator rows are never stored) and saves their L2 bytes
          const bool a1 = c.rows > 128;
          if (rank == 0)
            mbar_arrive_expect_tx(&full_bar[stage], GA ? 2 * C::B_BYTES
                                                    : (GB ? 2 * C::A_BYTES : 2 * C::STAGE_BYTES) - (a1 ? 0 : C::A_BYTES));
          if (!GA && (rank == 0 || a1)) {
            if (p.a_mn) {   // MN-major A: this CTA's 128 M columns as two 64-column blocks
              tma_load_2d_pair(sa, &tmA, full0, arow, kt * BK + ash);
              tma_load_2d_pair(sa + 8192, &tmA, full0, arow + 64, kt * BK + ash);
            } else {
              tma_load_2d_pair(sa, &tmA, full0, kx, arow + ash);
            }
          }
          if (GB) {
            // B arrives through the gather warps
          } else if (EPI != EPI_SWIGLU && p.b_mn) {   // MN-major B: this CTA's 128 columns, two 64-column blocks
            for (int b = 0; b < 2; ++b)
              tma_load_2d_pair(sa + C::A_BYTES + b * 8192, &tmB, full0, c.nt * C::BN + 128 * (int)rank + 64 * b,
                               c.group * p.b_rows_per_group + kt * BK);
          } else {
            tma_load_2d_pair(sa + C::A_BYTES, &tmB, full0, kx, brow);
            if (W2) tma_load_2d_pair(sa + C::A_BYTES + C::B_PART, &tmB, full0, kx, brow + C::BN);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0 && W2) {
      // ---------------- UMMA issuer, wide tiles (CTA 0) ----------------
      // Each k-tile feeds accumulator 0 (B part 0) and accumulator 1 (B part 1).  The epilogue
      // frees accumulator 0 first; until accumulator 1 is free as well, the MMAs into accumulator 0
      // run ahead by up to the ring's depth, so the tensor pipe keeps working while the epilogue
      // reads the previous tile's second half.
      constexpr uint32_t idesc = umma_idesc_bf16_f32(BM2, C::BN);
      uint32_t stage = 0, phase = 0;        // ring position of the next k-tile for accumulator 1
      uint32_t a_stage = 0, a_phase = 0;    // ring position of the next k-tile for accumulator 0
      int it = 0;
      auto mma_k_tile = [&](uint32_t st, int acc, bool acc_in) {
        const uint32_t sa = smem_u32(smem + st * C::STAGE_BYTES);
        const uint64_t a_desc = umma_sdesc_sw128(sa);
        const uint64_t b_desc = umma_sdesc_sw128(sa + C::A_BYTES + acc * C::B_PART);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::ACC_STRIDE);
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk)
          umma_bf16_pair(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (acc_in || kk > 0) ? 1u : 0u);
      };
      for (int t = pair; t < total_tiles; t += npairs, ++it) {
        const TileCoord c = decode_tile<BM2>(t, p, s_toff, s_goff);
        const uint32_t par = ((uint32_t)it & 1u) ^ 1u;   // each accumulator is used once per tile
        if (!mbar_wait_cluster(&tempty_bar[0], par, abort_flag, p.status)) break;
        tc_fence_after();
        bool ok = true, have1 = false;
        int ka = c.kt0;
        for (int kb = c.kt0; kb < c.kt1; ++kb) {
          // accumulator 0's MMAs for k-tile kb, and beyond it while accumulator 1 is busy
          while (ka <= kb ||
                 (!have1 && ka < c.kt1 && ka - kb < C::STAGES && !mbar_test(&tempty_bar[1], par))) {
            if (!mbar_wait_cluster(&full_bar[a_stage], a_phase, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            mma_k_tile(a_stage, 0, ka > c.kt0);
            ++ka;
            if (++a_stage == C::STAGES) { a_stage = 0; a_phase ^= 1u; }
          }
          if (!ok) break;
          if (!have1) {
            if (!mbar_wait_cluster(&tempty_bar[1], par, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            have1 = true;
          }
          mma_k_tile(stage, 1, kb > c.kt0);
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(&tfull_bar[0], 0x3);
        umma_commit_pair(&tfull_bar[1], 0x3);
      }
    } else if (lane == 0 && rank == 0) {
      // ---------------- UMMA issuer (CTA 0) ----------------
      constexpr uint32_t idesc = F8 ? umma_idesc_e4m3_f32(BM2, C::BN) : umma_idesc_bf16_f32(BM2, C::BN);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = pair; t < total_tiles; t += npairs, ++it) {
        const TileCoord c = decode_tile<BM2>(t, p, s_toff, s_goff);
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait_cluster(&tempty_bar[acc], (use & 1u) ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::ACC_STRIDE);
        bool ok = true;
        for (int kt = c.kt0; kt < c.kt1; ++kt) {
          if (!mbar_wait_cluster(&full_bar[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const bool amn = !GA && p.a_mn;
          const bool bmn = EPI != EPI_SWIGLU && p.b_mn;
          const uint64_t a_desc = amn ? umma_sdesc_mn_sw128(sa, 8192) : umma_sdesc_sw128(sa);
          const uint64_t b_desc = bmn ? umma_sdesc_mn_sw128(sa + C::A_BYTES, 8192) : umma_sdesc_sw128(sa + C::A_BYTES);
          const uint64_t a_step = amn ? 2048 / 16 : 2;
          const uint64_t b_step = bmn ? 2048 / 16 : 2;
          // bits 15 / 16 of the instruction descriptor: A / B is MN-major
          const uint32_t id = idesc | (amn ? (1u << 15) : 0u) | (bmn ? (1u << 16) : 0u);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            if (F8)
              umma_e4m3_pair(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, id, (kt > c.kt0 || kk > 0) ? 1u : 0u);
            else
              umma_bf16_pair(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, id, (kt > c.kt0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(&tfull_bar[acc], 0x3);
      }
    }
  } else if (warp < 2 + kEpiWarps) {
    // ---------------- epilogue: warps 2..9 of both CTAs ----------------
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quad * 32 + lane;
    uint4* stg = reinterpret_cast<uint4*>(smem + C::EPI_OFF) + (warp - 2) * 128;
    // SwiGLU backward: the first warp of each half issues its half's [u | g] boxes; every warp of
    // the half counts the chunks it has consumed, the issuer also those it has issued
    const bool pre_issuer = C::SWB && ((warp - 2) & 3) == 0 && lane == 0;
    uint32_t pre_issued = 0, pre_used = 0;
    int it = 0;
    for (int t = pair; t < total_tiles; t += npairs, ++it) {
      const TileCoord c = decode_tile<BM2>(t, p, s_toff, s_goff);
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      int ash = 0, live_end = 0;
      if constexpr (C::SWB) {
        ash = a_row_shift(p, c, s_goff, s_aoff);
        live_end = s_aoff[c.group + 1];
        // the tile's first two [u | g] chunks of this half, before the accumulator wait
        if (pre_issuer && c.rows > 128 * (int)rank)
          for (int j = 0; j < C::PRE_SLOTS; ++j)
            swb_pre_issue<C>(p, &tmP, smem, pre_full, pre_empty, half, pre_issued, c, (int)rank, ash, j, abort_flag);
      }
      if constexpr (W2) {
        // the tile's two n-tiles in turn, each accumulator released as soon as it has been read
        int ok = 1;
#pragma unroll 1
        for (int j = 0; j < 2 && ok; ++j) {
          if (lane == 0) ok = mbar_wait_cluster(&tfull_bar[j], (uint32_t)it & 1u, abort_flag, p.status) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(j * C::ACC_STRIDE);
          drain_wide_bf16(tb, c.row0 + 128 * (int)rank, c.rows - 128 * (int)rank, row_in_tile, 2 * c.nt + j, p, half,
                          stg, &tempty_bar[j]);
        }
        if (!ok) break;
        continue;
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait_cluster(&tfull_bar[acc], use & 1u, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * C::ACC_STRIDE);
      const float* cs = nullptr;
      const float* cs_gate = nullptr;
      if (F8) {
        const int brow = c.group * p.b_rows_per_group + c.nt * (EPI == EPI_SWIGLU ? C::BN / 2 : C::BN);
        cs = p.b_scale + brow;
        cs_gate = cs + p.b_gate_offset;
      }
      if constexpr (C::SWB) {
        swb_pair_tile<C>(tbase, c, (int)rank, row_in_tile, p, half, stg, smem, &tmP, pre_full, pre_empty, pre_issuer,
                         pre_issued, pre_used, ash, live_end, abort_flag);
      } else {
        // K-grouped: the group's output slice, zeros for a group without rows
        store_tile<C::BN, EPI, F8>(tbase, c.row0 + 128 * (int)rank, c.rows - 128 * (int)rank, row_in_tile, c.nt,
                                   c.split, p, half, stg, c.kt1 <= c.kt0, cs, cs_gate);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&tempty_bar[acc]), 0));
    }
  } else if constexpr (GA || GB) {
    // ---------------- gathered A rows (or B rows): warps 10..13 of both CTAs ----------------
    if (warp < kRelayWarp) {
      if constexpr (GA)
        gather_a_producer<BM2, C::STAGES, true>(p, s_toff, s_goff, pair, npairs, total_tiles, (int)rank, smem,
                                                C::STAGE_BYTES, empty_bar, gath_bar, abort_flag);
      else
        gather_b_mn_producer<C::STAGES>(p, s_toff, s_goff, pair, npairs, total_tiles, (int)rank, smem, C::STAGE_BYTES,
                                        C::A_BYTES, empty_bar, gath_bar, abort_flag);
    } else if (lane == 0) {
      gather_a_relay<BM2, C::STAGES, true>(p, s_toff, s_goff, pair, npairs, total_tiles, gath_bar, full_bar,
                                           abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // no CTA leaves while its partner may still touch its shared memory or TMEM
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) { }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*PFN_tmapEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                         const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                         CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                         CUtensorMapFloatOOBfill);

static PFN_tmapEncodeTiled get_encoder() {
  static PFN_tmapEncodeTiled fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_tmapEncodeTiled>(ptr);
  }
  return fn;
}

// (rows, cols) row-major matrix of bf16 (or e4m3 bytes), box of box_rows x 128 bytes, 128-byte swizzle.
static bool make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows, bool e4m3) {
  PFN_tmapEncodeTiled enc = get_encoder();
  if (!enc) return false;
  const int esize = e4m3 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor (rows x cols) read as box_cols x box_rows boxes with the given swizzle.
static bool make_tmap_box(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                          CUtensorMapSwizzle swizzle) {
  PFN_tmapEncodeTiled enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

int pick_bn_f32(int n_cols) {
  static const int cands[] = {256, 224, 128, 64, 32};
  int best = 256;
  long long best_cols = 1ll << 60;
  for (int bn : cands) {
    const long long padded = (long long)((n_cols + bn - 1) / bn) * bn;
    if (padded < best_cols) { best_cols = padded; best = bn; }
  }
  return best;
}

int pick_splits(int tiles, int K) {
  const int kt = (K + BK - 1) / BK;
  const int sms = num_sms();
  if (tiles * 2 > sms) return 1;
  int s = std::max(1, sms / std::max(1, tiles));
  s = std::min(s, std::max(1, kt / 4));  // at least 4 k-tiles per split
  const int per = (kt + s - 1) / s;
  return (kt + per - 1) / per;           // no empty split
}

template <int BN, int EPI, bool F8 = false, bool GA = false>
static cudaError_t launch_impl(const GemmProblem& q, const CUtensorMap& ta, const CUtensorMap& tb,
                               const GemmParams& gp, int grid, cudaStream_t stream) {
  using C = GemmCfg<BN>;
  auto kern = gemm_tc_kernel<BN, EPI, F8, GA>;
  static std::atomic<int> ready[kMaxDeviceSlots];
  const int dev = device_slot();
  if (dev < 0 || !ready[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0) ready[dev].store(1);
  }
  (void)q;
  launch_pdl(kern, grid, GA ? kThreadsGA : kThreads, C::SMEM_BYTES, stream, ta, tb, gp);
  return cudaGetLastError();
}

template <int EPI>
static cudaError_t launch_mx_impl(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& gp, int grid,
                                  cudaStream_t stream) {
  using C = GemmCfg<256>;
  auto kern = gemm_mx_kernel<EPI>;
  static std::atomic<int> ready[kMaxDeviceSlots];
  const int dev = device_slot();
  if (dev < 0 || !ready[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0) ready[dev].store(1);
  }
  launch_pdl(kern, grid, kThreadsMX, C::SMEM_BYTES, stream, ta, tb, gp);
  return cudaGetLastError();
}

template <int EPI, bool F8 = false, bool GA = false, bool GB = false, bool W2 = false>
static cudaError_t launch_pair_impl(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& gp, int tiles,
                                    cudaStream_t stream, const CUtensorMap* tp = nullptr) {
  using PairCfg = PairCfgT<EPI, W2>;
  auto kern = gemm_tc_pair_kernel<EPI, F8, GA, GB, W2>;
  constexpr int threads = GA || GB ? kThreadsGA : kThreads;
  static std::atomic<int> max_pairs_of[kMaxDeviceSlots];   // 0: not set up on that device yet
  const int dev = device_slot();
  int max_pairs = dev >= 0 ? max_pairs_of[dev].load() : 0;
  if (max_pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_sms());
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs = n > 0 ? n : 1;
    if (dev >= 0) max_pairs_of[dev].store(max_pairs);
  }
  int pairs = max_pairs;
  if (tiles > 0) pairs = std::min(pairs, tiles);
  launch_pdl(kern, 2 * pairs, threads, PairCfg::SMEM_BYTES, stream, ta, tb, tp ? *tp : ta, gp);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmProblem& q, cudaStream_t stream) {
  if (q.num_groups > kMaxGroups || q.k_groups > kMaxGroups) return cudaErrorInvalidValue;
  if (q.k_groups > 0 && (q.num_groups > 0 || q.splits > 1 || q.epilogue != EPI_F32)) return cudaErrorInvalidValue;
  if (q.mx) {
    // MXFP8 operands: 128 x 256 tiles on one CTA, both code operands TMA-loaded, K-major; the
    // block-scale rows 16-byte aligned (read as 16 scales: four 128-value k-tiles)
    if (q.bn != 256 || q.splits > 1 || q.k_groups > 0 || q.pair_tiles || q.e4m3 || q.a_gather || q.b_gather ||
        q.b_mn_major || q.a_mn_major || q.a_off || q.preact || q.K <= 0 || q.K % 128 || !q.a_mx_scale ||
        !q.b_mx_scale || q.a_mx_ld % 16 || q.b_mx_ld % 16 || q.a_mx_ld < q.K / 32 || q.b_mx_ld < q.K / 32 ||
        (reinterpret_cast<uintptr_t>(q.a_mx_scale) & 15) || (reinterpret_cast<uintptr_t>(q.b_mx_scale) & 15) ||
        (q.epilogue != EPI_SWIGLU && q.epilogue != EPI_BF16) || q.M < 0 ||
        (q.mx_out_codes && (q.epilogue != EPI_SWIGLU || !q.mx_out_scale || q.N % 32 || q.ldo % 16 ||
                            (reinterpret_cast<uintptr_t>(q.mx_out_codes) & 15) || q.mx_out_ld < q.N / 32)))
      return cudaErrorInvalidValue;
    if (q.M == 0) return cudaSuccess;
    CUtensorMap ta, tb;
    if (!make_tmap(&tb, q.B, q.b_rows_total, q.K, q.epilogue == EPI_SWIGLU ? 128 : 256, true) ||
        !make_tmap(&ta, q.A, q.M, q.K, BM, true))
      return cudaErrorInvalidValue;
    GemmParams gp{};
    gp.M = q.M;
    gp.N = q.N;
    gp.K = q.K;
    gp.num_groups = q.num_groups;
    gp.group_off = q.group_off;
    gp.tile_off = q.tile_off;
    gp.b_rows_per_group = q.b_rows_per_group;
    gp.b_gate_offset = q.b_gate_offset;
    gp.n_tiles = (q.N + (q.epilogue == EPI_SWIGLU ? 127 : 255)) / (q.epilogue == EPI_SWIGLU ? 128 : 256);
    gp.kt_total = q.K / 128;
    gp.splits = 1;
    gp.kt_per_split = gp.kt_total;
    gp.out = q.out;
    gp.ldo = q.ldo;
    gp.mx_a_scale = static_cast<const uint8_t*>(q.a_mx_scale);
    gp.mx_a_ld = q.a_mx_ld;
    gp.mx_a_rows = q.M;
    gp.mx_b_scale = static_cast<const uint8_t*>(q.b_mx_scale);
    gp.mx_b_ld = q.b_mx_ld;
    gp.mx_b_rows = q.b_rows_total;
    gp.mx_out_codes = static_cast<uint8_t*>(q.mx_out_codes);
    gp.mx_out_scale = static_cast<uint8_t*>(q.mx_out_scale);
    gp.mx_out_ld = q.mx_out_ld;
    gp.status = q.status;
    int grid = num_sms();
    if (q.num_groups == 0) grid = std::min(grid, ((q.M + BM - 1) / BM) * gp.n_tiles);
    return q.epilogue == EPI_SWIGLU ? launch_mx_impl<EPI_SWIGLU>(ta, tb, gp, grid, stream)
                                    : launch_mx_impl<EPI_BF16>(ta, tb, gp, grid, stream);
  }
  const bool pair = q.pair_tiles != 0;
  const bool f8 = q.e4m3 != 0;
  // router epilogue: dense 1-CTA tiles holding all N columns, no split-K
  if (q.epilogue == EPI_ROUTER &&
      (pair || f8 || q.splits > 1 || q.num_groups > 0 || q.k_groups > 0 || q.a_gather || q.b_mn_major ||
       q.a_mn_major || q.N > q.bn || q.router.k < 1 || q.router.k > kRouterFusedK || !q.router.idx || !q.router.w ||
       (q.bn != 32 && q.bn != 64 && q.bn != 128)))
    return cudaErrorInvalidValue;
  if (pair && (q.bn != 256 || q.splits > 1 || (q.epilogue == EPI_F32 && q.e4m3))) return cudaErrorInvalidValue;
  if (f8 && (q.bn != 256 || q.splits > 1 || q.k_groups > 0 || q.epilogue == EPI_F32 || !q.a_scale || !q.b_scale))
    return cudaErrorInvalidValue;
  // gathered A: grouped SwiGLU only; A rows are copied from a_src by the kernel, no A tensor map
  const bool ga = q.a_gather != nullptr;
  if (ga && (q.epilogue != EPI_SWIGLU || q.num_groups == 0 || q.splits > 1 || !q.a_src || q.a_src_rows < 0))
    return cudaErrorInvalidValue;
  // gathered B: K-grouped fp32 on CTA pairs, MN-major bf16 B
  const bool gb = q.b_gather != nullptr;
  if (gb && (q.k_groups == 0 || !pair || !q.b_mn_major || q.epilogue != EPI_F32 || f8 || ga || !q.b_src ||
             !q.b_goff || q.b_src_rows < 0 || q.N % 8))
    return cudaErrorInvalidValue;
  // MN-major B (bf16 / fp32 out, bf16 operands): group g's K rows x N columns; 64 x 64 boxes.
  // MN-major A: K-grouped only (1 CTA), K rows x M columns.
  if (q.b_mn_major && (f8 || ga || q.epilogue == EPI_SWIGLU || q.bn % 64 || q.K % BK ||
                       (q.num_groups > 0 && q.b_rows_per_group != q.K) || (q.k_groups > 0 && q.b_rows_per_group)))
    return cudaErrorInvalidValue;
  if (q.a_mn_major && (q.num_groups > 0 || f8 || q.K % BK || (q.a_cols && q.a_cols < q.M) ||
                       (q.mn_rows && q.mn_rows > q.K)))
    return cudaErrorInvalidValue;
  // A rows read from a_off[g] on: grouped (M or K) bf16 operands, TMA-loaded A
  if (q.a_off && (ga || f8 || (q.num_groups == 0 && q.k_groups == 0) || (q.k_groups > 0 && !q.a_mn_major) ||
                  q.a_rows < 0))
    return cudaErrorInvalidValue;
  if (q.a_rows && (q.a_mn_major || !q.a_off)) return cudaErrorInvalidValue;
  // pre-activations kept by the SwiGLU epilogue (or read by the SwiGLU backward's): whole 32-column
  // chunks of u and of g
  if (q.preact && ((q.epilogue != EPI_SWIGLU && q.epilogue != EPI_SWIGLU_BWD) || q.N % 32 ||
                   q.preact_ld < 2 * (int64_t)q.N || q.preact_ld % 8))
    return cudaErrorInvalidValue;
  // SwiGLU backward: M-grouped bf16 with A row offsets, [u | g] in, dUG (ldo >= 2N) and H out
  if (q.epilogue == EPI_SWIGLU_BWD &&
      (q.num_groups == 0 || !q.a_off || !q.preact || !q.out2 || f8 || ga || q.bn != 256 || q.splits > 1 ||
       q.ldo < 2 * (int64_t)q.N || q.ldo % 8 || q.ldo2 < q.N || q.ldo2 % 8))
    return cudaErrorInvalidValue;
  const int b_box = (q.epilogue == EPI_SWIGLU || pair) ? q.bn / 2 : q.bn;
  CUtensorMap ta, tb;
  if (gb) {
    // B is gathered by the kernel: no B tensor map (the A map fills the slot below)
  } else if (q.b_mn_major) {
    if (!make_tmap(&tb, q.B, q.b_rows_total, q.N, BK, false)) return cudaErrorInvalidValue;
  } else if (!make_tmap(&tb, q.B, q.b_rows_total, q.K, b_box, f8)) {
    return cudaErrorInvalidValue;
  }
  if (ga)
    ta = tb;   // unused
  else if (q.a_mn_major ? !make_tmap(&ta, q.A, q.mn_rows ? q.mn_rows : q.K, q.a_cols ? q.a_cols : q.M, BK, false)
                        : !make_tmap(&ta, q.A, q.a_rows ? q.a_rows : q.M, q.K, BM, f8))
    return cudaErrorInvalidValue;
  if (gb) tb = ta;   // unused

  GemmParams gp;
  gp.M = q.M;
  gp.N = q.N;
  gp.K = q.K;
  gp.num_groups = q.num_groups;
  gp.group_off = q.group_off;
  gp.tile_off = q.tile_off;
  gp.b_rows_per_group = q.b_rows_per_group;
  gp.b_gate_offset = q.b_gate_offset;
  const int out_cols_per_tile = q.epilogue == EPI_SWIGLU ? q.bn / 2 : q.bn;
  gp.n_tiles = (q.N + out_cols_per_tile - 1) / out_cols_per_tile;
  const int k_per_tile = f8 ? 2 * BK : BK;   // elements of K per 128-byte k-tile
  gp.kt_total = (q.K + k_per_tile - 1) / k_per_tile;
  gp.splits = std::max(1, q.splits);
  gp.kt_per_split = (gp.kt_total + gp.splits - 1) / gp.splits;
  gp.out = q.out;
  gp.ldo = q.ldo;
  gp.split_stride = q.split_stride;
  gp.k_groups = q.k_groups;
  gp.k_off = q.k_off;
  gp.a_scale = q.a_scale;
  gp.b_scale = q.b_scale;
  gp.a_gather = q.a_gather;
  gp.a_src = static_cast<const uint8_t*>(q.a_src);
  gp.a_ld_bytes = (long long)q.K * (f8 ? 1 : 2);
  gp.a_src_rows = q.a_src_rows;
  gp.b_mn = q.b_mn_major;
  gp.b_gather = q.b_gather;
  gp.b_src = static_cast<const uint8_t*>(q.b_src);
  gp.b_goff = q.b_goff;
  gp.b_ld_bytes = (long long)q.N * 2;
  gp.b_src_rows = q.b_src_rows;
  gp.a_mn = q.a_mn_major;
  gp.a_off = q.a_off;
  gp.preact = q.preact;
  gp.preact_ld = q.preact_ld;
  gp.preact_dense = q.preact_dense;
  gp.out2 = q.out2;
  gp.ldo2 = q.ldo2;
  gp.a_keep = ga ? q.a_keep : 0;
  gp.router = q.router;
  gp.status = q.status;

  // Wide pair tiles (two n-tiles per tile, each k-tile of A feeding both) for the bf16-out GEMMs
  // with TMA-loaded A over an even number of n-tiles, at least two tiles per CTA pair: the latent
  // projections and grouped GEMM 2.  A stage then brings 48 KB per 1024 MMA cycles instead of
  // 32 KB per 512, and shared memory, which also feeds the MMAs their operands, is no longer the
  // limit (latent prefill: latent down-projection 0.605 -> 0.528 ms, up 0.611 -> 0.571 ms; on
  // another box grouped GEMM 2 1.088 -> 1.045 ms).  Measured slower and not used: grouped GEMM 1
  // with its gathered rows (OlmoE shape 0.376 -> 0.394 ms, latent prefill 2.05 -> 2.10 ms) and
  // fp32 out, whose epilogue does not release the accumulator early (sigmoid-wide grouped GEMM 2
  // 1.83 -> 1.89 ms, the 896-expert router 0.309 -> 0.315 ms).
  const bool wide = pair && !ga && !f8 && !gb && q.k_groups == 0 && gp.splits == 1 && !q.b_mn_major &&
                    !q.a_mn_major && q.epilogue == EPI_BF16 && gp.n_tiles % 2 == 0 &&
                    (int64_t)((q.M + BM2 - 1) / BM2) * (gp.n_tiles / 2) >= num_sms();
  if (wide) gp.n_tiles /= 2;

  if (ga) {
    if (pair)
      return f8 ? launch_pair_impl<EPI_SWIGLU, true, true>(ta, tb, gp, 0, stream)
                : launch_pair_impl<EPI_SWIGLU, false, true>(ta, tb, gp, 0, stream);
    const int grid = num_sms();
    return f8 ? launch_impl<256, EPI_SWIGLU, true, true>(q, ta, tb, gp, grid, stream)
              : launch_impl<256, EPI_SWIGLU, false, true>(q, ta, tb, gp, grid, stream);
  }
  if (pair) {
    const int tiles = q.num_groups == 0 ? ((q.M + BM2 - 1) / BM2) * gp.n_tiles * std::max(1, q.k_groups) : 0;
    if (f8) {
      if (q.epilogue == EPI_SWIGLU) return launch_pair_impl<EPI_SWIGLU, true>(ta, tb, gp, tiles, stream);
      return launch_pair_impl<EPI_BF16, true>(ta, tb, gp, tiles, stream);
    }
    if (wide) return launch_pair_impl<EPI_BF16, false, false, false, true>(ta, tb, gp, tiles, stream);
    if (q.epilogue == EPI_SWIGLU) return launch_pair_impl<EPI_SWIGLU>(ta, tb, gp, tiles, stream);
    if (gb) return launch_pair_impl<EPI_F32, false, false, true>(ta, tb, gp, tiles, stream);   // K-grouped, B gathered
    if (q.epilogue == EPI_F32)   // fp32 out: dense, or grouped (the layer's fp32 expert rows)
      return launch_pair_impl<EPI_F32>(ta, tb, gp, tiles, stream);
    if (q.epilogue == EPI_SWIGLU_BWD) {
      // the [u | g] rows as 128 x 32 boxes, 64-byte swizzle (the epilogue reads a row per lane)
      CUtensorMap tp;
      const int64_t prow = q.preact_dense ? q.a_rows : q.M;
      if (!make_tmap_box(&tp, q.preact, prow, q.preact_ld, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
      return launch_pair_impl<EPI_SWIGLU_BWD>(ta, tb, gp, tiles, stream, &tp);
    }
    return launch_pair_impl<EPI_BF16>(ta, tb, gp, tiles, stream);
  }
  int grid = num_sms();
  if (q.num_groups == 0) {
    const int tiles = ((q.M + BM - 1) / BM) * gp.n_tiles * (q.k_groups > 0 ? q.k_groups : gp.splits);
    grid = std::min(grid, std::max(1, tiles));
  }

  if (f8) {
    if (q.epilogue == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, true>(q, ta, tb, gp, grid, stream);
    return launch_impl<256, EPI_BF16, true>(q, ta, tb, gp, grid, stream);
  }
  switch (q.epilogue) {
    case EPI_SWIGLU:
      if (q.bn == 256) return launch_impl<256, EPI_SWIGLU>(q, ta, tb, gp, grid, stream);
      break;
    case EPI_BF16:
      if (q.bn == 256) return launch_impl<256, EPI_BF16>(q, ta, tb, gp, grid, stream);
      break;
    case EPI_SWIGLU_BWD:
      return launch_impl<256, EPI_SWIGLU_BWD>(q, ta, tb, gp, grid, stream);
    case EPI_ROUTER:
      switch (q.bn) {
        case 128: return launch_impl<128, EPI_ROUTER>(q, ta, tb, gp, grid, stream);
        case 64: return launch_impl<64, EPI_ROUTER>(q, ta, tb, gp, grid, stream);
        case 32: return launch_impl<32, EPI_ROUTER>(q, ta, tb, gp, grid, stream);
      }
      break;
    case EPI_F32:
      switch (q.bn) {
        case 256: return launch_impl<256, EPI_F32>(q, ta, tb, gp, grid, stream);
        case 224: return launch_impl<224, EPI_F32>(q, ta, tb, gp, grid, stream);
        case 128: return launch_impl<128, EPI_F32>(q, ta, tb, gp, grid, stream);
        case 64: return launch_impl<64, EPI_F32>(q, ta, tb, gp, grid, stream);
        case 32: return launch_impl<32, EPI_F32>(q, ta, tb, gp, grid, stream);
      }
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
