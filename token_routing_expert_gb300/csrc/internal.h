// Launchers shared between the translation units of the library (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// EPI_SWIGLU_BWD: the product is dH of the SwiGLU experts (rounded to bf16); the epilogue reads the
// pre-activations [u | g] of the same rows and writes dUG = [dU | dG] to out and H to out2 (bf16).
enum GemmEpilogue { EPI_F32 = 0, EPI_BF16 = 1, EPI_SWIGLU = 2, EPI_SWIGLU_BWD = 3, EPI_ROUTER = 4 };

// Router GEMM tiles that hold every expert of their rows (one n-tile, no split-K) can run the
// gating, top-k, weights, normalisation and scalings in their epilogue (EPI_ROUTER), for top_k up
// to this many.
constexpr int kRouterFusedK = 8;
struct RouterEpilogue {
  const float* b_router;     // (E) or NULL: added to the logits
  const float* score_bias;   // (E) or NULL: added to the scores for selection only
  float* logits;             // (T, E) or NULL: the logits (with the router bias) are also stored
  int32_t* idx;              // (T, k)
  float* w;                  // (T, k)
  int gating, k, restore, orig_k;
  float sig_eps, p_norm, ews;
};

// C[M, N] = A[M, K] * B[N, K]^T per group, A and B bf16 K-major, fp32 accumulate.
// Groups (optional) are contiguous row ranges of A / C given by device
// offsets; group g multiplies with B rows [g * b_rows_per_group, ...).
struct GemmProblem {
  const void* A;          // (M, K) bf16
  const void* B;          // (b_rows_total, K) bf16
  int64_t b_rows_total;
  int M, N, K;            // N: valid output columns per group
  int num_groups;         // 0 = dense (one group of M rows)
  const int* group_off;   // device (G+1) row offsets, grouped only
  const int* tile_off;    // device (G+1) prefix sums of ceil(rows_g / 128), grouped only
  int b_rows_per_group;
  int b_gate_offset;      // swiglu: offset of the gate rows inside a group (= h)
  int epilogue;           // GemmEpilogue
  int bn;                 // UMMA N / B rows per tile (swiglu: up rows + gate rows)
  int splits;             // split-K: >1 writes fp32 partial slices
  int pair_tiles;         // 1: 256-row tiles on CTA pairs (tcgen05 cta_group::2); bn 256, no split-K,
                          //    and tile_off counts 256-row tiles
  void* out;
  int64_t ldo;            // elements
  int64_t split_stride;   // elements between split-K slices
  int k_groups;           // > 0: K-grouped GEMM (fp32 out only): group g multiplies A[:, K_g] by B[:, K_g]^T
                          //      and writes slice g (split_stride apart); K_g = k-tiles [k_off[g], k_off[g+1])
  const int* k_off;       // device (k_groups+1) offsets in 64-column k-tiles
  int e4m3;               // 1: A and B are e4m3 bytes (kind::f8f6f4) with per-row scales below
  const float* a_scale;   // (M) scale of each A row
  const float* b_scale;   // (b_rows_total) scale of each B row
  int b_mn_major;         // 1 (bf16 operands, bf16 / fp32 out): B is stored K rows x N columns (N contiguous),
                          //    group g's rows [g * K, (g + 1) * K); K a multiple of 64; no transposed copy needed
  int a_mn_major;         // 1 (1 CTA, K-grouped or dense): A is stored K rows x a_cols columns (M <= a_cols used)
  int64_t mn_rows;        // MN-major A: rows present (0: K); rows up to K beyond them read as zeros
  int64_t a_cols;         // MN-major A: columns per row (0: M)
  const int* a_gather;    // non-NULL (grouped SwiGLU only): A row r is row a_gather[r] of a_src, -1 a zero
                          // row; A is then unused.  e4m3: a_scale is per a_src row.
  const void* a_src;      // (a_src_rows, K) bf16 or e4m3
  int a_src_rows;
  const int* a_off;       // non-NULL (grouped bf16, TMA-loaded A): group g's A rows start at A row a_off[g]
                          //   (M-grouped: in place of group_off[g]; K-grouped MN-major A: in place of
                          //   64 k_off[g]); rows a tile reads past the group are A's next rows or, past
                          //   A's end, zeros, so the other operand must be zero there
  int64_t a_rows;         // with a_off, M-grouped: rows present in A (0: M)
  void* preact;           // SwiGLU: non-NULL also stores [u | g] bf16, preact_ld elements per output row;
                          // SwiGLU backward: the [u | g] rows read (preact_dense: at A's rows, i.e. the
                          // output row shifted by a_off as for A; else at the output's own rows)
  int64_t preact_ld;
  int preact_dense;
  void* out2;             // SwiGLU backward: H (bf16, ldo2 elements per row)
  int64_t ldo2;
  const int* b_gather;    // non-NULL (K-grouped, MN-major B, CTA pairs): B is gathered by the kernel: group g's
                          //   K row r is row b_gather[b_goff[g] + r] of b_src (b_src_rows x N bf16) while
                          //   r < b_goff[g+1] - b_goff[g], zeros past it; B is then unused
  const void* b_src;
  const int* b_goff;      // device (k_groups + 1) row offsets of the groups in b_gather
  int b_src_rows;
  int mx;                 // 1: A and B are e4m3 codes with E8M0 block scales (one per 32 K values of a row,
                          //    kind::mxf8f6f4.block_scale); K a multiple of 128; grouped or dense SwiGLU / bf16
                          //    out on 128 x 256 tiles, TMA-loaded A
  const void* a_mx_scale; // (M, a_mx_ld) bytes: row r's scale of K block b at [r * a_mx_ld + b]
  int64_t a_mx_ld;        // a multiple of 16, >= K / 32 (and both scale pointers 16-byte aligned)
  const void* b_mx_scale; // (b_rows_total, b_mx_ld) bytes
  int64_t b_mx_ld;
  void* mx_out_codes;     // MXFP8 SwiGLU only, non-NULL: H is written as MXFP8 (codes (M, ldo) bytes, ldo a
  void* mx_out_scale;     //   multiple of 16; scales (M, mx_out_ld) bytes) instead of bf16 to out
  int64_t mx_out_ld;
  int a_keep;             // gathered A: 1 reads the source rows with an evict_last L2 policy (for a_src that
                          //   fits the L2 beside the streamed weights, so its rows are not fetched again)
  RouterEpilogue router;  // EPI_ROUTER
  int* status;
};

int num_sms();
// Device address of the per-device status word on the current device (NULL without a device).
int* device_status();
cudaError_t launch_gemm(const GemmProblem& p, cudaStream_t stream);
// UMMA N chosen for a dense fp32 GEMM with n_cols output columns.
int pick_bn_f32(int n_cols);
// split-K factor that fills the GPU for a dense GEMM with `tiles` output tiles and K.
int pick_splits(int tiles, int K);

// Split-K router slices that top-k adds up itself; with more, logits must hold one more slice
// (partial_stride floats) for their sum.
constexpr int kTopkFusedSlices = 4;
cudaError_t launch_topk(const float* logits, int n_partials, int64_t partial_stride, const float* b_router,
                        const float* score_bias, int T, int E, int k, int gating, float sig_eps, float p_norm,
                        int restore, float ews, int orig_k, float* logits_out, int32_t* idx, float* w,
                        int* status, cudaStream_t stream);

// chunk: assignments per block, a multiple of 256 in [256, 4096]; blk_scratch holds
// permute_blocks(R, chunk) * E ints.
// tile_off (optional, E + 1 ints): also the grouped GEMMs' tile table, prefix sums of
// ceil(count / rows_per_tile), as launch_tile_table would write it.
// The permutation of R assignments over E experts runs as one cluster launch (else three kernels).
bool permute_fits_cluster(int R, int E);
cudaError_t launch_permute(const int32_t* idx, int R, int E, int32_t* counts, int32_t* offsets,
                           int32_t* gather_idx, int32_t* scatter_idx, int k, int chunk, int32_t* blk_scratch,
                           int* status, cudaStream_t stream, int rows_per_tile = 0, int32_t* tile_off = nullptr);
int permute_blocks(int R, int chunk);
int permute_chunk(int R);

cudaError_t launch_tile_table(const int32_t* offsets, int E, int rows_per_tile, int32_t* tile_off,
                              cudaStream_t stream);
cudaError_t launch_gather_rows(const void* src, const int32_t* gather_idx, int R, int T, int cols, void* dst,
                               int allow_padding, int* status, cudaStream_t stream);
// Capacity slots from a dense stable permutation (see moe_permute in moe.h).
cudaError_t launch_capacity_remap(const int32_t* idx, int R, int E, int cap, const int32_t* counts,
                                  const int32_t* off_dense, const int32_t* gather_dense,
                                  const int32_t* scatter_dense, int32_t* offsets, int32_t* gather_idx,
                                  int32_t* scatter_idx, cudaStream_t stream);

// y_f32: the expert rows y are fp32 (no RMSNorm then); else bf16.
cudaError_t launch_combine(const void* y, const int32_t* scatter_idx, const float* w, int T, int k, int L,
                           int R, int rms, float eps, const void* gain, void* z, int allow_dropped, int* status,
                           cudaStream_t stream, int y_f32 = 0);
cudaError_t launch_rmsnorm(const void* z, int T, int L, float eps, const void* gain, void* out,
                           cudaStream_t stream);
// Padded row layout of the experts backward (expert e from row 64 k_off[e], zero rows to the next
// multiple of 64): its offsets (+ the M-grouped tile table), rows copied into it (gather optional,
// max_rows >= 64 k_off[E]), and scatter indices moved into it.
cudaError_t launch_pad_offsets(const int32_t* off, int E, int rows_per_tile, int32_t* k_off, int32_t* poff,
                               int32_t* tile_off, cudaStream_t st);
cudaError_t launch_pad_rows(const void* src, const int32_t* gather, const int32_t* off, const int32_t* k_off, int E,
                            int src_rows, int cols, long long max_rows, void* dst, int* status, cudaStream_t st);
cudaError_t launch_pad_scatter(const int32_t* scatter, int R, const int32_t* off, const int32_t* poff, int E,
                               int32_t* out, cudaStream_t st);
// RMSNorm backward of the latent restore: dz (bf16) and r (fp32, per row); with dgamma, also the
// gain's gradient through gain_part ((T + slab - 1) / slab x L fp32 partial sums).
cudaError_t launch_rmsnorm_backward(const void* z, const void* dn, const void* gamma, int T, int L, float eps,
                                    void* dz, float* r, float* gain_part, int slab, float* dgamma, cudaStream_t st);
// out = a + b (bf16, n elements, a multiple of 8).
cudaError_t launch_add_bf16(const void* a, const void* b, long long n, void* out, cudaStream_t st);
// Runs a bounded mbarrier wait that nothing completes (limit_ns) and copies its result to the
// host, synchronising the stream: result_host[0] = 1 if it gave up with the abort flag raised,
// result_host[1] = milliseconds waited.  The wait records MOE_ERR_TIMEOUT in *status.
cudaError_t launch_wait_timeout_check(uint64_t limit_ns, int* status, int* result_host, cudaStream_t st);
// MXFP8 codes (rows x cols bytes) and E8M0 block scales (rows x scale_ld bytes, cols / 32 used).
cudaError_t launch_quantize_mx_e4m3(const void* x, long long rows, int cols, void* q, void* scales, int scale_ld,
                                    cudaStream_t st);
cudaError_t launch_combine_backward(const void* dz, const void* y, const int32_t* scatter_idx, const float* w, int T,
                                    int k, int L, int rows, void* dy, float* dw, int* status, cudaStream_t st);
cudaError_t launch_zero_padding_rows(const int32_t* gather_idx, int rows, int cols, void* dst, cudaStream_t st);
cudaError_t launch_router_backward(const float* logits, const int32_t* idx, const float* dw, int T, int E, int k,
                                   int gating, float sig_eps, float p_norm, float scale, float* dlogits,
                                   void* dl_bf16, int Epad, cudaStream_t st);
cudaError_t launch_column_sum(const float* d, int T, int E, float* out, cudaStream_t st);
// out = sum of `splits` fp32 slices of n floats (n a multiple of 4), in slice order.
cudaError_t launch_sum_slices_f32(const float* part, int splits, long long n, float* out, cudaStream_t st);
cudaError_t launch_quantize_rowwise_e4m3(const void* x, long long rows, int cols, void* q, float* scale,
                                         cudaStream_t st);
// dst[p] = src[gather_idx[p]] for MXFP8 rows: row_bytes codes (a multiple of 16) and scale_ld scale bytes
// (a multiple of 4) per row; a padding slot (-1, capacity mode) gets zero codes and scales 2^0.
cudaError_t launch_gather_rows_mx(const void* src, const void* src_scale, const int32_t* gather_idx, int R, int T,
                                  int row_bytes, int scale_ld, void* dst, void* dst_scale, int allow_padding,
                                  int* status, cudaStream_t st);
cudaError_t launch_gather_rows_e4m3(const void* src, const float* src_scale, const int32_t* gather_idx, int R, int T,
                                    int row_bytes, void* dst, float* dst_scale, int allow_padding, int* status,
                                    cudaStream_t st);
cudaError_t launch_splitk_reduce_bf16(const float* partials, int splits, int64_t slice, void* out,
                                      cudaStream_t stream);

}  // namespace moe
