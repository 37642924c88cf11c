// C ABI of the MoE layer forward: argument checks, workspace plan, and the
// order of kernel launches.  See include/moe.h for the contract.
#include <atomic>
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Per-device status word (first error recorded by any kernel).
__device__ int g_status;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int*> g_status_ptr[kMaxDevices];

// Device address of g_status on the current device, looked up once per device; concurrent first
// calls store the same address.
int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_status) != cudaSuccess) return nullptr;
    p = static_cast<int*>(q);
    g_status_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

// Bound on the SM count used to size split-K buffers (the GPU's own count is
// used at launch, and never needs more).
constexpr int kSizingSms = 256;

int splits_for(int tiles, int K, int sms) {
  const int kt = (K + 63) / 64;
  if (tiles * 2 > sms) return 1;
  int s = std::max(1, sms / std::max(1, tiles));
  s = std::min(s, std::max(1, kt / 4));
  const int per = (kt + s - 1) / s;
  return (kt + per - 1) / per;
}

struct Plan {
  int64_t T, R;
  bool capacity;      // capacity-limited experts
  int64_t cap;        // slots per expert (capacity mode)
  int64_t rows;       // rows of the permuted order: R, or E * cap
  size_t gdense, sdense, odense;   // capacity mode: the dense stable permutation before slotting
  size_t xq, xs, xpq, xps, hq, hs;  // e4m3 experts: codes and scales of x_routed, its rows, H
  bool mx;            // MXFP8 experts (block scales); else rowwise e4m3 when expert_fp8
  int64_t sx_ld, sh_ld;   // MXFP8: bytes of block scales per row of x_routed / of H
  int D, E, k, h, L, Lr;   // Lr: routed dim (L or D)
  int sms;            // the SM count the plan was made for
  bool latent;
  bool y32;           // the inference forward's expert rows y are fp32 (fp32_expert_rows)
  int router_bn, n_router_tiles;
  int router_splits, down_splits, up_splits;
  int64_t logit_slice;
  size_t logits, idx, wts, counts, offsets, tile_off, blk, gather, scatter, xr, xp, H, Y, zn, part, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// roundup8(capacity_factor * top_k * T / E), in double precision; 0 when dropless.
int64_t capacity_of(const moe_config_t* c, int64_t T) {
  if (!(c->capacity_factor > 0.f)) return 0;
  const double ideal = (double)c->top_k * (double)T / (double)c->num_experts;
  const double x = (double)c->capacity_factor * ideal;
  return 8 * (int64_t)std::ceil(x / 8.0);
}

// Bytes of MXFP8 block scales per row of `cols` values: cols / 32, rounded up to 16.
int64_t mx_scale_ld(int64_t cols) { return (cols / 32 + 15) / 16 * 16; }

// Upper bound of sum_j |w[t, j]| over a token's routing weights, from the gating and the
// scalings: softmax probabilities sum to at most 1, sigmoid scores to k (1 + eps); a p-norm
// normalisation leaves at most k^(1 - 1/p) (p >= 1); restore_weight_scale multiplies by k,
// expert_weight_scale by |s|, original_top_k by sqrt(k0 / k).
double weight_sum_bound(const moe_config_t* c) {
  const double k = c->top_k;
  double s = c->gating == MOE_GATING_SIGMOID ? k * (1.0 + std::fabs((double)c->sigmoid_stability_epsilon)) : 1.0;
  const double pn = c->normalize_expert_weights;
  if (pn > 0) s = pn >= 1.0 ? std::pow(k, 1.0 - 1.0 / pn) : 1.0;
  if (c->restore_weight_scale) s *= k;
  if (c->expert_weight_scale != 0.f) s *= std::fabs((double)c->expert_weight_scale);
  if (c->original_top_k > 0 && c->original_top_k != c->top_k) s *= std::sqrt((double)c->original_top_k / k);
  return s;
}

// The inference forward keeps the expert rows y in fp32 when the combine can magnify their
// rounding: a bf16 y carries a relative error up to 2^-9, the combine multiplies it by up to the
// weights' sum, and a layer whose weights can add up to more than one would then carry more error
// into its bf16 output than that output's own rounding (sigmoid-gated, L1-normalised weights
// restored x 8: 3.2e-2 from bf16 y alone at |out| ~ 15).  A latent layer normalises z before its
// output and keeps bf16 y, as do the e4m3 experts and the training forward (whose kept bf16 y the
// backward reads).
bool fp32_expert_rows(const moe_config_t* c) {
  return c->latent_dim == 0 && !c->expert_fp8 && weight_sum_bound(c) > 1.0 + 1e-6;
}

// Groups averaging >= 192 rows run on CTA pairs with 256-row tiles; smaller ones keep 128-row
// tiles, which waste less of each group's last partial tile.  Pairs read half the bytes per FLOP
// and gather their rows in grouped GEMM 1, which outweighs their padding down to ~200 rows per
// group (OlmoE shape at T = 2,048, 256 rows per expert: 0.279 -> 0.262 ms; latent prefill, 292:
// 5.08 -> 4.92 ms).  p.rows and p.E must be set.

// The quantised expert weights the config's expert_fp8 mode reads.
bool fp8_weights_present(const moe_config_t* c, const moe_weights_t* w) {
  if (!w->w_up_gate_fp8 || !w->w_out_fp8) return false;
  return c->expert_fp8 == MOE_EXPERT_MXFP8 ? (w->w_up_gate_mx_scale && w->w_out_mx_scale)
                                           : (w->w_up_gate_scale && w->w_out_scale);
}

int use_pair_tiles(const Plan& p) { return !p.mx && p.rows >= (int64_t)192 * p.E ? 1 : 0; }

// Routed input rows up to this size are kept in the L2 while grouped GEMM 1 gathers them: each row
// is read by top_k experts' tiles, far apart in time, while the weights stream through (OlmoE
// shape, 33.5 MB of rows: 812 -> 752 MB of DRAM traffic per GEMM 1, the time unchanged).
constexpr int64_t kKeepBytes = int64_t(48) << 20;


void make_plan(const moe_config_t* c, int64_t T, int sms, Plan* p) {
  p->T = T;
  p->sms = sms;
  p->D = c->d_model;
  p->E = c->num_experts;
  p->k = c->top_k;
  p->h = c->hidden_size;
  p->latent = c->latent_dim > 0;
  p->L = c->latent_dim;
  p->Lr = p->latent ? c->latent_dim : c->d_model;
  p->R = T * p->k;
  p->capacity = c->capacity_factor > 0.f;
  p->cap = capacity_of(c, T);
  p->rows = p->capacity ? (int64_t)p->E * p->cap : p->R;
  p->mx = c->expert_fp8 == MOE_EXPERT_MXFP8;
  p->y32 = fp32_expert_rows(c);
  p->sx_ld = mx_scale_ld(p->Lr);
  p->sh_ld = mx_scale_ld(p->h);
  const int mt = (int)((T + 127) / 128);
  p->router_bn = pick_bn_f32(p->E);
  p->n_router_tiles = (p->E + p->router_bn - 1) / p->router_bn;
  p->router_splits = splits_for(mt * p->n_router_tiles, p->D, sms);
  p->down_splits = p->latent ? splits_for(mt * ((p->L + 255) / 256), p->D, sms) : 1;
  p->up_splits = p->latent ? splits_for(mt * ((p->D + 255) / 256), p->L, sms) : 1;

  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  // split-K: router_splits partial slices (padded to 16 bytes); top-k adds up to kTopkFusedSlices
  // of them itself, a deeper split gets one more slice for their sum
  p->logit_slice = ((int64_t)T * p->E + 3) & ~int64_t(3);
  const int slices = p->router_splits > kTopkFusedSlices ? p->router_splits + 1 : std::max(1, p->router_splits);
  p->logits = take((size_t)slices * p->logit_slice * 4);
  p->idx = take((size_t)p->R * 4);
  p->wts = take((size_t)p->R * 4);
  p->counts = take((size_t)p->E * 4);
  p->offsets = take((size_t)(p->E + 1) * 4);
  p->tile_off = take((size_t)(p->E + 1) * 4);
  p->blk = take((size_t)std::max(1, permute_blocks((int)p->R, permute_chunk((int)p->R))) * p->E * 4);
  p->gather = take((size_t)std::max(p->R, p->rows) * 4);
  p->scatter = take((size_t)p->R * 4);
  if (p->capacity) {
    p->gdense = take((size_t)p->R * 4);
    p->sdense = take((size_t)p->R * 4);
    p->odense = take((size_t)(p->E + 1) * 4);
  } else {
    p->gdense = p->sdense = p->odense = (size_t)-1;
  }
  p->xr = p->latent ? take((size_t)T * p->L * 2) : (size_t)-1;
  // 128-row tiles read the routed rows from a permuted copy; CTA-pair tiles gather them
  const bool gathered = use_pair_tiles(*p);
  p->xp = !gathered && !c->expert_fp8 ? take((size_t)p->rows * p->Lr * 2) : (size_t)-1;
  p->H = take((size_t)p->rows * p->h * 2);
  p->Y = take((size_t)p->rows * p->Lr * (p->y32 ? 4 : 2));
  p->zn = p->latent ? take((size_t)T * p->L * 2) : (size_t)-1;
  if (p->mx) {
    p->xq = take((size_t)T * p->Lr);
    p->xs = take((size_t)T * p->sx_ld);
    p->xpq = take((size_t)p->rows * p->Lr);
    p->xps = take((size_t)p->rows * p->sx_ld);
    p->hq = take((size_t)p->rows * p->h);
    p->hs = take((size_t)p->rows * p->sh_ld);
  } else if (c->expert_fp8) {
    p->xq = take((size_t)T * p->Lr);
    p->xs = take((size_t)T * 4);
    p->xpq = gathered ? (size_t)-1 : take((size_t)p->rows * p->Lr);
    p->xps = gathered ? (size_t)-1 : take((size_t)p->rows * 4);
    p->hq = take((size_t)p->rows * p->h);
    p->hs = take((size_t)p->rows * 4);
  } else {
    p->xq = p->xs = p->xpq = p->xps = p->hq = p->hs = (size_t)-1;
  }
  size_t part = 0;
  if (p->down_splits > 1) part = std::max(part, (size_t)p->down_splits * T * p->L * 4);
  if (p->up_splits > 1) part = std::max(part, (size_t)p->up_splits * T * p->D * 4);
  p->part = take(part);
  p->total = o;
}

int check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->d_model < 1 || c->num_experts < 1 || c->top_k < 1 || c->hidden_size < 1 || c->latent_dim < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->num_experts) return MOE_ERR_INVALID_ARG;
  if (c->gating < MOE_GATING_SOFTMAX || c->gating > MOE_GATING_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->normalize_expert_weights < 0.f || c->sigmoid_stability_epsilon < 0.f || c->original_top_k < 0 ||
      !(c->rms_eps >= 0.f) || std::isnan(c->expert_weight_scale) || !(c->capacity_factor >= 0.f) ||
      std::isinf(c->capacity_factor))
    return MOE_ERR_INVALID_ARG;
  if (c->activation != 0) return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 64 || c->hidden_size % 64 || (c->latent_dim > 0 && c->latent_dim % 64)) return MOE_ERR_UNSUPPORTED;
  if (c->num_experts > 1024 || c->top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (c->expert_fp8 < 0 || c->expert_fp8 > MOE_EXPERT_MXFP8) return MOE_ERR_INVALID_ARG;
  // MXFP8 experts contract 128-value k-tiles (four 32-value scale blocks) over d_model / latent_dim and hidden_size
  if (c->expert_fp8 == MOE_EXPERT_MXFP8 &&
      ((c->latent_dim > 0 ? c->latent_dim : c->d_model) % 128 || c->hidden_size % 128))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_call(const moe_config_t* c, int64_t T, void* ws, size_t ws_bytes, Plan* plan) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * c->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  if (c->capacity_factor > 0.f && (double)c->num_experts * (double)capacity_of(c, T) > 2147483000.0)
    return MOE_ERR_UNSUPPORTED;
  make_plan(c, T, std::min(num_sms(), kSizingSms), plan);
  Plan sizing;
  make_plan(c, T, kSizingSms, &sizing);
  if (T > 0 && (!ws || ((uintptr_t)ws & 255) || ws_bytes < sizing.total)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// CTA-pair tiles (256 rows) pay off when the average group holds several of them.

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// C = A * B^T, dense, with split-K through fp32 partials when the output has few tiles.
// b_mn_rows > 0: B is stored K rows x N columns (MN-major) with only its first b_mn_rows rows
// present (the ones up to K read as zeros).
int dense_gemm_bf16(const void* A, const void* B, int M, int N, int K, void* out, int splits, float* part,
                    int* status, cudaStream_t st, int b_mn_rows = 0) {
  GemmProblem q{};
  q.A = A;
  q.B = B;
  q.b_rows_total = b_mn_rows > 0 ? b_mn_rows : N;
  q.b_mn_major = b_mn_rows > 0 ? 1 : 0;
  q.M = M;
  q.N = N;
  q.K = K;
  q.num_groups = 0;
  q.b_rows_per_group = 0;
  q.bn = 256;
  q.status = status;
  if (splits > 1) {
    q.epilogue = EPI_F32;
    q.splits = splits;
    q.out = part;
    q.ldo = N;
    q.split_stride = (int64_t)M * N;
    int s = cuda_status(launch_gemm(q, st));
    if (s != MOE_OK) return s;
    return cuda_status(launch_splitk_reduce_bf16(part, splits, (int64_t)M * N, out, st));
  }
  q.epilogue = EPI_BF16;
  q.splits = 1;
  q.out = out;
  q.ldo = N;
  q.split_stride = 0;
  q.pair_tiles = M >= 1024 ? 1 : 0;   // 256-row tiles on CTA pairs: half the B bytes per CTA
  return cuda_status(launch_gemm(q, st));
}

void mark(cudaEvent_t* ev, int i, cudaStream_t st) {
  if (ev && ev[i]) cudaEventRecord(ev[i], st);
}

// Up to 128 experts and top_k <= kRouterFusedK, when the row tiles alone fill the GPU (no split-K
// would be taken), the router GEMM's tiles hold every expert of their rows and its epilogue does
// the gating, top-k, weights and scalings: no logits round trip, one launch less.  With fewer row
// tiles the split-K GEMM and the top-k kernel are faster (OlmoE shape, T = 8,192: 64 row tiles,
// 28.6 us split and separate against 43.6 us fused, on different boxes).
bool router_fused(const Plan& p) {
  return p.E <= 128 && p.k <= kRouterFusedK && splits_for((int)((p.T + 127) / 128), p.D, p.sms) == 1;
}

int run_router(const moe_config_t* c, const moe_weights_t* w, const void* x, const Plan& p, float* logits_user,
               int32_t* idx, float* wts, void* ws, int* status, cudaStream_t st, cudaEvent_t* ev = nullptr) {
  if (router_fused(p)) {
    GemmProblem q{};
    q.A = x;
    q.B = w->w_router;
    q.b_rows_total = p.E;
    q.M = (int)p.T;
    q.N = p.E;
    q.K = p.D;
    q.epilogue = EPI_ROUTER;
    q.bn = p.E <= 32 ? 32 : p.E <= 64 ? 64 : 128;
    q.splits = 1;
    q.ldo = p.E;
    q.router.b_router = c->router_bias ? static_cast<const float*>(w->b_router) : nullptr;
    q.router.score_bias = c->has_score_bias ? static_cast<const float*>(w->score_bias) : nullptr;
    q.router.logits = logits_user;
    q.router.idx = idx;
    q.router.w = wts;
    q.router.gating = c->gating;
    q.router.k = p.k;
    q.router.restore = c->restore_weight_scale;
    q.router.orig_k = c->original_top_k;
    q.router.sig_eps = c->sigmoid_stability_epsilon;
    q.router.p_norm = c->normalize_expert_weights;
    q.router.ews = c->expert_weight_scale;
    q.status = status;
    const int s = cuda_status(launch_gemm(q, st));
    mark(ev, 2, st);
    return s;
  }
  float* gemm_out = (p.router_splits == 1 && logits_user) ? logits_user : at<float>(ws, p.logits);
  GemmProblem q{};
  q.A = x;
  q.B = w->w_router;
  q.b_rows_total = p.E;
  q.M = (int)p.T;
  q.N = p.E;
  q.K = p.D;
  q.num_groups = 0;
  q.epilogue = EPI_F32;
  q.bn = p.router_bn;
  q.splits = p.router_splits;
  if (p.router_splits == 1 && p.T >= 1024 && p.E > 128) {   // many experts: 256 x 256 tiles on CTA pairs
    q.bn = 256;
    q.pair_tiles = 1;
  }
  q.out = gemm_out;
  q.ldo = p.E;
  q.split_stride = p.logit_slice;
  q.status = status;
  int s = cuda_status(launch_gemm(q, st));
  if (s != MOE_OK) return s;
  mark(ev, 2, st);
  const bool rewrite = logits_user && (p.router_splits > 1 || (c->router_bias && w->b_router));
  float* logits_out = rewrite ? logits_user : nullptr;
  return cuda_status(launch_topk(gemm_out, p.router_splits, p.logit_slice, c->router_bias ? w->b_router : nullptr,
                                 c->has_score_bias ? w->score_bias : nullptr, (int)p.T, p.E, p.k, c->gating,
                                 c->sigmoid_stability_epsilon, c->normalize_expert_weights,
                                 c->restore_weight_scale, c->expert_weight_scale, c->original_top_k, logits_out, idx,
                                 wts, status, st));
}

// The experts on rowwise e4m3 operands: quantise x_routed per token, GEMM 1 on the code rows in
// permuted order (SwiGLU, scales in the epilogue) -> H bf16, quantise H per row, GEMM 2.
int run_experts_fp8(const moe_config_t* c, const moe_weights_t* w, const void* xr, const int32_t* gather,
                    const int32_t* offsets, const Plan& p, void* y, void* ws, int* status, cudaStream_t st,
                    cudaEvent_t* ev, bool tiles_ready, void* preact) {
  int32_t* tile_off = at<int32_t>(ws, p.tile_off);
  void* H = at<void>(ws, p.H);
  void* xq = at<void>(ws, p.xq);
  float* xs = at<float>(ws, p.xs);
  void* hq = at<void>(ws, p.hq);
  float* hs = at<float>(ws, p.hs);
  const int pair = use_pair_tiles(p);
  int s = tiles_ready ? MOE_OK : cuda_status(launch_tile_table(offsets, p.E, pair ? 256 : 128, tile_off, st));
  if (s == MOE_OK) s = cuda_status(launch_quantize_rowwise_e4m3(xr, p.T, p.Lr, xq, xs, st));
  if (s == MOE_OK && !pair)   // 128-row tiles: a permuted copy of the code rows and their scales
    s = cuda_status(launch_gather_rows_e4m3(xq, xs, gather, (int)p.rows, (int)p.T, p.Lr, at<void>(ws, p.xpq),
                                            at<float>(ws, p.xps), p.capacity ? 1 : 0, status, st));
  if (s != MOE_OK) return s;
  mark(ev, 5, st);
  GemmProblem g1{};
  if (pair) {               // the GEMM copies the code rows in permuted order itself
    g1.a_gather = gather;
    g1.a_src = xq;
    g1.a_src_rows = (int)p.T;
  } else {
    g1.A = at<void>(ws, p.xpq);
  }
  g1.B = w->w_up_gate_fp8;
  g1.b_rows_total = (int64_t)p.E * 2 * p.h;
  g1.M = (int)p.rows;
  g1.N = p.h;
  g1.K = p.Lr;
  g1.num_groups = p.E;
  g1.group_off = offsets;
  g1.tile_off = tile_off;
  g1.b_rows_per_group = 2 * p.h;
  g1.b_gate_offset = p.h;
  g1.epilogue = EPI_SWIGLU;
  g1.bn = 256;
  g1.splits = 1;
  g1.pair_tiles = pair;
  g1.e4m3 = 1;
  g1.a_scale = pair ? xs : at<float>(ws, p.xps);   // gathered: per token, looked up through a_gather
  g1.b_scale = w->w_up_gate_scale;
  g1.out = H;
  g1.ldo = p.h;
  g1.preact = preact;
  g1.preact_ld = 2 * (int64_t)p.h;
  g1.status = status;
  s = cuda_status(launch_gemm(g1, st));
  if (s != MOE_OK) return s;
  mark(ev, 6, st);   // the stage of GEMM 1 alone; quantising H counts with GEMM 2
  s = cuda_status(launch_quantize_rowwise_e4m3(H, p.rows, p.h, hq, hs, st));
  if (s != MOE_OK) return s;
  GemmProblem g2{};
  g2.A = hq;
  g2.B = w->w_out_fp8;
  g2.b_rows_total = (int64_t)p.E * p.Lr;
  g2.M = (int)p.rows;
  g2.N = p.Lr;
  g2.K = p.h;
  g2.num_groups = p.E;
  g2.group_off = offsets;
  g2.tile_off = tile_off;
  g2.b_rows_per_group = p.Lr;
  g2.epilogue = EPI_BF16;
  g2.bn = 256;
  g2.splits = 1;
  g2.pair_tiles = pair;
  g2.e4m3 = 1;
  g2.a_scale = hs;
  g2.b_scale = w->w_out_scale;
  g2.out = y;
  g2.ldo = p.Lr;
  g2.status = status;
  s = cuda_status(launch_gemm(g2, st));
  if (s != MOE_OK) return s;
  mark(ev, 7, st);
  return MOE_OK;
}

// The experts on MXFP8 operands: quantise x_routed in 32-value blocks, copy the code rows and
// their scales in permuted order, GEMM 1 (block-scaled MMAs; the SwiGLU epilogue rounds H to bf16
// and writes it as MXFP8 codes and scales), GEMM 2 -> Y bf16.
int run_experts_mx(const moe_config_t* c, const moe_weights_t* w, const void* xr, const int32_t* gather,
                   const int32_t* offsets, const Plan& p, void* y, void* ws, int* status, cudaStream_t st,
                   cudaEvent_t* ev, bool tiles_ready) {
  (void)c;
  int32_t* tile_off = at<int32_t>(ws, p.tile_off);
  void* xq = at<void>(ws, p.xq);
  void* xs = at<void>(ws, p.xs);
  void* hq = at<void>(ws, p.hq);
  void* hs = at<void>(ws, p.hs);
  int s = tiles_ready ? MOE_OK : cuda_status(launch_tile_table(offsets, p.E, 128, tile_off, st));
  if (s == MOE_OK) s = cuda_status(launch_quantize_mx_e4m3(xr, p.T, p.Lr, xq, xs, (int)p.sx_ld, st));
  if (s == MOE_OK)
    s = cuda_status(launch_gather_rows_mx(xq, xs, gather, (int)p.rows, (int)p.T, p.Lr, (int)p.sx_ld,
                                          at<void>(ws, p.xpq), at<void>(ws, p.xps), p.capacity ? 1 : 0, status, st));
  if (s != MOE_OK) return s;
  mark(ev, 5, st);
  GemmProblem g1{};
  g1.A = at<void>(ws, p.xpq);
  g1.B = w->w_up_gate_fp8;
  g1.b_rows_total = (int64_t)p.E * 2 * p.h;
  g1.M = (int)p.rows;
  g1.N = p.h;
  g1.K = p.Lr;
  g1.num_groups = p.E;
  g1.group_off = offsets;
  g1.tile_off = tile_off;
  g1.b_rows_per_group = 2 * p.h;
  g1.b_gate_offset = p.h;
  g1.epilogue = EPI_SWIGLU;
  g1.bn = 256;
  g1.splits = 1;
  g1.mx = 1;
  g1.a_mx_scale = at<void>(ws, p.xps);
  g1.a_mx_ld = p.sx_ld;
  g1.b_mx_scale = w->w_up_gate_mx_scale;
  g1.b_mx_ld = p.sx_ld;
  g1.mx_out_codes = hq;   // the SwiGLU epilogue quantises H itself: one 32-column chunk is one block
  g1.mx_out_scale = hs;
  g1.mx_out_ld = p.sh_ld;
  g1.ldo = p.h;
  g1.status = status;
  s = cuda_status(launch_gemm(g1, st));
  if (s != MOE_OK) return s;
  mark(ev, 6, st);
  GemmProblem g2{};
  g2.A = hq;
  g2.B = w->w_out_fp8;
  g2.b_rows_total = (int64_t)p.E * p.Lr;
  g2.M = (int)p.rows;
  g2.N = p.Lr;
  g2.K = p.h;
  g2.num_groups = p.E;
  g2.group_off = offsets;
  g2.tile_off = tile_off;
  g2.b_rows_per_group = p.Lr;
  g2.epilogue = EPI_BF16;
  g2.bn = 256;
  g2.splits = 1;
  g2.mx = 1;
  g2.a_mx_scale = hs;
  g2.a_mx_ld = p.sh_ld;
  g2.b_mx_scale = w->w_out_mx_scale;
  g2.b_mx_ld = p.sh_ld;
  g2.out = y;
  g2.ldo = p.Lr;
  g2.status = status;
  s = cuda_status(launch_gemm(g2, st));
  if (s != MOE_OK) return s;
  mark(ev, 7, st);
  return MOE_OK;
}

// tiles_ready: the tile table in the workspace was already written (by run_permute).
// preact (optional): grouped GEMM 1 also stores the pre-activations [u | g] there, rows x 2h bf16.
// y32: y is written in fp32 (bf16 experts only).
int run_experts(const moe_config_t* c, const moe_weights_t* w, const void* xr, const int32_t* gather,
                const int32_t* offsets, const Plan& p, void* y, void* ws, int* status, cudaStream_t st,
                cudaEvent_t* ev = nullptr, bool tiles_ready = false, void* preact = nullptr, bool y32 = false) {
  int32_t* tile_off = at<int32_t>(ws, p.tile_off);
  void* H = at<void>(ws, p.H);
  if (p.mx) {
    if (preact) return MOE_ERR_UNSUPPORTED;
    return run_experts_mx(c, w, xr, gather, offsets, p, y, ws, status, st, ev, tiles_ready);
  }
  if (c->expert_fp8) {
    if (y32) return MOE_ERR_UNSUPPORTED;
    return run_experts_fp8(c, w, xr, gather, offsets, p, y, ws, status, st, ev, tiles_ready, preact);
  }
  // large groups run on CTA pairs with 256-row tiles; small ones keep 128-row tiles,
  // which waste less of the last partial tile of each group
  const int pair = use_pair_tiles(p);
  int s = tiles_ready ? MOE_OK : cuda_status(launch_tile_table(offsets, p.E, pair ? 256 : 128, tile_off, st));
  if (s != MOE_OK) return s;
  // CTA-pair tiles: GEMM 1 copies the rows of x_routed in permuted order itself (cp.async into
  // its A stages).  128-row tiles read a permuted copy through TMA.  (A TMA tile::gather4 A-load
  // was measured 3x slower than a separate copy.)
  if (!pair) {
    s = cuda_status(launch_gather_rows(xr, gather, (int)p.rows, (int)p.T, p.Lr, at<void>(ws, p.xp), p.capacity ? 1 : 0,
                                       status, st));
    if (s != MOE_OK) return s;
  }
  mark(ev, 5, st);
  GemmProblem g1{};
  if (pair) {
    g1.a_gather = gather;
    g1.a_src = xr;
    g1.a_src_rows = (int)p.T;
  } else {
    g1.A = at<void>(ws, p.xp);
  }
  g1.B = w->w_up_gate;
  g1.b_rows_total = (int64_t)p.E * 2 * p.h;
  g1.M = (int)p.rows;
  g1.N = p.h;
  g1.K = p.Lr;
  g1.num_groups = p.E;
  g1.group_off = offsets;
  g1.tile_off = tile_off;
  g1.b_rows_per_group = 2 * p.h;
  g1.b_gate_offset = p.h;
  g1.epilogue = EPI_SWIGLU;
  g1.bn = 256;
  g1.splits = 1;
  g1.pair_tiles = pair;
  g1.out = H;
  g1.ldo = p.h;
  g1.preact = preact;
  g1.preact_ld = 2 * (int64_t)p.h;
  g1.a_keep = pair && (int64_t)p.T * p.Lr * 2 <= kKeepBytes ? 1 : 0;
  g1.status = status;
  s = cuda_status(launch_gemm(g1, st));
  if (s != MOE_OK) return s;
  mark(ev, 6, st);
  GemmProblem g2{};
  g2.A = H;
  g2.B = w->w_out;
  g2.b_rows_total = (int64_t)p.E * p.Lr;
  g2.M = (int)p.rows;
  g2.N = p.Lr;
  g2.K = p.h;
  g2.num_groups = p.E;
  g2.group_off = offsets;
  g2.tile_off = tile_off;
  g2.b_rows_per_group = p.Lr;
  g2.epilogue = y32 ? EPI_F32 : EPI_BF16;
  g2.bn = 256;
  g2.splits = 1;
  g2.pair_tiles = pair;
  g2.out = y;
  g2.ldo = p.Lr;
  g2.split_stride = 0;
  g2.status = status;
  s = cuda_status(launch_gemm(g2, st));
  if (s != MOE_OK) return s;
  mark(ev, 7, st);
  return MOE_OK;
}

// The permutation, dense or into capacity slots.
// tiles_done (optional): the dropless permutation also writes the grouped GEMMs' tile table into
// the workspace, and *tiles_done says so.
int run_permute(const int32_t* idx, const Plan& p, int32_t* counts, int32_t* offsets, int32_t* gather,
                int32_t* scatter, void* ws, int* status, cudaStream_t st, bool* tiles_done = nullptr) {
  if (tiles_done) *tiles_done = false;
  if (!p.capacity) {
    int32_t* tile_off = tiles_done ? at<int32_t>(ws, p.tile_off) : nullptr;
    const int s = cuda_status(launch_permute(idx, (int)p.R, p.E, counts, offsets, gather, scatter, p.k,
                                             permute_chunk((int)p.R), at<int32_t>(ws, p.blk), status, st,
                                             use_pair_tiles(p) ? 256 : 128, tile_off));
    if (s == MOE_OK && tiles_done) *tiles_done = true;
    return s;
  }
  int32_t* gd = at<int32_t>(ws, p.gdense);
  int32_t* sd = at<int32_t>(ws, p.sdense);
  int32_t* od = at<int32_t>(ws, p.odense);
  int s = cuda_status(launch_permute(idx, (int)p.R, p.E, counts, od, gd, sd, p.k, permute_chunk((int)p.R),
                                     at<int32_t>(ws, p.blk), status, st));
  if (s != MOE_OK) return s;
  return cuda_status(launch_capacity_remap(idx, (int)p.R, p.E, (int)p.cap, counts, od, gd, sd, offsets, gather, scatter,
                                           st));
}

int run_restore(const moe_config_t* c, const moe_weights_t* w, const void* z, bool z_is_normalised, const Plan& p,
                void* out, void* ws, int* status, cudaStream_t st) {
  const void* n = z;
  if (c->up_proj_norm && !z_is_normalised) {
    void* zn = at<void>(ws, p.zn);
    int s = cuda_status(launch_rmsnorm(z, (int)p.T, p.L, c->rms_eps, w->rms_weight, zn, st));
    if (s != MOE_OK) return s;
    n = zn;
  }
  return dense_gemm_bf16(n, w->w_up_latent, (int)p.T, p.D, p.L, out, p.up_splits, at<float>(ws, p.part), status, st);
}

// Workspace of the experts' backward.
struct BwdPlan {
  int64_t rows, kpad;
  size_t xp, ug, h, dug, dxp, k_off, poff, tile_off, scat, total;
};

void make_bwd_plan(const moe_config_t* c, int64_t T, BwdPlan* b) {
  const int64_t E = c->num_experts, h = c->hidden_size;
  const int64_t Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  b->rows = c->capacity_factor > 0.f ? E * capacity_of(c, T) : T * c->top_k;
  b->kpad = ((b->rows + 64 * E) + 63) / 64 * 64;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  // every activation in the padded row layout: kpad rows, expert e from row 64 k_off[e]
  b->xp = take((size_t)b->kpad * Lr * 2);
  b->ug = take((size_t)b->kpad * 2 * h * 2);
  b->h = take((size_t)b->kpad * h * 2);
  b->dug = take((size_t)b->kpad * 2 * h * 2);
  b->dxp = take((size_t)b->kpad * Lr * 2);
  b->k_off = take((size_t)(E + 1) * 4);
  b->poff = take((size_t)(E + 1) * 4);
  b->tile_off = take((size_t)(E + 1) * 4);
  b->scat = take((size_t)T * c->top_k * 4);
  b->total = o;
}

// Workspace of the latent projections' backward.
struct LatentBwdPlan {
  int64_t Tpad;
  int dn_splits, dx_splits, slab;
  size_t n, dn, r, gpart, part, total;
};

void make_latent_bwd_plan(const moe_config_t* c, int64_t T, int sms, LatentBwdPlan* b) {
  const int64_t D = c->d_model, L = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  b->Tpad = (T + 63) / 64 * 64;
  b->dn_splits = splits_for((int)(((T + 127) / 128) * ((L + 255) / 256)), (int)D, sms);
  b->dx_splits = splits_for((int)(((T + 127) / 128) * ((D + 255) / 256)), (int)L, sms);
  b->slab = 256;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  b->n = take((size_t)T * L * 2);
  b->dn = take((size_t)T * L * 2);
  b->r = take((size_t)T * 4);
  b->gpart = take((size_t)((T + b->slab - 1) / b->slab) * L * 4);
  const size_t dn_part = b->dn_splits > 1 ? (size_t)b->dn_splits * T * L * 4 : 0;
  const size_t dx_part = b->dx_splits > 1 ? (size_t)b->dx_splits * T * D * 4 : 0;
  b->part = take(std::max(dn_part, dx_part));
  b->total = o;
}

// A weight gradient (M x N fp32) = A^T B contracted over the T token rows of A (T x M) and B (T x N),
// both read as stored (MN-major operands); rows up to the padded T read as zeros.
int token_contraction_f32(const void* A, int M, const void* B, int N, int64_t T, int64_t Tpad, float* out,
                          int* status, cudaStream_t st) {
  GemmProblem g{};
  g.A = A;
  g.a_mn_major = 1;
  g.mn_rows = T;
  g.a_cols = M;
  g.B = B;
  g.b_mn_major = 1;
  g.b_rows_total = T;
  g.M = M;
  g.N = N;
  g.K = (int)Tpad;
  g.num_groups = 0;
  g.epilogue = EPI_F32;
  g.pair_tiles = M >= 256 && N % 256 == 0 ? 1 : 0;
  g.bn = g.pair_tiles || N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64);
  g.splits = 1;
  g.out = out;
  g.ldo = N;
  g.status = status;
  return cuda_status(launch_gemm(g, st));
}

// Workspace of the router backward.
struct RouterBwdPlan {
  int64_t Epad, Tpad;
  int dx_splits, dw_splits;
  size_t dl, part, total;
};

void make_router_bwd_plan(const moe_config_t* c, int64_t T, int sms, RouterBwdPlan* b) {
  const int64_t E = c->num_experts, D = c->d_model;
  b->Epad = (E + 63) / 64 * 64;
  b->Tpad = (T + 63) / 64 * 64;
  b->dx_splits = splits_for((int)(((T + 127) / 128) * ((D + 255) / 256)), (int)b->Epad, sms);
  b->dw_splits = splits_for((int)(((E + 127) / 128) * ((D + 255) / 256)), (int)b->Tpad, sms);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  b->dl = take((size_t)T * b->Epad * 2);
  const size_t dx_part = b->dx_splits > 1 ? (size_t)b->dx_splits * T * D * 4 : 0;
  const size_t dw_part = b->dw_splits > 1 ? (size_t)b->dw_splits * ((E * D + 3) / 4 * 4) * 4 : 0;
  b->part = take(std::max(dx_part, dw_part));
  b->total = o;
}

// M-grouped bf16 GEMM out = A B^T over the experts' row groups.
// b_mn: B is stored K rows x N columns per group (N contiguous) instead of N rows x K.
// a_off (optional): group e's A rows start at A row a_off[e] (A has a_rows rows) instead of offsets[e].
int grouped_bf16(const void* A, int64_t rows, const void* B, int64_t b_rows_total, int b_rows_per_group, int N, int K,
                 const int32_t* offsets, const int32_t* tile_off, int E, int pair, void* out, int* status,
                 cudaStream_t st, int b_mn = 0, const int32_t* a_off = nullptr, int64_t a_rows = 0) {
  GemmProblem g{};
  g.A = A;
  g.a_off = a_off;
  g.a_rows = a_off ? a_rows : 0;
  g.B = B;
  g.b_rows_total = b_rows_total;
  g.M = (int)rows;
  g.N = N;
  g.K = K;
  g.num_groups = E;
  g.group_off = offsets;
  g.tile_off = tile_off;
  g.b_rows_per_group = b_rows_per_group;
  g.epilogue = EPI_BF16;
  g.bn = 256;
  g.splits = 1;
  g.pair_tiles = pair;
  g.b_mn_major = b_mn;
  g.out = out;
  g.ldo = N;
  g.status = status;
  return cuda_status(launch_gemm(g, st));
}

// K-grouped fp32 GEMM: out[e] (M x N) = A[:, K_e] B[:, K_e]^T.
// K-grouped fp32 GEMM on the padded row layout: out[e] (M x N) = A[K_e rows]^T B[K_e rows], A stored
// kpad rows x M columns and B kpad rows x N columns (both MN-major operands), K_e = the 64-row
// tiles [k_off[e], k_off[e+1]).
// a_off (optional): group e's K rows of A start at A row a_off[e] (A has a_rows rows) instead of 64 k_off[e].
// b_gather (optional, CTA pairs): B's K rows of group e are rows b_gather[b_goff[e] + r] of B itself
// (b_rows rows), read by the kernel, instead of a padded copy.
int kgrouped_f32(const void* A, int M, const void* B, int N, int64_t kpad, const int32_t* k_off, int E, float* out,
                 int* status, cudaStream_t st, const int32_t* a_off = nullptr, int64_t a_rows = 0,
                 const int32_t* b_gather = nullptr, const int32_t* b_goff = nullptr, int64_t b_rows = 0) {
  GemmProblem g{};
  g.A = A;
  g.a_mn_major = 1;
  g.a_off = a_off;
  g.mn_rows = a_off ? a_rows : 0;
  g.B = B;
  g.b_mn_major = 1;
  g.b_rows_total = kpad;
  g.b_rows_per_group = 0;
  g.M = M;
  g.N = N;
  g.K = (int)kpad;
  g.num_groups = 0;
  g.epilogue = EPI_F32;
  g.pair_tiles = M >= 256 ? 1 : 0;   // 256 x 256 tiles on CTA pairs: half the B bytes per CTA
  g.bn = g.pair_tiles || N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64);
  g.splits = 1;
  g.k_groups = E;
  g.k_off = k_off;
  g.out = out;
  g.ldo = N;
  g.split_stride = (int64_t)M * N;
  g.status = status;
  if (b_gather && g.pair_tiles) {
    g.b_gather = b_gather;
    g.b_src = B;
    g.b_goff = b_goff;
    g.b_src_rows = (int)b_rows;
    g.B = nullptr;
  }
  return cuda_status(launch_gemm(g, st));
}

}  // namespace

int* device_status() { return status_ptr(); }

}  // namespace moe

using namespace moe;

extern "C" {

int moe_validate_config(const moe_config_t* cfg) { return check_config(cfg); }

int moe_num_params(const moe_config_t* c, int64_t* out) {
  if (!c || !out) return MOE_ERR_INVALID_ARG;
  if (c->d_model < 1 || c->num_experts < 1 || c->top_k < 1 || c->hidden_size < 1 || c->latent_dim < 0)
    return MOE_ERR_INVALID_ARG;
  const int64_t Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  const int64_t router = (int64_t)c->d_model * c->num_experts + (c->router_bias ? c->num_experts : 0);
  *out = router + 3 * Lr * c->hidden_size * c->num_experts;
  return MOE_OK;
}

int moe_num_active_params(const moe_config_t* c, int64_t* out) {
  int64_t total = 0;
  int s = moe_num_params(c, &total);
  if (s != MOE_OK) return s;
  const int64_t Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  *out = total - 3 * Lr * c->hidden_size * c->num_experts + 3 * Lr * c->hidden_size * c->top_k;
  return MOE_OK;
}

int moe_latent_proj_params(const moe_config_t* c, int with_norm_gain, int64_t* out) {
  if (!c || !out || c->d_model < 1 || c->latent_dim < 0) return MOE_ERR_INVALID_ARG;
  if (c->latent_dim == 0) {
    *out = 0;
    return MOE_OK;
  }
  *out = 2 * (int64_t)c->d_model * c->latent_dim + (with_norm_gain && c->up_proj_norm ? c->latent_dim : 0);
  return MOE_OK;
}

int moe_expert_capacity(const moe_config_t* c, int64_t T, int64_t* capacity) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !capacity) return MOE_ERR_INVALID_ARG;
  *capacity = capacity_of(c, T);
  return MOE_OK;
}

int moe_permuted_rows(const moe_config_t* c, int64_t T, int64_t* rows) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !rows) return MOE_ERR_INVALID_ARG;
  *rows = c->capacity_factor > 0.f ? (int64_t)c->num_experts * capacity_of(c, T) : T * c->top_k;
  return MOE_OK;
}

int moe_workspace_size(const moe_config_t* c, int64_t T, size_t* bytes) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
  Plan p;
  make_plan(c, T, kSizingSms, &p);
  *bytes = p.total;
  return MOE_OK;
}

int moe_workspace_layout(const moe_config_t* c, int64_t T, int64_t o[10]) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !o) return MOE_ERR_INVALID_ARG;
  Plan p;
  make_plan(c, T, std::min(num_sms(), kSizingSms), &p);
  o[0] = (int64_t)p.logits;
  o[1] = (int64_t)p.idx;
  o[2] = (int64_t)p.wts;
  o[3] = (int64_t)p.counts;
  o[4] = (int64_t)p.offsets;
  o[5] = (int64_t)p.gather;
  o[6] = (int64_t)p.scatter;
  o[7] = p.latent ? (int64_t)p.xr : -1;
  o[8] = (int64_t)p.Y;
  o[9] = p.latent ? (int64_t)p.zn : -1;
  return MOE_OK;
}

int moe_layer_expert_rows_fp32(const moe_config_t* c, int32_t* is_fp32) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (!is_fp32) return MOE_ERR_INVALID_ARG;
  *is_fp32 = fp32_expert_rows(c) ? 1 : 0;
  return MOE_OK;
}

int moe_router(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, float* logits, int32_t* idx,
               float* weights, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!w || !w->w_router || !x || !idx || !weights) return MOE_ERR_INVALID_ARG;
  if ((c->router_bias && !w->b_router) || (c->has_score_bias && !w->score_bias)) return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  return run_router(c, w, x, p, logits, idx, weights, ws, status, (cudaStream_t)stream);
}

int moe_permute(const moe_config_t* c, const int32_t* idx, int64_t T, int32_t* counts, int32_t* offsets,
                int32_t* gather_idx, int32_t* scatter_idx, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!idx || !gather_idx || !scatter_idx || !ws)) return MOE_ERR_INVALID_ARG;
  if (T == 0 && (!ws || ((uintptr_t)ws & 255))) return MOE_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  return run_permute(idx, p, counts, offsets, gather_idx, scatter_idx, ws, status, (cudaStream_t)stream);
}

int moe_grouped_swiglu(const moe_config_t* c, const moe_weights_t* w, const void* x_routed, const int32_t* gather_idx,
                       const int32_t* offsets, int64_t T, void* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_grouped_swiglu_preact(c, w, x_routed, gather_idx, offsets, T, y, nullptr, ws, ws_bytes, stream);
}

int moe_grouped_swiglu_preact(const moe_config_t* c, const moe_weights_t* w, const void* x_routed,
                              const int32_t* gather_idx, const int32_t* offsets, int64_t T, void* y, void* preact,
                              void* ws, size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!w || !w->w_up_gate || !w->w_out || !x_routed || !gather_idx || !offsets || !y) return MOE_ERR_INVALID_ARG;
  if (c->expert_fp8 && !fp8_weights_present(c, w))
    return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  if (preact && c->hidden_size % 32) return MOE_ERR_UNSUPPORTED;
  return run_experts(c, w, x_routed, gather_idx, offsets, p, y, ws, status, (cudaStream_t)stream, nullptr, false,
                     preact);
}

int moe_combine(const moe_config_t* c, const void* y, const int32_t* scatter_idx, const float* weights, int64_t T,
                void* z, moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !scatter_idx || !weights || !z) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * c->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  const int Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  const bool capacity = c->capacity_factor > 0.f;
  const int64_t rows = capacity ? (int64_t)c->num_experts * capacity_of(c, T) : T * c->top_k;
  if (rows > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_combine(y, scatter_idx, weights, (int)T, c->top_k, Lr, (int)rows, 0, 0.f, nullptr, z,
                                    capacity ? 1 : 0, status, (cudaStream_t)stream));
}

int moe_latent_down(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, void* x_routed, void* ws,
                    size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (!p.latent) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!w || !w->w_down_latent || !x || !x_routed) return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  return dense_gemm_bf16(x, w->w_down_latent, (int)T, p.L, p.D, x_routed, p.down_splits, at<float>(ws, p.part),
                         status, (cudaStream_t)stream);
}

int moe_latent_restore(const moe_config_t* c, const moe_weights_t* w, const void* z, int64_t T, void* out, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (!p.latent) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!w || !w->w_up_latent || !z || !out) return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  return run_restore(c, w, z, false, p, out, ws, status, (cudaStream_t)stream);
}

namespace {
int layer_forward(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, void* out, void* preact,
                  float* logits, void* ws, size_t ws_bytes, moe_stream_t stream, void* const* stage_events) {
  Plan p;
  int s = check_call(c, T, ws, ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!w || !x || !out || !w->w_router || !w->w_up_gate || !w->w_out) return MOE_ERR_INVALID_ARG;
  if (p.latent && (!w->w_down_latent || !w->w_up_latent)) return MOE_ERR_INVALID_ARG;
  if ((c->router_bias && !w->b_router) || (c->has_score_bias && !w->score_bias)) return MOE_ERR_INVALID_ARG;
  if (c->expert_fp8 && !fp8_weights_present(c, w))
    return MOE_ERR_INVALID_ARG;
  if (x == out) return MOE_ERR_INVALID_ARG;
  if (preact && c->hidden_size % 32) return MOE_ERR_UNSUPPORTED;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(stage_events));

  mark(ev, 0, st);
  const void* xr = x;
  if (p.latent) {
    void* xl = at<void>(ws, p.xr);
    s = dense_gemm_bf16(x, w->w_down_latent, (int)T, p.L, p.D, xl, p.down_splits, at<float>(ws, p.part), status, st);
    if (s != MOE_OK) return s;
    xr = xl;
  }
  mark(ev, 1, st);
  int32_t* idx = at<int32_t>(ws, p.idx);
  float* wts = at<float>(ws, p.wts);
  s = run_router(c, w, x, p, logits, idx, wts, ws, status, st, ev);
  if (s != MOE_OK) return s;
  mark(ev, 3, st);
  int32_t* counts = at<int32_t>(ws, p.counts);
  int32_t* offsets = at<int32_t>(ws, p.offsets);
  int32_t* gather = at<int32_t>(ws, p.gather);
  int32_t* scatter = at<int32_t>(ws, p.scatter);
  bool tiles_ready = false;
  s = run_permute(idx, p, counts, offsets, gather, scatter, ws, status, st, &tiles_ready);
  if (s != MOE_OK) return s;
  mark(ev, 4, st);
  void* Y = at<void>(ws, p.Y);
  const bool y32 = p.y32 && !preact;   // the training forward keeps bf16 y for the backward
  s = run_experts(c, w, xr, gather, offsets, p, Y, ws, status, st, ev, tiles_ready, preact, y32);
  if (s != MOE_OK) return s;
  if (!p.latent) {
    s = cuda_status(launch_combine(Y, scatter, wts, (int)T, p.k, p.Lr, (int)p.rows, 0, 0.f, nullptr, out,
                                   p.capacity ? 1 : 0, status, st, y32 ? 1 : 0));
    mark(ev, 8, st);
    mark(ev, 9, st);
    return s;
  }
  void* zn = at<void>(ws, p.zn);
  s = cuda_status(launch_combine(Y, scatter, wts, (int)T, p.k, p.L, (int)p.rows, c->up_proj_norm, c->rms_eps,
                                 w->rms_weight, zn, p.capacity ? 1 : 0, status, st));
  if (s != MOE_OK) return s;
  mark(ev, 8, st);
  s = run_restore(c, w, zn, true, p, out, ws, status, st);
  mark(ev, 9, st);
  return s;
}

}  // namespace

int moe_layer_forward_staged(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, void* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream, void* const* stage_events) {
  return layer_forward(c, w, x, T, out, nullptr, nullptr, ws, ws_bytes, stream, stage_events);
}

int moe_layer_forward(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, void* out, void* ws,
                      size_t ws_bytes, moe_stream_t stream) {
  return layer_forward(c, w, x, T, out, nullptr, nullptr, ws, ws_bytes, stream, nullptr);
}

int moe_layer_forward_preact(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, void* out,
                             void* preact, float* logits, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!preact && T > 0) return MOE_ERR_INVALID_ARG;
  return layer_forward(c, w, x, T, out, preact, logits, ws, ws_bytes, stream, nullptr);
}


// ---------------------------------------------------------------------------
// Host batches: copies in and out overlapped with the compute of neighbouring batches
// ---------------------------------------------------------------------------
namespace {
struct HostPipe {
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, h2d[2] = {nullptr, nullptr}, fwd[2] = {nullptr, nullptr},
              d2h[2] = {nullptr, nullptr};
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
  HostPipe& hp = g_pipe[dev];
  if (!hp.cin) {
    HostPipe n;
    bool ok = cudaStreamCreateWithFlags(&n.cin, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&n.cout, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&n.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&n.end, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
      ok = cudaEventCreateWithFlags(&n.h2d[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&n.fwd[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&n.d2h[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return MOE_ERR_CUDA;
    hp = n;
  }
  *out = &hp;
  return MOE_OK;
}
}  // namespace

int moe_host_workspace_size(const moe_config_t* c, int64_t T, size_t* bytes) {
  size_t lw = 0;
  int s = moe_workspace_size(c, T, &lw);
  if (s != MOE_OK) return s;
  const size_t xb = align256((size_t)T * c->d_model * 2);
  *bytes = align256(lw) + 4 * xb;
  return MOE_OK;
}

int moe_layer_forward_host_batches(const moe_config_t* c, const moe_weights_t* w, const void* const* x_host,
                                   void* const* out_host, int32_t n_batches, int64_t T, void* ws, size_t ws_bytes,
                                   moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (n_batches < 0 || T < 0) return MOE_ERR_INVALID_ARG;
  if (n_batches == 0 || T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  for (int b = 0; b < n_batches; ++b)
    if (!x_host[b] || !out_host[b]) return MOE_ERR_INVALID_ARG;
  size_t need = 0, lw = 0;
  if ((s = moe_host_workspace_size(c, T, &need)) != MOE_OK) return s;
  if ((s = moe_workspace_size(c, T, &lw)) != MOE_OK) return s;
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_WORKSPACE;
  HostPipe* hp = nullptr;
  if ((s = host_pipe(&hp)) != MOE_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t bytes = (size_t)T * c->d_model * 2;
  const size_t xb = align256(bytes);
  uint8_t* base = static_cast<uint8_t*>(ws) + align256(lw);
  void* xs[2] = {base, base + xb};
  void* os[2] = {base + 2 * xb, base + 3 * xb};
  auto ck = [](cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; };
  // the copy streams start after everything already enqueued on the caller's stream
  if ((s = ck(cudaEventRecord(hp->start, st))) != MOE_OK) return s;
  if ((s = ck(cudaStreamWaitEvent(hp->cin, hp->start, 0))) != MOE_OK) return s;
  if ((s = ck(cudaStreamWaitEvent(hp->cout, hp->start, 0))) != MOE_OK) return s;
  for (int b = 0; b < n_batches && s == MOE_OK; ++b) {
    const int k = b & 1;
    // input slot k is free once batch b-2's forward has read it
    if (b >= 2 && (s = ck(cudaStreamWaitEvent(hp->cin, hp->fwd[k], 0))) != MOE_OK) break;
    if ((s = ck(cudaMemcpyAsync(xs[k], x_host[b], bytes, cudaMemcpyHostToDevice, hp->cin))) != MOE_OK) break;
    if ((s = ck(cudaEventRecord(hp->h2d[k], hp->cin))) != MOE_OK) break;
    if ((s = ck(cudaStreamWaitEvent(st, hp->h2d[k], 0))) != MOE_OK) break;
    // output slot k is free once batch b-2's result has been copied out
    if (b >= 2 && (s = ck(cudaStreamWaitEvent(st, hp->d2h[k], 0))) != MOE_OK) break;
    if ((s = moe_layer_forward(c, w, xs[k], T, os[k], ws, lw, stream)) != MOE_OK) break;
    if ((s = ck(cudaEventRecord(hp->fwd[k], st))) != MOE_OK) break;
    if ((s = ck(cudaStreamWaitEvent(hp->cout, hp->fwd[k], 0))) != MOE_OK) break;
    if ((s = ck(cudaMemcpyAsync(out_host[b], os[k], bytes, cudaMemcpyDeviceToHost, hp->cout))) != MOE_OK) break;
    if ((s = ck(cudaEventRecord(hp->d2h[k], hp->cout))) != MOE_OK) break;
  }
  // join: the caller's stream completes after the last copy out (also on an error, so that
  // nothing enqueued here outlives the stream)
  int j = ck(cudaEventRecord(hp->end, hp->cout));
  if (j == MOE_OK) j = ck(cudaStreamWaitEvent(st, hp->end, 0));
  return s != MOE_OK ? s : j;
}

int moe_layer_forward_launches(const moe_config_t* c, int64_t T, int32_t* n) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !n) return MOE_ERR_INVALID_ARG;
  if (T == 0) {
    *n = 0;
    return MOE_OK;
  }
  Plan p;
  make_plan(c, T, std::min(num_sms(), kSizingSms), &p);
  int k = 0;
  if (p.latent) k += p.down_splits > 1 ? 2 : 1;  // latent down (+ split-K reduce)
  // router GEMM (with the top-k in its epilogue up to 128 experts), or GEMM, (sum of a deep split-K,) top-k
  k += router_fused(p) ? 1 : p.router_splits > kTopkFusedSlices ? 3 : 2;
  // permute: one cluster launch or count, scan, place (, capacity slots)
  k += (permute_fits_cluster((int)p.R, p.E) ? 1 : 3) + (p.capacity ? 1 : 0);
  k += p.capacity ? 1 : 0;                       // tile table (the dropless scan writes it itself)
  k += use_pair_tiles(p) ? 0 : 1;                // row gather for 128-row tiles (on CTA pairs grouped
                                                 // GEMM 1 gathers its rows)
  k += 2;                                        // grouped GEMM 1 (SwiGLU), grouped GEMM 2
  if (c->expert_fp8) k += p.mx ? 1 : 2;          // e4m3 quantisation of x_routed and of H (MXFP8: H is
                                                 // quantised by GEMM 1's epilogue)
  k += 1;                                        // combine (+ RMSNorm when latent)
  if (p.latent) k += p.up_splits > 1 ? 2 : 1;    // latent up (+ split-K reduce)
  *n = k;
  return MOE_OK;
}

int moe_backward_workspace_size(const moe_config_t* c, int64_t T, size_t* bytes) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
  BwdPlan b;
  make_bwd_plan(c, T, &b);
  RouterBwdPlan r;
  make_router_bwd_plan(c, T, kSizingSms, &r);
  *bytes = std::max(b.total, r.total);
  if (c->latent_dim > 0) {
    LatentBwdPlan l;
    make_latent_bwd_plan(c, T, kSizingSms, &l);
    *bytes = std::max(*bytes, l.total);
  }
  return MOE_OK;
}

int moe_latent_restore_backward(const moe_config_t* c, const moe_weights_t* w, const void* z, int64_t T,
                                const void* dout, void* dz, float* dw_up, float* drms_weight, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (c->latent_dim <= 0 || T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (T > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  if (!w || !w->w_up_latent || !z || !dout || !dz || !dw_up) return MOE_ERR_INVALID_ARG;
  LatentBwdPlan sizing, l;
  make_latent_bwd_plan(c, T, kSizingSms, &sizing);
  make_latent_bwd_plan(c, T, std::min(num_sms(), kSizingSms), &l);
  if (!ws || ((uintptr_t)ws & 255) || ws_bytes < sizing.total) return MOE_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int D = c->d_model, L = c->latent_dim;
  float* part = at<float>(ws, l.part);
  // n: the norm's output as the forward computed it (bf16), or z itself without the norm
  const void* n = z;
  if (c->up_proj_norm) {
    n = at<void>(ws, l.n);
    s = cuda_status(launch_rmsnorm(z, (int)T, L, c->rms_eps, w->rms_weight, const_cast<void*>(n), st));
    if (s != MOE_OK) return s;
  }
  // dn = dout W_up (W_up read as stored: D rows x L columns, an MN-major B)
  void* dn = c->up_proj_norm ? at<void>(ws, l.dn) : dz;
  s = dense_gemm_bf16(dout, w->w_up_latent, (int)T, L, D, dn, l.dn_splits, part, status, st, D);
  // dW_up = dout^T n, contracted over the tokens
  if (s == MOE_OK) s = token_contraction_f32(dout, D, n, L, T, l.Tpad, dw_up, status, st);
  if (s == MOE_OK && c->up_proj_norm)
    s = cuda_status(launch_rmsnorm_backward(z, dn, w->rms_weight, (int)T, L, c->rms_eps, dz, at<float>(ws, l.r),
                                            at<float>(ws, l.gpart), l.slab, drms_weight, st));
  return s;
}

int moe_latent_down_backward(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T,
                             const void* dx_routed, void* dx, float* dw_down, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (c->latent_dim <= 0 || T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (T > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  if (!w || !w->w_down_latent || !x || !dx_routed || !dx || !dw_down) return MOE_ERR_INVALID_ARG;
  LatentBwdPlan sizing, l;
  make_latent_bwd_plan(c, T, kSizingSms, &sizing);
  make_latent_bwd_plan(c, T, std::min(num_sms(), kSizingSms), &l);
  if (!ws || ((uintptr_t)ws & 255) || ws_bytes < sizing.total) return MOE_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int D = c->d_model, L = c->latent_dim;
  // dx = dx_routed W_down (W_down read as stored: L rows x D columns, an MN-major B)
  s = dense_gemm_bf16(dx_routed, w->w_down_latent, (int)T, D, L, dx, l.dx_splits, at<float>(ws, l.part), status, st,
                      L);
  // dW_down = dx_routed^T x, contracted over the tokens
  if (s == MOE_OK) s = token_contraction_f32(dx_routed, L, x, D, T, l.Tpad, dw_down, status, st);
  return s;
}

int moe_router_backward(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, const float* logits,
                        const int32_t* idx, const float* dweights, float* dlogits, void* dx, float* dw_router,
                        float* db_router, void* ws, size_t ws_bytes, moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if ((int64_t)T * c->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  if (!w || !w->w_router || !x || !logits || !idx || !dweights || !dlogits || !dx || !dw_router)
    return MOE_ERR_INVALID_ARG;
  RouterBwdPlan sizing, r;
  make_router_bwd_plan(c, T, kSizingSms, &sizing);
  make_router_bwd_plan(c, T, std::min(num_sms(), kSizingSms), &r);
  if (!ws || ((uintptr_t)ws & 255) || ws_bytes < sizing.total) return MOE_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int E = c->num_experts, D = c->d_model;
  float scale = 1.f;
  if (c->restore_weight_scale) scale *= (float)c->top_k;
  if (c->expert_weight_scale != 0.f) scale *= c->expert_weight_scale;
  if (c->original_top_k > 0 && c->original_top_k != c->top_k) scale *= sqrtf((float)c->original_top_k / (float)c->top_k);
  void* dl = at<void>(ws, r.dl);
  float* part = at<float>(ws, r.part);
  s = cuda_status(launch_router_backward(logits, idx, dweights, (int)T, E, c->top_k, c->gating,
                                         c->sigmoid_stability_epsilon, c->normalize_expert_weights, scale, dlogits, dl,
                                         (int)r.Epad, st));
  // dx = dlogits W_router: W_router read as stored (E rows x D columns, an MN-major B; the rows up
  // to the padded E read as zeros, as do dl's padding columns)
  if (s == MOE_OK) s = dense_gemm_bf16(dl, w->w_router, (int)T, D, (int)r.Epad, dx, r.dx_splits, part, status, st, E);
  // dW_router = dlogits^T x, contracted over the tokens: dl (T x Epad) and x (T x D) read as stored
  // (MN-major A and B), the tokens up to the padded T read as zeros
  if (s == MOE_OK) {
    GemmProblem g{};
    g.A = dl;
    g.a_mn_major = 1;
    g.mn_rows = T;
    g.a_cols = r.Epad;
    g.B = x;
    g.b_mn_major = 1;
    g.b_rows_total = T;
    g.M = E;
    g.N = D;
    g.K = (int)r.Tpad;
    g.num_groups = 0;
    g.epilogue = EPI_F32;
    g.bn = D % 256 == 0 ? 256 : (D % 128 == 0 ? 128 : 64);
    g.splits = r.dw_splits;
    g.ldo = D;
    g.status = status;
    if (r.dw_splits > 1) {
      const int64_t slice = ((int64_t)E * D + 3) / 4 * 4;
      g.out = part;
      g.split_stride = slice;
      s = cuda_status(launch_gemm(g, st));
      if (s == MOE_OK) s = cuda_status(launch_sum_slices_f32(part, r.dw_splits, slice, dw_router, st));
    } else {
      g.out = dw_router;
      s = cuda_status(launch_gemm(g, st));
    }
  }
  if (s == MOE_OK && c->router_bias && db_router) s = cuda_status(launch_column_sum(dlogits, (int)T, E, db_router, st));
  return s;
}

int moe_combine_backward(const moe_config_t* c, const void* dz, const void* y, const int32_t* scatter_idx,
                         const int32_t* gather_idx, const float* weights, int64_t T, void* dy, float* dweights,
                         moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!dz || !y || !scatter_idx || !weights || !dy || !dweights) return MOE_ERR_INVALID_ARG;
  const bool capacity = c->capacity_factor > 0.f;
  if (capacity && !gather_idx) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * c->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  const int64_t rows = capacity ? (int64_t)c->num_experts * capacity_of(c, T) : T * c->top_k;
  if (rows > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  if (capacity) {
    s = cuda_status(launch_zero_padding_rows(gather_idx, (int)rows, Lr, dy, st));
    if (s != MOE_OK) return s;
  }
  return cuda_status(
      launch_combine_backward(dz, y, scatter_idx, weights, (int)T, c->top_k, Lr, (int)rows, dy, dweights, status, st));
}

int moe_grouped_swiglu_backward(const moe_config_t* c, const moe_weights_t* w, const void* x_routed,
                                const int32_t* gather_idx, const int32_t* offsets, const int32_t* scatter_idx,
                                int64_t T, const void* dy, void* dx_routed, float* dw_up_gate, float* dw_out,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_grouped_swiglu_backward_preact(c, w, x_routed, gather_idx, offsets, scatter_idx, T, dy, nullptr,
                                            dx_routed, dw_up_gate, dw_out, ws, ws_bytes, stream);
}

int moe_grouped_swiglu_backward_preact(const moe_config_t* c, const moe_weights_t* w, const void* x_routed,
                                       const int32_t* gather_idx, const int32_t* offsets, const int32_t* scatter_idx,
                                       int64_t T, const void* dy, const void* preact, void* dx_routed,
                                       float* dw_up_gate, float* dw_out, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * c->top_k > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  BwdPlan b;
  make_bwd_plan(c, T, &b);
  if (b.rows > (int64_t)0x7fffffff - 128 || b.kpad > (int64_t)0x7fffffff - 128) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!ws || ((uintptr_t)ws & 255) || ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  if (!w || !w->w_up_gate || !w->w_out || !x_routed || !gather_idx || !offsets || !scatter_idx || !dy ||
      !dx_routed || !dw_up_gate || !dw_out)
    return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  const int E = c->num_experts, h = c->hidden_size, k = c->top_k;
  const int Lr = c->latent_dim > 0 ? c->latent_dim : c->d_model;
  const bool capacity = c->capacity_factor > 0.f;
  const int rows = (int)b.rows;
  const int pair = rows >= 384 * E ? 1 : 0;
  int32_t* tile_off = at<int32_t>(ws, b.tile_off);
  int32_t* k_off = at<int32_t>(ws, b.k_off);
  int32_t* poff = at<int32_t>(ws, b.poff);
  int32_t* scat = at<int32_t>(ws, b.scat);
  void* xp = at<void>(ws, b.xp);
  void* UG = at<void>(ws, b.ug);
  void* H = at<void>(ws, b.h);
  void* dUG = at<void>(ws, b.dug);
  void* dXp = at<void>(ws, b.dxp);
  const int prows = (int)b.kpad;   // rows of the padded layout (the ones past 64 k_off[E] are never read)

  // padded layout: offsets, the scatter moved into it, and the routed rows copied into it where a GEMM
  // cannot gather them itself (the recomputation of the pre-activations; 1-CTA weight-gradient tiles)
  // dW_up_gate on CTA pairs can read x_routed through the gather indices itself.  That pays off when
  // the padded copy it saves is dear: many small experts, whose padding adds many rows (latent
  // prefill shape, 292 rows per expert: experts backward 10.26 -> 9.49 ms); with ~1,000 rows per
  // expert the copy is cheaper than gathering in the GEMM (OlmoE shape: 1.40 ms copying vs 1.47)
  const bool gather_b = preact != nullptr && 2 * h >= 256 && (int64_t)rows < 512 * (int64_t)E;
  s = cuda_status(launch_pad_offsets(offsets, E, pair ? 256 : 128, k_off, poff, tile_off, st));
  if (s == MOE_OK && !gather_b)
    s = cuda_status(launch_pad_rows(x_routed, gather_idx, offsets, k_off, E, (int)T, Lr, prows, xp, status, st));
  if (s == MOE_OK) s = cuda_status(launch_pad_scatter(scatter_idx, (int)T * k, offsets, poff, E, scat, st));
  // pre-activations [u | g]: the forward's (dense rows), or recomputed in the padded layout
  if (s == MOE_OK && !preact)
    s = grouped_bf16(xp, prows, w->w_up_gate, (int64_t)E * 2 * h, 2 * h, 2 * h, Lr, poff, tile_off, E, pair, UG,
                     status, st);
  // dH = dY W_out with the SwiGLU backward in its epilogue: dY read at its dense rows (each group's
  // A rows from offsets[e]; what a tile reads past the group only reaches padding rows, which get
  // zeros), [u | g] read beside each dH chunk, dUG = [dU | dG] and H written in the padded layout.
  // Then dXp = dUG W_up_gate and dx = the sum over a token's rows.  The weights are read as stored
  // (K rows x N columns: MN-major B operands).
  if (s == MOE_OK) {
    GemmProblem g{};
    g.A = dy;
    g.a_off = offsets;
    g.a_rows = rows;
    g.B = w->w_out;
    g.b_mn_major = 1;
    g.b_rows_total = (int64_t)E * Lr;
    g.b_rows_per_group = Lr;
    g.M = prows;
    g.N = h;
    g.K = Lr;
    g.num_groups = E;
    g.group_off = poff;
    g.tile_off = tile_off;
    g.epilogue = EPI_SWIGLU_BWD;
    g.bn = 256;
    g.splits = 1;
    g.pair_tiles = pair;
    g.preact = preact ? const_cast<void*>(preact) : UG;
    g.preact_ld = 2 * (int64_t)h;
    g.preact_dense = preact ? 1 : 0;
    g.out = dUG;
    g.ldo = 2 * (int64_t)h;
    g.out2 = H;
    g.ldo2 = h;
    g.status = status;
    s = cuda_status(launch_gemm(g, st));
  }
  if (s == MOE_OK)
    s = grouped_bf16(dUG, prows, w->w_up_gate, (int64_t)E * 2 * h, 2 * h, Lr, 2 * h, poff, tile_off, E, pair, dXp,
                     status, st, 1);
  if (s == MOE_OK)
    s = cuda_status(launch_combine(dXp, scat, nullptr, (int)T, k, Lr, prows, 0, 0.f, nullptr, dx_routed,
                                   capacity ? 1 : 0, status, st));
  // weight gradients, K-grouped over each expert's 64-row tiles, read as stored (MN-major A and B):
  // dW_out from dY's dense rows (a tile's rows past the expert meet H's zero padding rows) and H,
  // dW_up_gate from dUG and the padded routed rows
  if (s == MOE_OK) s = kgrouped_f32(dy, Lr, H, h, b.kpad, k_off, E, dw_out, status, st, offsets, rows);
  if (s == MOE_OK) {
    if (gather_b)
      s = kgrouped_f32(dUG, 2 * h, x_routed, Lr, b.kpad, k_off, E, dw_up_gate, status, st, nullptr, 0, gather_idx,
                       offsets, T);
    else
      s = kgrouped_f32(dUG, 2 * h, xp, Lr, b.kpad, k_off, E, dw_up_gate, status, st);
  }
  return s;
}

// Whole-layer backward: the buffers it keeps between its steps, then room for the steps' own
// workspaces (the largest of them).
struct LayerBwdPlan {
  size_t zc, dz, dy, dwts, dlogits, dxr, dxo, sub, sub_bytes, total;
};

void make_layer_bwd_plan(const moe_config_t* c, int64_t T, LayerBwdPlan* b) {
  const int64_t E = c->num_experts, k = c->top_k, D = c->d_model;
  const bool latent = c->latent_dim > 0;
  const int64_t Lr = latent ? c->latent_dim : D;
  const int64_t rows = c->capacity_factor > 0.f ? E * capacity_of(c, T) : T * k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  b->zc = take(latent ? (size_t)T * Lr * 2 : 0);
  b->dz = take(latent ? (size_t)T * Lr * 2 : 0);
  b->dy = take((size_t)rows * Lr * 2);
  b->dwts = take((size_t)T * k * 4);
  b->dlogits = take((size_t)T * E * 4);
  b->dxr = take((size_t)T * Lr * 2);
  b->dxo = take((size_t)T * D * 2);
  size_t sub = 0;
  moe_backward_workspace_size(c, T, &sub);
  b->sub = o;
  b->sub_bytes = sub;
  b->total = o + align256(sub);
}

int moe_layer_backward_workspace_size(const moe_config_t* c, int64_t T, size_t* bytes) {
  int s = check_config(c);
  if (s != MOE_OK) return s;
  if (T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
  LayerBwdPlan b;
  make_layer_bwd_plan(c, T, &b);
  *bytes = b.total;
  return MOE_OK;
}

int moe_layer_backward(const moe_config_t* c, const moe_weights_t* w, const void* x, int64_t T, const void* fwd_ws,
                       size_t fwd_ws_bytes, const void* preact, const float* logits, const void* dout, void* dx,
                       const moe_grads_t* g, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Plan p;
  int s = check_call(c, T, const_cast<void*>(fwd_ws), fwd_ws_bytes, &p);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  const bool latent = p.latent;
  if (!w || !x || !logits || !dout || !dx || !g || !g->dw_router || !g->dw_up_gate || !g->dw_out)
    return MOE_ERR_INVALID_ARG;
  if (latent && (!g->dw_down_latent || !g->dw_up_latent)) return MOE_ERR_INVALID_ARG;
  LayerBwdPlan b;
  make_layer_bwd_plan(c, T, &b);
  if (!ws || ((uintptr_t)ws & 255) || ws_bytes < b.total) return MOE_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  void* fws = const_cast<void*>(fwd_ws);
  const int32_t* idx = at<int32_t>(fws, p.idx);
  const float* wts = at<float>(fws, p.wts);
  const int32_t* offsets = at<int32_t>(fws, p.offsets);
  const int32_t* gather = at<int32_t>(fws, p.gather);
  const int32_t* scatter = at<int32_t>(fws, p.scatter);
  const void* Y = at<void>(fws, p.Y);
  const void* xr = latent ? at<void>(fws, p.xr) : x;
  void* sub = at<void>(ws, b.sub);
  void* dy = at<void>(ws, b.dy);
  float* dwts = at<float>(ws, b.dwts);
  void* dxr = at<void>(ws, b.dxr);
  void* dxo = at<void>(ws, b.dxo);
  // d z: through the up-projection and its norm (z recomputed by the combine), or dout itself
  const void* dz = dout;
  if (latent) {
    void* zc = at<void>(ws, b.zc);
    s = cuda_status(launch_combine(Y, scatter, wts, (int)T, p.k, p.L, (int)p.rows, 0, 0.f, nullptr, zc,
                                   p.capacity ? 1 : 0, status, st));
    if (s == MOE_OK)
      s = moe_latent_restore_backward(c, w, zc, T, dout, at<void>(ws, b.dz), g->dw_up_latent, g->drms_weight, sub,
                                      b.sub_bytes, stream);
    dz = at<void>(ws, b.dz);
  }
  if (s == MOE_OK) s = moe_combine_backward(c, dz, Y, scatter, gather, wts, T, dy, dwts, stream);
  if (s == MOE_OK)
    s = moe_grouped_swiglu_backward_preact(c, w, xr, gather, offsets, scatter, T, dy, preact, dxr, g->dw_up_gate,
                                           g->dw_out, sub, b.sub_bytes, stream);
  // the layer input's gradient: the experts' path (through the down-projection when latent) plus
  // the router's
  const void* dx_experts = dxr;
  if (s == MOE_OK && latent) {
    s = moe_latent_down_backward(c, w, x, T, dxr, dx, g->dw_down_latent, sub, b.sub_bytes, stream);
    dx_experts = dx;
  }
  if (s == MOE_OK)
    s = moe_router_backward(c, w, x, T, logits, idx, dwts, at<float>(ws, b.dlogits), dxo, g->dw_router, g->db_router,
                            sub, b.sub_bytes, stream);
  if (s == MOE_OK) s = cuda_status(launch_add_bf16(dx_experts, dxo, T * (int64_t)p.D, dx, st));
  return s;
}

int moe_check_wait_timeout(int32_t limit_ms, int32_t* waited_ms, moe_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 2000 || !waited_ms) return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  int before = 0;
  if (cudaMemcpyAsync(&before, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (before != MOE_OK) return before;   // an earlier error stays reported, untouched
  int res[2] = {0, 0};
  if (launch_wait_timeout_check((uint64_t)limit_ms * 1000000ull, status, res, st) != cudaSuccess) return MOE_ERR_CUDA;
  int after = 0;
  if (cudaMemcpyAsync(&after, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  *waited_ms = res[1];
  return (res[0] == 1 && after == MOE_ERR_TIMEOUT) ? MOE_OK : MOE_ERR_CUDA;
}

int moe_quantize_mxfp8(const void* x, int64_t rows, int32_t cols, void* codes, void* scales, int32_t scale_ld,
                       moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 32 || scale_ld < cols / 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mx_e4m3(x, rows, cols, codes, scales, scale_ld, (cudaStream_t)stream));
}

int moe_get_status(moe_stream_t stream, int32_t* device_status, int clear) {
  if (!device_status) return MOE_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return MOE_ERR_NO_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  int host = 0;
  if (cudaMemcpyAsync(&host, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (clear) {
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = host;
  return MOE_OK;
}

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BOUNDS: return "index out of range on the device";
    case MOE_ERR_NO_DEVICE: return "no CUDA device";
    default: return "unknown status";
  }
}

}  // extern "C"
