/*
 * moe.h — C ABI of the GB300 (sm_103a) routed / latent Mixture-of-Experts
 * layer forward.
 *
 * The operations follow the page "Как устроен Olmo-core 3: обучение больших
 * MoE-моделей" (sarnas.ru); each entry point names the section it implements.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers named "device" point to GPU memory the caller allocated; the
 *    library never allocates, frees or retains them past the call.
 *  - Every array is dense row-major.  Activations and weights are bf16
 *    (passed as void*), logits / routing weights / biases are fp32, indices
 *    are int32.  Weights follow the linear-layer layout (out, in).
 *  - Device work is enqueued on `stream` and is asynchronous; no entry point
 *    synchronises, except moe_get_status and moe_check_wait_timeout.
 *  - `ws` is a caller-owned device workspace of at least
 *    moe_workspace_size(cfg, T) bytes, 256-byte aligned.  Its contents on
 *    entry are irrelevant; entry points overwrite parts of it.
 *  - Return value: MOE_OK, or an error code for bad arguments detected on the
 *    host (nothing is enqueued then) or a launch failure.  Errors found on
 *    the device (an expert index out of range, a pipeline wait that ran out
 *    of time) are recorded in a per-device status word that moe_get_status
 *    reads; a kernel that records an error skips the bad access and returns.
 *  - Calls on one stream are ordered; concurrent calls sharing one workspace
 *    on different streams race.
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same handle as cudaStream_t; NULL = legacy default stream */

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent config */
  MOE_ERR_UNSUPPORTED = 2, /* valid per the page but outside this library's kernels (see moe_validate_config) */
  MOE_ERR_WORKSPACE = 3,   /* ws smaller than moe_workspace_size, or misaligned */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,     /* device: a pipeline wait ran out of time (kernel returned early) */
  MOE_ERR_BOUNDS = 6,      /* device: an index outside its range was met and skipped */
  MOE_ERR_NO_DEVICE = 7    /* no usable sm_103 device for this call */
};

/* moe_config_t.expert_fp8: operands of the experts' GEMMs.  MXFP8 needs d_model (latent_dim when
 * latent) and hidden_size to be multiples of 128, and no kept pre-activations. */
enum {
  MOE_EXPERT_BF16 = 0,
  MOE_EXPERT_FP8_ROWWISE = 1,   /* e4m3 codes with one fp32 scale per row */
  MOE_EXPERT_MXFP8 = 2          /* e4m3 codes with an E8M0 scale per 32 values of a row */
};

/* Gating functions, section "Маршрутизация: как роутер выбирает экспертов". */
typedef enum {
  MOE_GATING_SOFTMAX = 0,      /* scores = softmax(logits) over experts; weights gathered from scores */
  MOE_GATING_TOPK_SOFTMAX = 1, /* select on logits (+score_bias); weights = softmax over selected logits */
  MOE_GATING_SIGMOID = 2       /* scores = sigmoid(logits) + sigmoid_stability_epsilon, per expert */
} moe_gating_t;

/*
 * Layer configuration: the fields of MoEConfig / MoERouterConfigV2 (section
 * "Как задаётся конфигурация MoE") and LatentMoEConfig (section "Латентная
 * проекция экспертов").  A zero in an optional field means "unset".
 */
typedef struct {
  int32_t d_model;     /* D: model width */
  int32_t num_experts; /* E: routed experts */
  int32_t top_k;       /* k: experts per token */
  int32_t hidden_size; /* h: expert MLP width */
  int32_t latent_dim;  /* L: 0 = no latent MoE (experts run in d_model) */
  int32_t up_proj_norm;/* latent only: 1 = bias-free RMSNorm before the up-projection, 0 = none */
  float rms_eps;       /* RMSNorm epsilon (the page gives none; 1e-6 is this library's default) */
  int32_t gating;      /* moe_gating_t */
  float sigmoid_stability_epsilon; /* added to sigmoid scores; 0 = unset */
  float normalize_expert_weights;  /* p of the p-norm dividing the weights; 0 = unset */
  int32_t restore_weight_scale;    /* 1: weights x top_k after normalisation */
  float expert_weight_scale;       /* weights x this; 0 = unset */
  int32_t original_top_k;          /* != top_k and > 0: weights x sqrt(original_top_k / top_k) */
  int32_t router_bias;             /* 1: the router linear layer has a bias (E fp32) */
  int32_t has_score_bias;          /* 1: a score_bias (E fp32) is added for selection only */
  int32_t activation;              /* 0 = swiglu (the only expert activation supported) */
  float capacity_factor;           /* > 0: capacity-limited experts (section "Ёмкость эксперта и
                                      переполнение"); 0 = dropless */
  int32_t expert_fp8;              /* the experts' GEMM operands (section "Rowwise FP8 и MXFP8"):
                                      MOE_EXPERT_BF16, MOE_EXPERT_FP8_ROWWISE or MOE_EXPERT_MXFP8;
                                      the e4m3 modes need the *_fp8 weights below */
} moe_config_t;

/*
 * Device pointers to the layer's weights (bf16 unless noted).
 */
typedef struct {
  const void* w_router;      /* (E, D) */
  const float* b_router;     /* (E) fp32; read only when cfg.router_bias */
  const float* score_bias;   /* (E) fp32; read only when cfg.has_score_bias */
  const void* w_down_latent; /* (L, D); latent only */
  const void* w_up_latent;   /* (D, L); latent only */
  const void* rms_weight;    /* (L) bf16 gain, or NULL for ones; latent with up_proj_norm only */
  const void* w_up_gate;     /* (E, 2h, L'): per expert rows [0,h) = up, rows [h,2h) = gate; L' = L or D */
  const void* w_out;         /* (E, L', h): expert down-projection */
  /* expert_fp8 only: the expert weights quantised row by row with moe_quantize_rowwise_fp8 */
  const void* w_up_gate_fp8;    /* (E, 2h, L') e4m3 codes */
  const float* w_up_gate_scale; /* (E * 2h) fp32 row scales */
  const void* w_out_fp8;        /* (E, L', h) e4m3 codes */
  const float* w_out_scale;     /* (E * L') fp32 row scales */
  /* MOE_EXPERT_MXFP8 only: the *_fp8 codes above are moe_quantize_mxfp8 codes, and these are their
   * E8M0 block scales, scale_ld = (cols / 32 + 15) / 16 * 16 bytes per row */
  const void* w_up_gate_mx_scale; /* (E * 2h, scale_ld(L')) bytes */
  const void* w_out_mx_scale;     /* (E * L', scale_ld(h)) bytes */
} moe_weights_t;

/* ---- host-only functions (no device, no stream) ------------------------- */

/* Checks a configuration.  MOE_ERR_INVALID_ARG: sizes < 1, top_k > num_experts,
 * unknown gating, negative options.  MOE_ERR_UNSUPPORTED: activation != swiglu,
 * d_model / latent_dim / hidden_size not multiples of 64, num_experts > 1024,
 * top_k > 32. */
int moe_validate_config(const moe_config_t* cfg);

/* Total parameters: router (D*E, +E with a router bias) + 3 * L' * h * E
 * (section "Как задаётся конфигурация MoE"; L' = latent_dim or d_model).
 * The latent projections are not part of it; see moe_latent_proj_params. */
int moe_num_params(const moe_config_t* cfg, int64_t* out);

/* Active parameters per token: total - 3*L'*h*E + 3*L'*h*top_k (same section). */
int moe_num_active_params(const moe_config_t* cfg, int64_t* out);

/* Latent down- and up-projection weights: 2 * d_model * latent_dim (+ L with an RMSNorm gain). */
int moe_latent_proj_params(const moe_config_t* cfg, int with_norm_gain, int64_t* out);

/* Expert capacity for T tokens, section "Ёмкость эксперта и переполнение":
 * roundup8(capacity_factor * top_k * T / num_experts) (single device: EP degree 1),
 * computed in double precision; 0 in dropless mode. */
int moe_expert_capacity(const moe_config_t* cfg, int64_t T, int64_t* capacity);

/* Rows of the permuted order: T * top_k (dropless) or num_experts * capacity. */
int moe_permuted_rows(const moe_config_t* cfg, int64_t T, int64_t* rows);

/* Rowwise e4m3 quantisation, section "Rowwise FP8 и MXFP8": for each row of x
 * (rows, cols) bf16, scales[r] = amax / 448 in fp32 (1 for a zero row) and
 * codes[r, c] = e4m3(x[r, c] / scales[r]) (fp32 division, nearest-even,
 * saturating at 448).  cols a multiple of 16.  codes device (rows, cols) bytes;
 * scales device (rows) fp32.  Device call on `stream`. */
int moe_quantize_rowwise_fp8(const void* x, int64_t rows, int32_t cols, void* codes, float* scales,
                             moe_stream_t stream);

/* Workspace bytes that every entry point below needs for T tokens. */
int moe_workspace_size(const moe_config_t* cfg, int64_t T, size_t* bytes);

/* ---- device entry points ------------------------------------------------ */

/*
 * Router, section "Маршрутизация: как роутер выбирает экспертов".
 * logits = x W_router^T (+ b_router) in fp32; scores by the gating function;
 * top-k on the selection key (score, or logit for topk_softmax, + score_bias),
 * descending, equal keys -> lower expert index first (section "Разрешение
 * равенства логитов и квантизация"); weights from the unbiased scores (or a
 * softmax over the selected logits); p-norm normalisation and the scalings
 * restore_weight_scale, expert_weight_scale, original_top_k in that order.
 *   x       device (T, D) bf16
 *   logits  device (T, E) fp32 output, or NULL to keep them in ws only
 *   idx     device (T, k) int32 output: chosen experts, best first
 *   weights device (T, k) fp32 output: routing weights matching idx
 */
int moe_router(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, float* logits,
               int32_t* idx, float* weights, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Token permutation, section "Пересылка токенов между экспертами", and the
 * tokens-per-expert histogram, section "Балансировка нагрузки и
 * вспомогательные штрафы".  Assignment f = t*k + j (token t, choice j) goes
 * to expert idx[f]; rows are grouped by expert, ascending f inside a group.
 *   idx         device (T, k) int32 input, values in [0, E) (others: MOE_ERR_BOUNDS, skipped)
 *   counts      device (E) int32 output: assignments per expert
 *   offsets     device (E+1) int32 output: exclusive prefix sum of counts (the bins)
 *   gather_idx  device (T*k) int32 output: token of permuted row p
 *   scatter_idx device (T*k) int32 output: permuted row of assignment f
 * Capacity mode (cfg.capacity_factor > 0): every expert owns exactly C =
 * moe_expert_capacity slots; its assignments fill them in the same ascending
 * order and the ones beyond C are dropped.  Then offsets[e] = e * C,
 * gather_idx has E * C entries (-1 = padding slot), scatter_idx[f] is the
 * slot or -1 (dropped), and counts still holds the choices before dropping.
 */
int moe_permute(const moe_config_t* cfg, const int32_t* idx, int64_t T, int32_t* counts, int32_t* offsets,
                int32_t* gather_idx, int32_t* scatter_idx, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Grouped SwiGLU experts, sections "Вычисления экспертов и точность" and
 * "SwiGLU с квантизацией": for permuted row p of expert e's group
 * [offsets[e], offsets[e+1]):  u = W_up[e] r, g = W_gate[e] r with
 * r = x_routed[gather_idx[p]];  H = silu(g) * u rounded to bf16;
 * y[p] = W_out[e] H rounded to bf16 (the experts return bf16).
 *   x_routed   device (T, L') bf16: the experts' input (x, or the latent projection)
 *   gather_idx device (rows) int32, offsets device (E+1) int32 (as from moe_permute)
 *   y          device (rows, L') bf16 output, permuted row order
 * rows = moe_permuted_rows(cfg, T); a padding slot (capacity mode) computes a zero row.
 */
int moe_grouped_swiglu(const moe_config_t* cfg, const moe_weights_t* w, const void* x_routed,
                       const int32_t* gather_idx, const int32_t* offsets, int64_t T, void* y, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/*
 * moe_grouped_swiglu that also keeps the pre-activations for the backward
 * (training).  Section "SwiGLU с квантизацией": the SwiGLU function saves its
 * input, the up and gate projections, and its backward works from them; here
 * grouped GEMM 1 stores them from its epilogue next to H, so the backward does
 * not recompute them.
 *   preact device (rows, 2h) bf16 output: row p = [u | g], u = W_up[e] x and
 *   g = W_gate[e] x rounded to bf16 (e4m3 experts: the scaled e4m3 products),
 *   in y's row order; a padding slot (capacity mode) gets a zero row.
 * hidden_size must be a multiple of 32 (else MOE_ERR_UNSUPPORTED).
 */
int moe_grouped_swiglu_preact(const moe_config_t* cfg, const moe_weights_t* w, const void* x_routed,
                              const int32_t* gather_idx, const int32_t* offsets, int64_t T, void* y, void* preact,
                              void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Weighted un-permute / combine, section "Пересылка токенов между экспертами":
 * z[t] = sum_j weights[t, j] * y[scatter_idx[t*k + j]], accumulated in fp32, stored bf16.
 * In capacity mode a dropped assignment (scatter_idx -1) adds nothing.
 *   y device (rows, L') bf16, scatter_idx device (T*k) int32, weights device (T, k) fp32
 *   z device (T, L') bf16 output
 */
int moe_combine(const moe_config_t* cfg, const void* y, const int32_t* scatter_idx, const float* weights,
                int64_t T, void* z, moe_stream_t stream);

/*
 * prepare_routed_input, section "Латентная проекция экспертов":
 * x_routed = x W_down^T (fp32 accumulate, bf16 out).  Latent configs only.
 *   x device (T, D) bf16;  x_routed device (T, L) bf16 output
 */
int moe_latent_down(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, void* x_routed,
                    void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * restore_routed_output, section "Латентная проекция экспертов":
 * n = z / sqrt(mean(z^2) + rms_eps) * gain in fp32, cast to bf16 (the
 * up-projection's dtype), out = n W_up^T.  Without up_proj_norm, n = z.
 * Latent configs only.
 *   z device (T, L) bf16;  out device (T, D) bf16 output
 */
int moe_latent_restore(const moe_config_t* cfg, const moe_weights_t* w, const void* z, int64_t T, void* out,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * The whole layer forward: [latent down] -> router -> permutation -> grouped
 * SwiGLU experts -> weighted combine -> [RMSNorm + latent up].  No host
 * synchronisation: per-expert counts stay on the device.
 *   x device (T, D) bf16;  out device (T, D) bf16 output (may not alias x)
 * Intermediate results stay in ws; moe_workspace_layout reports where.
 */
int moe_layer_forward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, void* out,
                      void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_forward for training: identical results, and the experts'
 * pre-activations are kept in `preact` (device, (rows, 2h) bf16, rows =
 * moe_permuted_rows(cfg, T), as moe_grouped_swiglu_preact writes them) for
 * moe_grouped_swiglu_backward_preact / moe_layer_backward.  preact must not be
 * NULL when T > 0.  logits: device (T, E) fp32 output (x W_router^T + b_router,
 * as moe_router returns them), or NULL.
 */
int moe_layer_forward_preact(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, void* out,
                             void* preact, float* logits, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_forward with stage timing: when stage_events is not NULL it
 * points to 10 cudaEvent_t handles (created by the caller on the current
 * device; a NULL handle is skipped) that are recorded on `stream` at the
 * stage boundaries:
 *   [0] start, [1] after the latent down-projection, [2] after the router
 *   GEMM, [3] after top-k, [4] after the permutation, [5] after the group
 *   tile table (and, for e4m3 experts, the quantisation of x_routed),
 *   [6] after grouped GEMM 1 (SwiGLU, which gathers its input rows),
 *   [7] after grouped GEMM 2,
 *   [8] after the combine (+ RMSNorm), [9] after the latent up-projection.
 * Stages that a configuration does not have record at the same point as the
 * previous boundary.  Results are identical to moe_layer_forward.
 */
int moe_layer_forward_staged(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, void* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream, void* const* stage_events);

/* Host only: number of kernels one moe_layer_forward launches for T tokens on
 * the current device (the split-K choices depend on its SM count). */
int moe_layer_forward_launches(const moe_config_t* cfg, int64_t T, int32_t* n);

/*
 * The layer forward over n_batches batches that live in HOST memory, with the
 * copies overlapped.  The page has no counterpart: this is a library
 * convenience for callers whose tokens arrive in host memory (a serving front
 * end, a data loader) and who want the host <-> device traffic hidden behind
 * the compute instead of paying it between batches.
 *
 *   x_host[b]    host (T, d_model) bf16 inputs, b < n_batches (pinned memory
 *                lets the copies run asynchronously; pageable memory works but
 *                each copy then blocks the host)
 *   out_host[b]  host (T, d_model) bf16 outputs
 *   ws           device workspace of moe_host_workspace_size(cfg, T) bytes:
 *                the layer's workspace followed by two input and two output
 *                staging buffers
 *
 * Batch b is copied in on an internal copy stream while batch b-1 computes on
 * `stream`, and its output is copied out on a second internal stream while
 * batch b+1 computes.  Everything is ordered after the work already on
 * `stream`, and the call returns once it is all enqueued: out_host is complete
 * when `stream` is (synchronise it before reading).  The internal streams and
 * events are created on the first call on a device and reused, so calls on one
 * device from several host threads at once race with each other.  Host
 * buffers must stay valid until `stream` completes.  Errors as for
 * moe_layer_forward; MOE_ERR_WORKSPACE when ws is smaller than
 * moe_host_workspace_size.
 */
int moe_host_workspace_size(const moe_config_t* cfg, int64_t T, size_t* bytes);
int moe_layer_forward_host_batches(const moe_config_t* cfg, const moe_weights_t* w, const void* const* x_host,
                                   void* const* out_host, int32_t n_batches, int64_t T, void* ws, size_t ws_bytes,
                                   moe_stream_t stream);

/*
 * Backward of the weighted combine and of the grouped SwiGLU experts (training).
 * The page's SwiGLU backward (section "SwiGLU с квантизацией"): split into up
 * and gate, sigmoid, gate * sigmoid, its derivative and the two gradients in
 * fp32, stored back in bf16.  rows = moe_permuted_rows(cfg, T).
 *
 * moe_combine_backward: for each assignment (t, j) with row p:
 *   dy[p] = weights[t, j] * dz[t] (bf16) and dweights[t, j] = <dz[t], y[p]> (fp32);
 *   dropped assignments (capacity mode) get dweights 0; padding rows of dy are zeroed.
 *   dz device (T, L') bf16; y device (rows, L') bf16 (the forward's expert outputs);
 *   scatter_idx (T*k), gather_idx (rows, capacity mode only, else may be NULL),
 *   weights (T, k) fp32; dy device (rows, L') bf16 out; dweights device (T, k) fp32 out.
 *
 * moe_grouped_swiglu_backward: given the forward's inputs and dy (rows, L'):
 *   dx_routed (T, L') bf16 out: each token's input gradient, summed over its rows;
 *   dw_up_gate (E, 2h, L') fp32 out and dw_out (E, L', h) fp32 out: weight
 *   gradients (an expert without rows gets zeros).  Pre-activations are
 *   recomputed; ws must hold moe_backward_workspace_size(cfg, T) bytes.
 *
 * moe_grouped_swiglu_backward_preact: the same from the forward's saved
 *   pre-activations (preact device (rows, 2h) bf16, as moe_grouped_swiglu_preact
 *   or moe_layer_forward_preact wrote them; NULL: recomputed), which saves the
 *   recomputation GEMM (4 rows L' h FLOPs).
 */
int moe_backward_workspace_size(const moe_config_t* cfg, int64_t T, size_t* bytes);

/*
 * Router backward for the forward's choice of experts (section "Маршрутизация:
 * как роутер выбирает экспертов"; the selection is discrete, score_bias only
 * moves it and gets no gradient).  The routing-weight gradient is taken back
 * through the scalings, the p-norm and the gating function to the logits, then
 * through the linear layer:
 *   x (T, D) bf16; logits (T, E) fp32 as moe_router returned them (with bias);
 *   idx (T, k); dweights (T, k) fp32;
 *   dlogits (T, E) fp32 out; dx (T, D) bf16 out (the router's share of the
 *   input gradient); dw_router (E, D) fp32 out; db_router (E) fp32 out, or NULL
 *   (written only with a router bias).  ws: moe_backward_workspace_size bytes.
 */
int moe_router_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, const float* logits,
                        const int32_t* idx, const float* dweights, float* dlogits, void* dx, float* dw_router,
                        float* db_router, void* ws, size_t ws_bytes, moe_stream_t stream);
int moe_combine_backward(const moe_config_t* cfg, const void* dz, const void* y, const int32_t* scatter_idx,
                         const int32_t* gather_idx, const float* weights, int64_t T, void* dy, float* dweights,
                         moe_stream_t stream);
int moe_grouped_swiglu_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x_routed,
                                const int32_t* gather_idx, const int32_t* offsets, const int32_t* scatter_idx,
                                int64_t T, const void* dy, void* dx_routed, float* dw_up_gate, float* dw_out,
                                void* ws, size_t ws_bytes, moe_stream_t stream);
int moe_grouped_swiglu_backward_preact(const moe_config_t* cfg, const moe_weights_t* w, const void* x_routed,
                                       const int32_t* gather_idx, const int32_t* offsets, const int32_t* scatter_idx,
                                       int64_t T, const void* dy, const void* preact, void* dx_routed,
                                       float* dw_up_gate, float* dw_out, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/*
 * Backward of the latent projections (training; latent configs only), section
 * "Латентная проекция экспертов": the derivative of restore_routed_output
 * (bias-free RMSNorm with gain gamma, then the up-projection) and of
 * prepare_routed_input (the down-projection).  ws: moe_backward_workspace_size
 * bytes.
 *
 * moe_latent_restore_backward: from z (the combine's output, device (T, L)
 *   bf16) and dout (device (T, D) bf16): n = RMSNorm(z) gamma recomputed as the
 *   forward does (bf16; n = z without up_proj_norm), dn = dout W_up (bf16),
 *   dW_up = dout^T n (device (D, L) fp32 out), and with the norm
 *   dz = r gamma dn - z r^3 mean(z gamma dn), r = 1 / sqrt(mean(z^2) + eps)
 *   (device (T, L) bf16 out) and dgamma = sum over tokens of dn z r
 *   (drms_weight, device (L) fp32 out, or NULL to skip); without the norm dz = dn.
 * moe_latent_down_backward: from x (device (T, D) bf16) and dx_routed (device
 *   (T, L) bf16, e.g. from moe_grouped_swiglu_backward): dx = dx_routed W_down
 *   (device (T, D) bf16 out; the router's share of the input gradient is
 *   separate, moe_router_backward) and dW_down = dx_routed^T x (device (L, D)
 *   fp32 out).
 * Weight gradients are fp32 and contract over the tokens in one pass (no
 * atomics: the same inputs give the same bits).
 */
int moe_latent_restore_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* z, int64_t T,
                                const void* dout, void* dz, float* dw_up, float* drms_weight, void* ws,
                                size_t ws_bytes, moe_stream_t stream);
int moe_latent_down_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T,
                             const void* dx_routed, void* dx, float* dw_down, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/*
 * The whole layer's backward (training), after moe_layer_forward_preact on the
 * same x and weights: every step's derivative, in order
 *   [latent: z recomputed by the combine, moe_latent_restore_backward] ->
 *   moe_combine_backward -> moe_grouped_swiglu_backward_preact ->
 *   [latent: moe_latent_down_backward] -> moe_router_backward,
 * and dx = the experts' share (through the down-projection when latent) plus
 * the router's, summed in fp32 and stored bf16.  score_bias gets no gradient.
 *   fwd_ws / fwd_ws_bytes: the forward's workspace, unchanged since; its
 *     intermediates (moe_workspace_layout) are read, not written.
 *   preact: the forward's kept pre-activations (NULL: recomputed);
 *   logits: the forward's logits output (device (T, E) fp32, required);
 *   dout device (T, D) bf16: the gradient of the layer output;
 *   dx device (T, D) bf16 out;
 *   g: the weight gradients (device fp32 outputs, shapes as the weights):
 *     dw_router, db_router (NULL: skipped; written only with a router bias),
 *     dw_up_gate, dw_out, and when latent dw_down_latent, dw_up_latent and
 *     drms_weight (NULL: skipped; written only with up_proj_norm).
 *   ws: moe_layer_backward_workspace_size(cfg, T) bytes, 256-byte aligned.
 */
typedef struct {
  float* dw_router;        /* (E, D) */
  float* db_router;        /* (E) or NULL */
  float* dw_up_gate;       /* (E, 2h, L') */
  float* dw_out;           /* (E, L', h) */
  float* dw_down_latent;   /* (L, D), latent */
  float* dw_up_latent;     /* (D, L), latent */
  float* drms_weight;      /* (L) or NULL, latent with up_proj_norm */
} moe_grads_t;

int moe_layer_backward_workspace_size(const moe_config_t* cfg, int64_t T, size_t* bytes);
int moe_layer_backward(const moe_config_t* cfg, const moe_weights_t* w, const void* x, int64_t T, const void* fwd_ws,
                       size_t fwd_ws_bytes, const void* preact, const float* logits, const void* dout, void* dx,
                       const moe_grads_t* g, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Load-balancing counters, section "Счётчики и bias-корректировка" (run between
 * training steps or batches; E <= 1024, one small kernel each).
 *
 * moe_accumulate_counts: accum[e] += counts[e] (counts as from moe_permute).
 *   counts device (E) int32; accum device (E) int64, in / out.
 * moe_load_imbalance: *imbalance = max(counts) / mean(counts), NaN when no token
 *   was routed.  counts device (E), int32 or int64 (counts_are_int64 = 1);
 *   imbalance device float scalar.
 * moe_score_bias_update: ideal = mean(accum); score_bias[e] += bias_gamma *
 *   sign(ideal - accum[e]) (the sign decided exactly in integers); then accum
 *   is zeroed.  accum device (E) int64 in / out; score_bias device (E) fp32 in / out.
 */
int moe_accumulate_counts(const int32_t* counts, int32_t num_experts, int64_t* accum, moe_stream_t stream);
int moe_load_imbalance(const void* counts, int32_t counts_are_int64, int32_t num_experts, float* imbalance,
                       moe_stream_t stream);
int moe_score_bias_update(int64_t* accum, int32_t num_experts, float bias_gamma, float* score_bias,
                          moe_stream_t stream);

/* Byte offsets in ws of the layer forward's intermediates, for inspection:
 * [0] router GEMM output (split-K partial logits without the router bias),
 * [1] idx (T,k) int32, [2] weights (T,k) fp32,
 * [3] counts (E), [4] offsets (E+1), [5] gather_idx (T*k), [6] scatter_idx (T*k),
 * [7] x_routed (T,L) bf16 (latent only, else -1), [8] y (T*k, L') bf16,
 * [9] z or normalised z (T, L') bf16 (latent only, else -1). */
int moe_workspace_layout(const moe_config_t* cfg, int64_t T, int64_t offsets_out[10]);

/* Whether moe_layer_forward keeps the experts' rows y (offset [8] above) in fp32 instead of bf16
 * for this configuration: *is_fp32 = 1 when the layer is not latent, its experts are bf16, and
 * its routing weights can add up to more than one per token (sigmoid gating without a p-norm,
 * a p-norm with p > 1, restore_weight_scale, expert_weight_scale or original_top_k).  The
 * combine multiplies y's rounding error by up to that sum, and bf16 y would then put more error
 * into the bf16 output than the output's own rounding.  The page's experts return bf16
 * (section "Вычисления экспертов и точность"); this is a deviation toward more precision.
 * moe_layer_forward_preact (the training forward) always keeps y in bf16, which the backward
 * reads; the workspace reserves 4 bytes per value of y whenever *is_fp32 is 1. */
int moe_layer_expert_rows_fp32(const moe_config_t* cfg, int32_t* is_fp32);

/*
 * moe_permute without a workspace: for callers that may not allocate device
 * memory at all.  The page has no counterpart; this is a library convenience.
 * Such callers include serving loops that hand every byte of device memory to
 * their own pool at start-up (cudaMalloc later would fail, or block the device
 * while it synchronises), and plug-in hosts that give a library only its
 * input and output buffers.
 *
 * Same arguments, results and device-side checks as moe_permute, minus ws.
 * The histogram scratch lives in one 2 MiB array of static device memory,
 * which every GPU that loads this library keeps until the process exits.
 * Limit: ceil(T * top_k / 4096) * num_experts <= 524288 (for 896 experts,
 * T * top_k up to about 2.39 million); larger calls, and capacity-mode
 * configurations, return MOE_ERR_UNSUPPORTED and enqueue nothing.  Within the
 * limit it splits the assignments into moe_permute's chunks when their
 * histograms fit the array, else into chunks of 4096.
 * The first call on each device looks up the array's device address (a
 * runtime query, no allocation); make that first call before any stream
 * capture.  The call allocates and frees nothing.
 * All calls share the one array and it keeps the last call's contents (each
 * call overwrites every entry it reads, so no clearing is needed): calls that
 * can overlap on the GPU -- different streams, or different host threads --
 * race on it and must be ordered by the caller.
 */
int moe_permute_noalloc(const moe_config_t* cfg, const int32_t* idx, int64_t T, int32_t* counts, int32_t* offsets,
                        int32_t* gather_idx, int32_t* scatter_idx, moe_stream_t stream);

/*
 * MXFP8 quantisation (section "Rowwise FP8 и MXFP8", read as the OCP microscaling
 * format): each block of 32 consecutive values of a row shares the scale
 * 2^(e - 127), e = floor(log2 amax) - 8 + 127 clamped to [0, 254] (0 for an
 * all-zero block), stored as the byte e (E8M0); codes[r, c] = e4m3(x[r, c] /
 * 2^(e - 127)), nearest-even, saturating at +-448.
 *   x device (rows, cols) bf16, cols a multiple of 32; codes device (rows, cols)
 *   bytes out; scales device (rows, scale_ld) bytes out, cols / 32 used per row.
 */
int moe_quantize_mxfp8(const void* x, int64_t rows, int32_t cols, void* codes, void* scales, int32_t scale_ld,
                       moe_stream_t stream);

/* Synchronises `stream`, then returns (and clears, if `clear`) the device
 * status word of the current device in *device_status. */
int moe_get_status(moe_stream_t stream, int32_t* device_status, int clear);

/*
 * Health check of the device-side failure path (host function; synchronises
 * the stream).  Every pipelined kernel waits on mbarriers with a bound: after
 * 2 s it records MOE_ERR_TIMEOUT in the status word, raises its CTA's abort flag
 * and returns instead of hanging.  This runs that same wait on a barrier nothing
 * completes, for limit_ms (1..2000) milliseconds, reads the status word back and
 * clears it again.  Returns MOE_OK when the wait gave up after the limit and
 * reported MOE_ERR_TIMEOUT (*waited_ms = how long it waited), MOE_ERR_CUDA if
 * not, or the status word's earlier error, left untouched.
 */
int moe_check_wait_timeout(int32_t limit_ms, int32_t* waited_ms, moe_stream_t stream);

/* Static, human-readable name of a status code. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
