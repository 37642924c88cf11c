"""Plain, slow CPU float64 oracle of the routed (optionally latent) MoE layer forward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module.  It
shares no code with the CUDA path and imports nothing from the product package.

Source of every definition below: the page "Как устроен Olmo-core 3: обучение
больших MoE-моделей" (sarnas.ru blog), cited as [Olmo-core 3] plus its section
heading.  All arithmetic is numpy float64; bf16 inputs are upcast exactly.

Readings where the page is silent (each is also listed in the design notes):
  * top-k order: descending key, equal keys -> lower expert index first (the
    intent of ``_break_ties`` in [Olmo-core 3, §"Разрешение равенства логитов
    и квантизация"]);
  * order inside an expert group: ascending flat assignment index t*k + j
    (a stable sort; [Olmo-core 3, §"Пересылка токенов между экспертами"] only
    says "sorted");
  * the router reads the layer input x (shape (..., d_model)), not the latent
    projection;
  * combine happens in latent space, then RMSNorm, then one up-projection per
    token ([Olmo-core 3, §"Латентная проекция экспертов"]: the experts' output
    is restored as a whole);
  * RMSNorm: z / sqrt(mean(z^2) + eps) * gamma, eps = 1e-6 and gamma = 1
    unless given ("bias-free" only rules out a bias);
  * SwiGLU: expert up-projection rows [0, h) are "up", rows [h, 2h) are "gate",
    activation = silu(gate) * up ([Olmo-core 3, §"SwiGLU с квантизацией"]
    splits the last dim in half into up and gate);
  * unset router options (p, scales, epsilon, biases) mean "not applied".

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against closed forms, library routines, brute force or invariants.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import numpy as np

GATING_SOFTMAX = 0
GATING_TOPK_SOFTMAX = 1
GATING_SIGMOID = 2


@dataclass
class OracleConfig:
    """Fields of MoEConfig / MoERouterConfigV2 / LatentMoEConfig.

    [Olmo-core 3, §"Как задаётся конфигурация MoE"] (num_experts, hidden_size,
    d_model, top_k), §"Латентная проекция экспертов" (latent_dim, up-proj input
    norm) and §"Маршрутизация: как роутер выбирает экспертов" (gating,
    sigmoid_stability_epsilon, normalize_expert_weights, restore_weight_scale,
    expert_weight_scale, original_top_k, score_bias).
    """

    d_model: int
    num_experts: int
    top_k: int
    hidden_size: int
    latent_dim: int = 0            # 0: no latent MoE (latent_dim = d_model)
    up_proj_norm: bool = True      # latent only: bias-free RMSNorm before up-proj
    rms_eps: float = 1e-6
    gating: int = GATING_SOFTMAX
    sigmoid_stability_epsilon: float = 0.0   # 0: unset
    normalize_expert_weights: float = 0.0    # p; 0: unset
    restore_weight_scale: bool = False
    expert_weight_scale: float = 0.0         # 0: unset
    original_top_k: int = 0                  # 0 or == top_k: unset
    router_bias: bool = False
    has_score_bias: bool = False

    @property
    def is_latent(self) -> bool:
        return self.latent_dim > 0

    @property
    def routed_dim(self) -> int:
        return self.latent_dim if self.latent_dim > 0 else self.d_model


# --------------------------------------------------------------------------
# Parameter counts  [Olmo-core 3, §"Как задаётся конфигурация MoE"]
# --------------------------------------------------------------------------

def up_factor(activation: str = "swiglu") -> int:
    """2 for the gated activations (swiglu, gpt_oss_swiglu), 1 otherwise."""
    return 2 if activation in ("swiglu", "gpt_oss_swiglu") else 1


def router_params(cfg: OracleConfig) -> int:
    """Router: d_model * num_experts weights, plus num_experts if it has a bias."""
    return cfg.d_model * cfg.num_experts + (cfg.num_experts if cfg.router_bias else 0)


def expert_params_each(cfg: OracleConfig, activation: str = "swiglu") -> int:
    """One routed expert: (up_factor + 1) * dim * hidden_size (no expert bias).

    The experts are built with d_model = latent_dim when latent
    ([Olmo-core 3, §"Латентная проекция экспертов"]).
    """
    return (up_factor(activation) + 1) * cfg.routed_dim * cfg.hidden_size


def num_params(cfg: OracleConfig, shared_params: int = 0) -> int:
    """Total = router + 3 * latent_dim * hidden_size * num_experts + shared modules."""
    return router_params(cfg) + 3 * cfg.routed_dim * cfg.hidden_size * cfg.num_experts + shared_params


def num_active_params(cfg: OracleConfig, shared_params: int = 0) -> int:
    """Active = total - all expert params + top_k experts' params."""
    experts_all = 3 * cfg.routed_dim * cfg.hidden_size * cfg.num_experts
    experts_active = 3 * cfg.routed_dim * cfg.hidden_size * cfg.top_k
    return num_params(cfg, shared_params) - experts_all + experts_active


def latent_proj_params(cfg: OracleConfig) -> int:
    """Down (latent_dim x d_model) + up (d_model x latent_dim) projections.

    The page's total does not name them; they are reported separately.
    """
    if not cfg.is_latent:
        return 0
    return 2 * cfg.d_model * cfg.latent_dim


# --------------------------------------------------------------------------
# Router  [Olmo-core 3, §"Маршрутизация: как роутер выбирает экспертов"]
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray, b_router: Optional[np.ndarray] = None) -> np.ndarray:
    """Linear layer with weight (num_experts, d_model): logits (T, num_experts)."""
    logits = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if b_router is not None:
        logits = logits + np.asarray(b_router, np.float64)[None, :]
    return logits


def gate_scores(logits: np.ndarray, gating: int, sigmoid_eps: float = 0.0) -> np.ndarray:
    """softmax / topk_softmax: softmax over the experts axis; sigmoid: sigmoid + epsilon."""
    logits = np.asarray(logits, np.float64)
    if gating in (GATING_SOFTMAX, GATING_TOPK_SOFTMAX):
        shifted = logits - logits.max(axis=-1, keepdims=True)
        ex = np.exp(shifted)
        return ex / ex.sum(axis=-1, keepdims=True)
    if gating == GATING_SIGMOID:
        return 1.0 / (1.0 + np.exp(-logits)) + sigmoid_eps
    raise ValueError(f"unknown gating {gating}")


def selection_keys(logits: np.ndarray, scores: np.ndarray, gating: int,
                   score_bias: Optional[np.ndarray]) -> np.ndarray:
    """What top-k ranks: logits (+score_bias) for topk_softmax, else scores (+score_bias)."""
    base = logits if gating == GATING_TOPK_SOFTMAX else scores
    if score_bias is None:
        return np.array(base, np.float64, copy=True)
    return base + np.asarray(score_bias, np.float64)[None, :]


def top_k(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys per row, descending; equal keys: lower index first.

    k == 1 is an argmax (first maximum), as the page takes ``max`` for one expert.
    """
    keys = np.asarray(keys, np.float64)
    T, E = keys.shape
    if k == 1:
        return np.argmax(keys, axis=1).astype(np.int64)[:, None]
    out = np.empty((T, k), np.int64)
    expert_ids = np.arange(E)
    for t in range(T):
        # primary key: -keys (descending); secondary: expert index (ascending)
        order = np.lexsort((expert_ids, -keys[t]))
        out[t] = order[:k]
    return out


def routing_weights(logits: np.ndarray, scores: np.ndarray, idx: np.ndarray, gating: int) -> np.ndarray:
    """Unbiased weights of the chosen experts.

    topk_softmax: softmax over the selected logits only; otherwise the scores
    gathered at the chosen indices (never the bias-shifted keys).
    """
    if gating == GATING_TOPK_SOFTMAX:
        sel = np.take_along_axis(logits, idx, axis=1)
        sel = sel - sel.max(axis=1, keepdims=True)
        ex = np.exp(sel)
        return ex / ex.sum(axis=1, keepdims=True)
    return np.take_along_axis(scores, idx, axis=1).astype(np.float64)


def normalise_and_scale(w: np.ndarray, cfg: OracleConfig) -> np.ndarray:
    """Divide by the p-norm along the last axis, then the optional scalings in the page's order:
    x top_k (restore_weight_scale), x expert_weight_scale, x (original_top_k / top_k) ** 0.5.
    """
    w = np.array(w, np.float64, copy=True)
    p = cfg.normalize_expert_weights
    if p:
        norm = (np.abs(w) ** p).sum(axis=1, keepdims=True) ** (1.0 / p)
        w = w / norm
    if cfg.restore_weight_scale:
        w = w * cfg.top_k
    if cfg.expert_weight_scale:
        w = w * cfg.expert_weight_scale
    if cfg.original_top_k and cfg.original_top_k != cfg.top_k:
        w = w * math.sqrt(cfg.original_top_k / cfg.top_k)
    return w


@dataclass
class Routing:
    logits: np.ndarray   # (T, E) float64
    scores: np.ndarray   # (T, E) float64
    keys: np.ndarray     # (T, E) float64, what top-k ranked
    idx: np.ndarray      # (T, k) int64
    weights: np.ndarray  # (T, k) float64, after normalisation and scaling


def route(cfg: OracleConfig, x: np.ndarray, w_router: np.ndarray,
          b_router: Optional[np.ndarray] = None, score_bias: Optional[np.ndarray] = None,
          forced_idx: Optional[np.ndarray] = None) -> Routing:
    """The router's forward (inference: no jitter).

    ``forced_idx`` replaces the selection (for tokens whose choice is a
    near-tie); weights are still this oracle's, computed for those indices.
    """
    logits = router_logits(x, w_router, b_router if cfg.router_bias else None)
    scores = gate_scores(logits, cfg.gating, cfg.sigmoid_stability_epsilon)
    keys = selection_keys(logits, scores, cfg.gating, score_bias if cfg.has_score_bias else None)
    idx = top_k(keys, cfg.top_k) if forced_idx is None else np.asarray(forced_idx, np.int64)
    w = routing_weights(logits, scores, idx, cfg.gating)
    w = normalise_and_scale(w, cfg)
    return Routing(logits, scores, keys, idx, w)


# --------------------------------------------------------------------------
# Permutation  [Olmo-core 3, §"Пересылка токенов между экспертами"]
# --------------------------------------------------------------------------

@dataclass
class Permutation:
    counts: np.ndarray        # (E,) tokens per expert (the histogram)
    offsets: np.ndarray       # (E+1,) bins: exclusive cumulative sum of counts
    gather_token: np.ndarray  # (R,) token index of permuted row p
    scatter_pos: np.ndarray   # (R,) permuted row of assignment t*k + j


def permute(idx: np.ndarray, num_experts: int) -> Permutation:
    """Counting sort of the flat assignments t*k + j by expert.

    Histogram, exclusive cumulative sum (the bins), then placement in
    ascending flat order inside each expert's bin.
    """
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.zeros(num_experts, np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(num_experts + 1, np.int64)
    for e in range(num_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:-1].copy()
    gather_token = np.empty(T * k, np.int64)
    scatter_pos = np.empty(T * k, np.int64)
    for f, e in enumerate(flat):
        p = cursor[e]
        cursor[e] += 1
        gather_token[p] = f // k
        scatter_pos[f] = p
    return Permutation(counts, offsets, gather_token, scatter_pos)


# --------------------------------------------------------------------------
# Experts  [Olmo-core 3, §"Вычисления экспертов и точность", §"SwiGLU с квантизацией"]
# --------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_mlp(rows: np.ndarray, w_up: np.ndarray, w_gate: np.ndarray, w_out: np.ndarray) -> np.ndarray:
    """y = W_out (silu(W_gate r) * (W_up r)) for each row r."""
    u = rows @ w_up.T
    g = rows @ w_gate.T
    return (silu(g) * u) @ w_out.T


def rms_norm(z: np.ndarray, eps: float, gamma: Optional[np.ndarray] = None) -> np.ndarray:
    """Bias-free RMSNorm along the last axis."""
    z = np.asarray(z, np.float64)
    inv = 1.0 / np.sqrt((z * z).mean(axis=-1, keepdims=True) + eps)
    out = z * inv
    if gamma is not None:
        out = out * np.asarray(gamma, np.float64)
    return out


ExpertFn = Callable[[int], Sequence[np.ndarray]]


@dataclass
class OracleWeights:
    """Layer weights as float64 (or a per-expert provider for large layers).

    expert(e) -> (w_up (h, L), w_gate (h, L), w_out (L, h)).
    """

    w_router: np.ndarray
    expert: ExpertFn
    b_router: Optional[np.ndarray] = None
    score_bias: Optional[np.ndarray] = None
    w_down_latent: Optional[np.ndarray] = None   # (L, D)
    w_up_latent: Optional[np.ndarray] = None     # (D, L)
    rms_weight: Optional[np.ndarray] = None      # (L,) or None for ones


@dataclass
class LayerResult:
    routing: Routing
    perm: Permutation
    x_routed: np.ndarray  # (T, L) input of the experts
    y: np.ndarray         # (R, L) expert outputs in permuted order
    z: np.ndarray         # (T, L) weighted combine
    out: np.ndarray       # (T, D)


def prepare_routed_input(cfg: OracleConfig, x: np.ndarray, w_down_latent: Optional[np.ndarray]) -> np.ndarray:
    """Latent down-projection (*, d_model) -> (*, latent_dim); identity when not latent."""
    x = np.asarray(x, np.float64)
    if not cfg.is_latent:
        return x
    return x @ np.asarray(w_down_latent, np.float64).T


def expert_outputs(cfg: OracleConfig, x_routed: np.ndarray, perm: Permutation, expert: ExpertFn) -> np.ndarray:
    """y[p] = expert e's SwiGLU MLP of the token in permuted row p, for each bin e."""
    x_routed = np.asarray(x_routed, np.float64)
    y = np.zeros((perm.gather_token.size, x_routed.shape[1]), np.float64)
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        if hi == lo:
            continue
        w_up, w_gate, w_out = (np.asarray(a, np.float64) for a in expert(e))
        y[lo:hi] = swiglu_mlp(x_routed[perm.gather_token[lo:hi]], w_up, w_gate, w_out)
    return y


def combine(y: np.ndarray, scatter_pos: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """z[t] = sum_j weights[t, j] * y[scatter_pos[t*k + j]]: scatter back and weight."""
    y = np.asarray(y, np.float64)
    weights = np.asarray(weights, np.float64)
    T, k = weights.shape
    z = np.zeros((T, y.shape[1]), np.float64)
    for j in range(k):
        z += weights[:, j:j + 1] * y[np.asarray(scatter_pos)[np.arange(T) * k + j]]
    return z


def restore_routed_output(cfg: OracleConfig, z: np.ndarray, w_up_latent: Optional[np.ndarray],
                          rms_weight: Optional[np.ndarray] = None) -> np.ndarray:
    """RMSNorm (if configured), then the up-projection (*, latent_dim) -> (*, d_model); identity when not latent."""
    z = np.asarray(z, np.float64)
    if not cfg.is_latent:
        return z
    n = rms_norm(z, cfg.rms_eps, rms_weight) if cfg.up_proj_norm else z
    return n @ np.asarray(w_up_latent, np.float64).T


def layer_forward(cfg: OracleConfig, x: np.ndarray, wts: OracleWeights,
                  forced_idx: Optional[np.ndarray] = None) -> LayerResult:
    """The MoE layer forward, step by step.

    1. prepare_routed_input: latent down-projection (identity when not latent).
    2. router on the layer input x.
    3. permutation into per-expert bins.
    4. each expert's SwiGLU MLP on its bin.
    5. weighted un-permute / combine.
    6. restore_routed_output: RMSNorm then up-projection (identity when not latent).
    """
    x = np.asarray(x, np.float64)
    x_routed = prepare_routed_input(cfg, x, wts.w_down_latent)
    r = route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    perm = permute(r.idx, cfg.num_experts)
    y = expert_outputs(cfg, x_routed, perm, wts.expert)
    z = combine(y, perm.scatter_pos, r.weights)
    out = restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)
    return LayerResult(r, perm, x_routed, y, z, out)


# --------------------------------------------------------------------------
# Load balancing counters  [Olmo-core 3, §"Счётчики и bias-корректировка"]
# --------------------------------------------------------------------------

def accumulate_counts(accum: np.ndarray, counts: np.ndarray) -> np.ndarray:
    """The per-expert accumulator adds each step's tokens-per-expert histogram."""
    return np.asarray(accum, np.int64) + np.asarray(counts, np.int64)


def load_imbalance(counts: np.ndarray) -> float:
    """Maximum of the per-expert counter divided by its mean (NaN when no token was routed)."""
    c = np.asarray(counts, np.float64)
    mean = c.mean()
    return float(c.max() / mean) if mean > 0 else float("nan")


def score_bias_update(score_bias: np.ndarray, accum: np.ndarray, bias_gamma: float):
    """score_bias += bias_gamma * sign(ideal - actual), ideal = the mean count; then the accumulator is zeroed.

    Returns (new score_bias, zeroed accumulator).
    """
    a = np.asarray(accum, np.float64)
    ideal = a.mean()
    new = np.asarray(score_bias, np.float64) + bias_gamma * np.sign(ideal - a)
    return new, np.zeros_like(np.asarray(accum))


# --------------------------------------------------------------------------
# Expert capacity  [Olmo-core 3, §"Ёмкость эксперта и переполнение"]
# --------------------------------------------------------------------------

def expert_capacity(cfg: OracleConfig, T: int, capacity_factor: float, ep_degree: int = 1) -> int:
    """EP degree x (capacity_factor x ideal inputs per expert, rounded up to a multiple of 8),
    ideal inputs = top_k x local batch / num_experts."""
    ideal = cfg.top_k * T / cfg.num_experts
    local = 8 * math.ceil(capacity_factor * ideal / 8)
    return ep_degree * local


@dataclass
class CapacityPermutation:
    capacity: int
    counts: np.ndarray        # (E,) tokens chosen per expert, before dropping
    kept: np.ndarray          # (E,) min(count, capacity)
    slot_token: np.ndarray    # (E * capacity,) token in slot e*capacity + r; -1 = padding
    scatter_slot: np.ndarray  # (T*k,) slot of assignment t*k + j; -1 = dropped


def permute_with_capacity(idx: np.ndarray, num_experts: int, capacity: int) -> CapacityPermutation:
    """Every expert gets exactly `capacity` slots.  Its assignments fill them in
    ascending flat order; the ones beyond the capacity are dropped, free slots are padding."""
    idx = np.asarray(idx, np.int64)
    flat = idx.reshape(-1)
    E = num_experts
    counts = np.zeros(E, np.int64)
    slot_token = np.full(E * capacity, -1, np.int64)
    scatter_slot = np.full(flat.size, -1, np.int64)
    k = idx.shape[1] if idx.ndim == 2 else 1
    for f, e in enumerate(flat):
        r = counts[e]
        counts[e] += 1
        if r < capacity:
            s = e * capacity + r
            slot_token[s] = f // k
            scatter_slot[f] = s
    return CapacityPermutation(capacity, counts, np.minimum(counts, capacity), slot_token, scatter_slot)


def expert_outputs_capacity(cfg: OracleConfig, x_routed: np.ndarray, perm: CapacityPermutation,
                            expert: ExpertFn) -> np.ndarray:
    """y for every slot; a padding slot holds a zero row, whose SwiGLU output is zero."""
    x_routed = np.asarray(x_routed, np.float64)
    cap = perm.capacity
    y = np.zeros((cfg.num_experts * cap, x_routed.shape[1]), np.float64)
    for e in range(cfg.num_experts):
        n = int(perm.kept[e])
        if n == 0:
            continue
        w_up, w_gate, w_out = (np.asarray(a, np.float64) for a in expert(e))
        y[e * cap:e * cap + n] = swiglu_mlp(x_routed[perm.slot_token[e * cap:e * cap + n]], w_up, w_gate, w_out)
    return y


def combine_capacity(y: np.ndarray, scatter_slot: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """z[t] = sum over the kept assignments j of weights[t, j] * y[slot]; dropped ones add nothing."""
    y = np.asarray(y, np.float64)
    weights = np.asarray(weights, np.float64)
    T, k = weights.shape
    z = np.zeros((T, y.shape[1]), np.float64)
    for t in range(T):
        for j in range(k):
            s = scatter_slot[t * k + j]
            if s >= 0:
                z[t] += weights[t, j] * y[s]
    return z


def layer_forward_capacity(cfg: OracleConfig, x: np.ndarray, wts: OracleWeights, capacity_factor: float,
                           forced_idx: Optional[np.ndarray] = None):
    """The layer forward with capacity-limited experts (dropping at the permutation)."""
    x = np.asarray(x, np.float64)
    x_routed = prepare_routed_input(cfg, x, wts.w_down_latent)
    r = route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    cap = expert_capacity(cfg, x.shape[0], capacity_factor)
    perm = permute_with_capacity(r.idx, cfg.num_experts, cap)
    y = expert_outputs_capacity(cfg, x_routed, perm, wts.expert)
    z = combine_capacity(y, perm.scatter_slot, r.weights)
    out = restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)
    return r, perm, y, z, out


# --------------------------------------------------------------------------
# Backward of the experts and of the combine (training)
# [Olmo-core 3, §"SwiGLU с квантизацией": the SwiGLU backward computes the
#  sigmoid, gate*sigmoid, its derivative and the two gradients in float32]
# --------------------------------------------------------------------------

def silu_grad(g: np.ndarray) -> np.ndarray:
    """d silu / d g = sigmoid(g) * (1 + g * (1 - sigmoid(g)))."""
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def swiglu_mlp_backward(rows: np.ndarray, w_up: np.ndarray, w_gate: np.ndarray, w_out: np.ndarray,
                        dy: np.ndarray):
    """Gradients of y = W_out (silu(W_gate r) * W_up r) for a batch of rows r.

    Returns (d rows, d W_up, d W_gate, d W_out, H) where H = silu(g) * u is the
    activation the W_out gradient contracts with.
    """
    u = rows @ w_up.T
    g = rows @ w_gate.T
    h = silu(g) * u
    dh = dy @ w_out
    du = dh * silu(g)
    dg = dh * u * silu_grad(g)
    d_rows = du @ w_up + dg @ w_gate
    return d_rows, du.T @ rows, dg.T @ rows, dy.T @ h, h


def combine_backward(dz: np.ndarray, y: np.ndarray, scatter_pos: np.ndarray, weights: np.ndarray):
    """Gradients of z[t] = sum_j w[t, j] y[scatter_pos[t*k + j]]:
    dy[p] = w[t, j] dz[t] for the assignment (t, j) in row p; dw[t, j] = <dz[t], y[p]>."""
    dz = np.asarray(dz, np.float64)
    y = np.asarray(y, np.float64)
    weights = np.asarray(weights, np.float64)
    T, k = weights.shape
    dy = np.zeros_like(y)
    dw = np.zeros((T, k), np.float64)
    for t in range(T):
        for j in range(k):
            p = scatter_pos[t * k + j]
            if p < 0:
                continue
            dy[p] = weights[t, j] * dz[t]
            dw[t, j] = dz[t] @ y[p]
    return dy, dw


def experts_backward(cfg: OracleConfig, x_routed: np.ndarray, perm: Permutation, expert: ExpertFn, dy: np.ndarray):
    """Gradients of the grouped SwiGLU experts (y in permuted order, as expert_outputs).

    Returns (d x_routed (T, L), {e: (dW_up, dW_gate, dW_out)}): a token's input
    gradient sums its k assignments' row gradients.
    """
    x_routed = np.asarray(x_routed, np.float64)
    dy = np.asarray(dy, np.float64)
    dx = np.zeros_like(x_routed)
    grads = {}
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        w_up, w_gate, w_out = (np.asarray(a, np.float64) for a in expert(e))
        if hi == lo:
            grads[e] = (np.zeros_like(w_up), np.zeros_like(w_gate), np.zeros_like(w_out))
            continue
        tokens = perm.gather_token[lo:hi]
        d_rows, dwu, dwg, dwo, _ = swiglu_mlp_backward(x_routed[tokens], w_up, w_gate, w_out, dy[lo:hi])
        np.add.at(dx, tokens, d_rows)
        grads[e] = (dwu, dwg, dwo)
    return dx, grads


def router_backward(cfg: OracleConfig, x: np.ndarray, w_router: np.ndarray, b_router: Optional[np.ndarray],
                    score_bias: Optional[np.ndarray], idx: np.ndarray, dweights: np.ndarray):
    """Gradients of the routing weights for a fixed choice of experts.

    The selection itself is discrete; score_bias only moves the selection and
    gets no gradient.  Returns (dlogits (T, E), dx (T, D), dW_router (E, D),
    db_router (E,)).
    """
    x = np.asarray(x, np.float64)
    idx = np.asarray(idx, np.int64)
    r = route(cfg, x, w_router, b_router, score_bias, forced_idx=idx)
    T, k = idx.shape
    E = cfg.num_experts
    scale = 1.0
    if cfg.restore_weight_scale:
        scale *= cfg.top_k
    if cfg.expert_weight_scale:
        scale *= cfg.expert_weight_scale
    if cfg.original_top_k and cfg.original_top_k != cfg.top_k:
        scale *= math.sqrt(cfg.original_top_k / cfg.top_k)
    d_norm = np.asarray(dweights, np.float64) * scale
    w_raw = routing_weights(r.logits, r.scores, idx, cfg.gating)
    p = cfg.normalize_expert_weights
    if p:
        n = ((np.abs(w_raw) ** p).sum(axis=1, keepdims=True)) ** (1.0 / p)
        dn_dw = np.sign(w_raw) * np.abs(w_raw) ** (p - 1) * n ** (1 - p)
        d_raw = d_norm / n - (d_norm * w_raw).sum(axis=1, keepdims=True) / n ** 2 * dn_dw
    else:
        d_raw = d_norm
    dlogits = np.zeros((T, E), np.float64)
    rows = np.arange(T)[:, None]
    if cfg.gating == GATING_SOFTMAX:
        ds = np.zeros((T, E), np.float64)
        np.add.at(ds, (np.broadcast_to(rows, idx.shape), idx), d_raw)
        s = r.scores
        dlogits = s * (ds - (ds * s).sum(axis=1, keepdims=True))
    elif cfg.gating == GATING_TOPK_SOFTMAX:
        dsel = w_raw * (d_raw - (d_raw * w_raw).sum(axis=1, keepdims=True))
        np.add.at(dlogits, (np.broadcast_to(rows, idx.shape), idx), dsel)
    else:
        sig = 1.0 / (1.0 + np.exp(-np.take_along_axis(r.logits, idx, axis=1)))
        np.add.at(dlogits, (np.broadcast_to(rows, idx.shape), idx), d_raw * sig * (1.0 - sig))
    w_router = np.asarray(w_router, np.float64)
    return dlogits, dlogits @ w_router, dlogits.T @ x, dlogits.sum(axis=0)



# --------------------------------------------------------------------------
# Backward of the latent projections  [Olmo-core 3, §"Латентная проекция
# экспертов": prepare_routed_input (down-projection) and restore_routed_output
# (RMSNorm, then the up-projection)]
# The derivative of the forward as defined above; nothing on the page differs.
# --------------------------------------------------------------------------

def rms_norm_backward(z: np.ndarray, dn: np.ndarray, eps: float, gamma: Optional[np.ndarray] = None):
    """Gradients of n = z r gamma, r = 1 / sqrt(mean(z^2) + eps), along the last axis:
    dz = r (gamma dn) - z r^3 mean(z gamma dn), dgamma = sum over rows of dn z r."""
    z = np.asarray(z, np.float64)
    dn = np.asarray(dn, np.float64)
    g = np.ones(z.shape[-1]) if gamma is None else np.asarray(gamma, np.float64)
    r = 1.0 / np.sqrt((z * z).mean(axis=-1, keepdims=True) + eps)
    gdn = dn * g
    dz = r * gdn - z * r ** 3 * (z * gdn).mean(axis=-1, keepdims=True)
    dgamma = (dn * z * r).reshape(-1, z.shape[-1]).sum(axis=0)
    return dz, dgamma


def restore_routed_output_backward(cfg: OracleConfig, z: np.ndarray, w_up_latent: np.ndarray,
                                   dout: np.ndarray, rms_weight: Optional[np.ndarray] = None):
    """Gradients of out = W_up n (n = RMSNorm(z) gamma, or z without the norm):
    (dz, dW_up, dgamma; dgamma is None without the norm)."""
    z = np.asarray(z, np.float64)
    dout = np.asarray(dout, np.float64)
    w_up_latent = np.asarray(w_up_latent, np.float64)
    n = rms_norm(z, cfg.rms_eps, rms_weight) if cfg.up_proj_norm else z
    dn = dout @ w_up_latent
    dw_up = dout.T @ n
    if not cfg.up_proj_norm:
        return dn, dw_up, None
    dz, dgamma = rms_norm_backward(z, dn, cfg.rms_eps, rms_weight)
    return dz, dw_up, dgamma


def prepare_routed_input_backward(x: np.ndarray, w_down_latent: np.ndarray, dx_routed: np.ndarray):
    """Gradients of x_routed = x W_down^T: (dx, dW_down)."""
    x = np.asarray(x, np.float64)
    dx_routed = np.asarray(dx_routed, np.float64)
    return dx_routed @ np.asarray(w_down_latent, np.float64), dx_routed.T @ x

# --------------------------------------------------------------------------
# Rowwise FP8 experts  [Olmo-core 3, §"Rowwise FP8 и MXFP8": pre-quantised
# expert weights, quantised activations, the experts run on FP8 operands]
# Reading: one float32 scale per row (amax / 448, the largest e4m3 value), the
# row divided by it in float32 and rounded to e4m3 (nearest, ties to even,
# saturating at 448); the GEMMs accumulate exactly and apply both rows' scales.
# What is quantised: [Olmo-core 3, §"SwiGLU с квантизацией"] has the SwiGLU
# forward produce the activation and, from it, its quantised representations,
# so H is the activation in the input dtype (bf16) before it is quantised; and
# the experts' input is the bf16 tensor the layer hands them (in the latent
# case the dense down-projection's bf16 output).
# --------------------------------------------------------------------------

def _e4m3_positive_values() -> np.ndarray:
    """The non-negative finite e4m3 values in code order 0x00..0x7E (increasing)."""
    vals = []
    for code in range(0x7F):
        e, m = (code >> 3) & 0xF, code & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, np.float64)


_E4M3 = _e4m3_positive_values()


def round_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value, ties to the even code, magnitudes above 448 saturate to 448."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 1, len(_E4M3) - 1)
    lo = hi - 1
    dlo, dhi = a - _E4M3[lo], _E4M3[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    out = np.where(pick_hi, _E4M3[hi], _E4M3[lo])
    out = np.where(a == _E4M3[hi], _E4M3[hi], out)
    return np.sign(v) * out


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even) via float32."""
    f = np.asarray(v, np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize_rowwise_e4m3(x: np.ndarray):
    """(codes as float64 values, float32 scales): scale = amax / 448 in float32 (1 for a zero row),
    code = e4m3(x / scale) with the division in float32."""
    x32 = np.asarray(x, np.float32)
    amax = np.abs(x32).max(axis=1) if x32.size else np.zeros(x32.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = (x32 / scale[:, None]).astype(np.float32)
    return round_e4m3(y), scale


def quantize_expert_fp8(w_up: np.ndarray, w_gate: np.ndarray, w_out: np.ndarray):
    """Rowwise-quantised expert weights, returned dequantised (code * scale) in float64."""
    out = []
    for w in (w_up, w_gate, w_out):
        q, s = quantize_rowwise_e4m3(w)
        out.append(q * s.astype(np.float64)[:, None])
    return tuple(out)


def expert_outputs_fp8(cfg: OracleConfig, x_routed: np.ndarray, perm: Permutation, expert: ExpertFn) -> np.ndarray:
    """Experts on rowwise FP8 operands: x rows and weight rows quantised, H rounded to bf16
    and quantised again before the down projection."""
    xq, xs = quantize_rowwise_e4m3(np.asarray(x_routed, np.float64))
    xd = xq * xs.astype(np.float64)[:, None]
    y = np.zeros((perm.gather_token.size, x_routed.shape[1]), np.float64)
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        if hi == lo:
            continue
        wu, wg, wo = quantize_expert_fp8(*(np.asarray(a, np.float64) for a in expert(e)))
        rows = xd[perm.gather_token[lo:hi]]
        h = round_bf16(silu(rows @ wg.T) * (rows @ wu.T))
        hq, hs = quantize_rowwise_e4m3(h)
        y[lo:hi] = (hq * hs.astype(np.float64)[:, None]) @ wo.T
    return y


def layer_forward_fp8(cfg: OracleConfig, x: np.ndarray, wts: OracleWeights,
                      forced_idx: Optional[np.ndarray] = None) -> np.ndarray:
    """The layer forward with the experts on rowwise FP8 operands (bf16 x_routed as input)."""
    x = np.asarray(x, np.float64)
    x_routed = prepare_routed_input(cfg, x, wts.w_down_latent)
    if cfg.is_latent:
        x_routed = round_bf16(x_routed)   # the experts' input is stored in bf16
    r = route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    perm = permute(r.idx, cfg.num_experts)
    y = expert_outputs_fp8(cfg, x_routed, perm, wts.expert)
    z = combine(y, perm.scatter_pos, r.weights)
    return restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)


# --------------------------------------------------------------------------
# MXFP8 experts  [Olmo-core 3, §"Rowwise FP8 и MXFP8": the MXFP8 path of the
# experts].  The page names the format only; the reading is the OCP
# microscaling (MX) format: blocks of 32 consecutive values along the
# contraction share one power-of-two scale X = 2^(floor(log2 amax) - 8)
# (8 = the largest e4m3 exponent, 448 = 1.75 * 2^8), stored as its biased
# exponent (E8M0, X = 2^(e - 127)); each value is rounded to e4m3 as v / X
# (exact: X is a power of two), nearest, ties to even, saturating at 448.
# An all-zero block takes e = 0.  The GEMMs accumulate exactly and apply the
# two blocks' scales to each 32-wide partial product.
# --------------------------------------------------------------------------

MX_BLOCK = 32


def quantize_mx_e4m3(x: np.ndarray):
    """(codes as float64 values (rows, cols), scale exponents e (rows, cols / 32) as int):
    x[r, c] ~ code[r, c] * 2^(e[r, c // 32] - 127)."""
    x = np.asarray(x, np.float64)
    rows, cols = x.shape
    assert cols % MX_BLOCK == 0
    blocks = x.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    e = np.zeros(amax.shape, np.int64)
    nz = amax > 0
    e[nz] = np.floor(np.log2(amax[nz])).astype(np.int64) - 8 + 127
    e = np.clip(e, 0, 254)
    scale = np.ldexp(1.0, (e - 127).astype(np.int64))
    codes = round_e4m3(blocks / scale[:, :, None]).reshape(rows, cols)
    return codes, e


def dequantize_mx(codes: np.ndarray, e: np.ndarray) -> np.ndarray:
    rows, cols = codes.shape
    scale = np.ldexp(1.0, (np.asarray(e) - 127).astype(np.int64))
    return (codes.reshape(rows, cols // MX_BLOCK, MX_BLOCK) * scale[:, :, None]).reshape(rows, cols)


def expert_outputs_mxfp8(cfg: OracleConfig, x_routed: np.ndarray, perm: Permutation, expert: ExpertFn) -> np.ndarray:
    """Experts on MXFP8 operands: x rows and weight rows quantised in 32-wide blocks along the
    contraction, H rounded to bf16 and quantised the same way before the down projection."""
    xd = dequantize_mx(*quantize_mx_e4m3(np.asarray(x_routed, np.float64)))
    y = np.zeros((perm.gather_token.size, x_routed.shape[1]), np.float64)
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        if hi == lo:
            continue
        wu, wg, wo = (dequantize_mx(*quantize_mx_e4m3(np.asarray(a, np.float64))) for a in expert(e))
        rows = xd[perm.gather_token[lo:hi]]
        h = round_bf16(silu(rows @ wg.T) * (rows @ wu.T))
        y[lo:hi] = dequantize_mx(*quantize_mx_e4m3(h)) @ wo.T
    return y


def layer_forward_mxfp8(cfg: OracleConfig, x: np.ndarray, wts: OracleWeights,
                        forced_idx: Optional[np.ndarray] = None) -> np.ndarray:
    """The layer forward with the experts on MXFP8 operands (bf16 x_routed as input)."""
    x = np.asarray(x, np.float64)
    x_routed = prepare_routed_input(cfg, x, wts.w_down_latent)
    if cfg.is_latent:
        x_routed = round_bf16(x_routed)   # the experts' input is stored in bf16
    r = route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    perm = permute(r.idx, cfg.num_experts)
    y = expert_outputs_mxfp8(cfg, x_routed, perm, wts.expert)
    z = combine(y, perm.scatter_pos, r.weights)
    return restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)
