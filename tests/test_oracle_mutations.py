"""Planted mistakes in the oracle (on the CPU) must each fail one of its pins.

Each case swaps one oracle function for a plausible wrong version and runs
the pin that should catch it.
"""
import numpy as np
import pytest

from oracle import moe_ref as ref
from tests import test_oracle_layer as L
from tests import test_oracle_permute as P
from tests import test_oracle_balance as B
from tests import test_oracle_router as R
from tests import test_oracle_fp8 as F

_ORIG_PERMUTE = ref.permute
_ORIG_GATE_SCORES = ref.gate_scores
_ORIG_TOP_K = ref.top_k
_ORIG_QUANTIZE_MX = ref.quantize_mx_e4m3


def _silu_dropped(g):
    return g


def _swapped_swiglu(rows, w_up, w_gate, w_out):
    u = rows @ w_gate.T
    g = rows @ w_up.T
    return (ref.silu(g) * u) @ w_out.T


def _weights_from_keys(logits, scores, idx, gating):
    # wrong: gathers the bias-shifted keys instead of the scores
    keys = ref.selection_keys(logits, scores, gating, _weights_from_keys.bias)
    return np.take_along_axis(keys, idx, axis=1)


_weights_from_keys.bias = np.array([1.0, 0.0, 0.0, -1.0])


def _topk_full_softmax(logits, scores, idx, gating):
    # wrong: topk_softmax weights taken from the softmax over all experts
    return np.take_along_axis(scores, idx, axis=1)


def _topk_high_index_wins(keys, k):
    # wrong: equal keys resolved in favour of the higher expert index
    E = keys.shape[1]
    rev = _ORIG_TOP_K(keys[:, ::-1], k)
    return (E - 1) - rev


def _unstable_permute(idx, E):
    # wrong: each expert's bin in reverse flat order
    p = _ORIG_PERMUTE(idx, E)
    g = p.gather_token.copy()
    s = np.empty_like(p.scatter_pos)
    flat = np.asarray(idx).reshape(-1)
    for e in range(E):
        lo, hi = p.offsets[e], p.offsets[e + 1]
        g[lo:hi] = p.gather_token[lo:hi][::-1]
    for f in range(flat.size):
        e = flat[f]
        lo, hi = p.offsets[e], p.offsets[e + 1]
        s[f] = lo + hi - 1 - p.scatter_pos[f]
    return ref.Permutation(p.counts, p.offsets, g, s)


def _rms_sum(z, eps, gamma=None):
    z = np.asarray(z, np.float64)
    return z / np.sqrt((z * z).sum(axis=-1, keepdims=True) + eps)


def _scale_then_normalise(w, cfg):
    w = np.array(w, np.float64)
    if cfg.restore_weight_scale:
        w = w * cfg.top_k
    p = cfg.normalize_expert_weights
    if p:
        w = w / (np.abs(w) ** p).sum(axis=1, keepdims=True) ** (1.0 / p)
    return w


def _no_epsilon_scores(logits, gating, sigmoid_eps=0.0):
    # wrong: the stability epsilon is dropped
    return _ORIG_GATE_SCORES(logits, gating, 0.0)


def _bias_update_wrong_sign(score_bias, accum, bias_gamma):
    # wrong: pushes over-loaded experts up
    a = np.asarray(accum, np.float64)
    return np.asarray(score_bias, np.float64) + bias_gamma * np.sign(a - a.mean()), np.zeros_like(accum)


def _imbalance_min_over_mean(counts):
    # wrong: minimum instead of maximum
    c = np.asarray(counts, np.float64)
    return float(c.min() / c.mean()) if c.mean() > 0 else float("nan")


def _mx_offset_seven(x):
    # wrong: scale exponent floor(log2 amax) - 7 (amax / scale in [128, 256))
    x = np.asarray(x, np.float64)
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // ref.MX_BLOCK, ref.MX_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    e = np.zeros(amax.shape, np.int64)
    nz = amax > 0
    e[nz] = np.floor(np.log2(amax[nz])).astype(np.int64) - 7 + 127
    e = np.clip(e, 0, 254)
    codes = ref.round_e4m3(blocks / np.ldexp(1.0, e - 127)[:, :, None]).reshape(rows, cols)
    return codes, e


def _mx_one_scale_per_row(x):
    # wrong: the whole row shares the scale of its largest block
    codes, e = _ORIG_QUANTIZE_MX(x)
    e_row = np.repeat(e.max(axis=1, keepdims=True), e.shape[1], axis=1)
    x = np.asarray(x, np.float64)
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // ref.MX_BLOCK, ref.MX_BLOCK)
    codes = ref.round_e4m3(blocks / np.ldexp(1.0, e_row - 127)[:, :, None]).reshape(rows, cols)
    return codes, e_row


def _mx_experts_h_unquantised(cfg, x_routed, perm, expert):
    # wrong: H goes to the down projection without its MXFP8 round trip
    xd = ref.dequantize_mx(*ref.quantize_mx_e4m3(np.asarray(x_routed, np.float64)))
    y = np.zeros((perm.gather_token.size, x_routed.shape[1]))
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        if hi == lo:
            continue
        wu, wg, wo = (ref.dequantize_mx(*ref.quantize_mx_e4m3(np.asarray(a, np.float64))) for a in expert(e))
        rows = xd[perm.gather_token[lo:hi]]
        y[lo:hi] = ref.round_bf16(ref.silu(rows @ wg.T) * (rows @ wu.T)) @ wo.T
    return y


_ORIG_QUANTIZE_ROWWISE = ref.quantize_rowwise_e4m3
_ORIG_LAYER_FP8 = ref.layer_forward_fp8


def _rowwise_per_column(x):
    # wrong: one scale per column (amax over the rows) instead of one per row; returned as
    # dequantised values with unit row scales so that callers multiply them back unchanged
    x32 = np.asarray(x, np.float32)
    amax = np.abs(x32).max(axis=0) if x32.size else np.zeros(x32.shape[1], np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = ref.round_e4m3((x32 / scale[None, :]).astype(np.float32))
    return codes * scale.astype(np.float64)[None, :], np.ones(x32.shape[0], np.float32)


def _fp8_experts_h_unquantised(cfg, x_routed, perm, expert):
    # wrong: H goes to the down projection without its rowwise e4m3 round trip
    xq, xs = ref.quantize_rowwise_e4m3(np.asarray(x_routed, np.float64))
    xd = xq * xs.astype(np.float64)[:, None]
    y = np.zeros((perm.gather_token.size, x_routed.shape[1]))
    for e in range(cfg.num_experts):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        if hi == lo:
            continue
        wu, wg, wo = ref.quantize_expert_fp8(*(np.asarray(a, np.float64) for a in expert(e)))
        rows = xd[perm.gather_token[lo:hi]]
        y[lo:hi] = ref.round_bf16(ref.silu(rows @ wg.T) * (rows @ wu.T)) @ wo.T
    return y


def _fp8_layer_unrounded_latent_input(cfg, x, wts, forced_idx=None):
    # wrong: the latent projection's output reaches the quantiser without its bf16 rounding
    x = np.asarray(x, np.float64)
    x_routed = ref.prepare_routed_input(cfg, x, wts.w_down_latent)
    r = ref.route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    perm = ref.permute(r.idx, cfg.num_experts)
    y = ref.expert_outputs_fp8(cfg, x_routed, perm, wts.expert)
    z = ref.combine(y, perm.scatter_pos, r.weights)
    return ref.restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)


def _mx_layer_unrounded_latent_input(cfg, x, wts, forced_idx=None):
    # wrong: the latent projection's output reaches the MX quantiser without its bf16 rounding
    x = np.asarray(x, np.float64)
    x_routed = ref.prepare_routed_input(cfg, x, wts.w_down_latent)
    r = ref.route(cfg, x, wts.w_router, wts.b_router, wts.score_bias, forced_idx)
    perm = ref.permute(r.idx, cfg.num_experts)
    y = ref.expert_outputs_mxfp8(cfg, x_routed, perm, wts.expert)
    z = ref.combine(y, perm.scatter_pos, r.weights)
    return ref.restore_routed_output(cfg, z, wts.w_up_latent, wts.rms_weight)


CASES = [
    ("score_bias_update", _bias_update_wrong_sign, lambda: B.test_score_bias_update_hand_values()),
    ("load_imbalance", _imbalance_min_over_mean, lambda: B.test_load_imbalance_hand_values()),
    ("silu", _silu_dropped, lambda: L.test_single_expert_is_dense_swiglu_mlp()),
    ("swiglu_mlp", _swapped_swiglu, lambda: L.test_single_expert_is_dense_swiglu_mlp()),
    ("routing_weights", _weights_from_keys, lambda: R.test_sigmoid_bias_for_selection_only()),
    ("routing_weights", _topk_full_softmax,
     lambda: R.test_topk_softmax_selects_on_biased_logits_and_weights_on_selected_logits()),
    ("top_k", _topk_high_index_wins, lambda: R.test_topk_ties_lower_index_first(6, 3)),
    ("permute", _unstable_permute, lambda: P.test_permutation_matches_stable_argsort(64, 8, 16)),
    ("rms_norm", _rms_sum, lambda: L.test_rms_norm_matches_library()),
    ("normalise_and_scale", _scale_then_normalise, lambda: R.test_normalisation_and_scalings(ref.GATING_SIGMOID)),
    ("gate_scores", _no_epsilon_scores, lambda: R.test_sigmoid_scores_match_library_plus_epsilon()),
    ("quantize_mx_e4m3", _mx_offset_seven, lambda: F.test_mx_quantiser_closed_forms()),
    ("quantize_mx_e4m3", _mx_one_scale_per_row, lambda: F.test_mx_quantiser_saturates_and_bounds_the_error()),
    ("expert_outputs_mxfp8", _mx_experts_h_unquantised, lambda: F.test_mx_experts_hand_computed_h_rounding()),
    ("quantize_rowwise_e4m3", _rowwise_per_column,
     lambda: F.test_rowwise_expert_weights_round_trip_when_representable()),
    ("quantize_rowwise_e4m3", _rowwise_per_column, lambda: F.test_fp8_experts_hand_computed_h_tie()),
    ("expert_outputs_fp8", _fp8_experts_h_unquantised, lambda: F.test_fp8_experts_hand_computed_h_tie()),
    ("layer_forward_fp8", _fp8_layer_unrounded_latent_input, lambda: F.test_fp8_latent_layer_hand_computed()),
    ("layer_forward_mxfp8", _mx_layer_unrounded_latent_input, lambda: F.test_mx_latent_layer_hand_computed()),
]


@pytest.mark.parametrize("name,bad,pin", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(ref, name, bad)
    with pytest.raises(AssertionError):
        pin()
