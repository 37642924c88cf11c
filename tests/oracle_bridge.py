"""Test-side glue: turn a drawn workload into the oracle's config and float64 weights."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_ref as ref
from token_routing_expert_gb300.workloads import GATING_NAMES, WorkloadSpec


def f64(t):
    if t is None:
        return None
    return t.to(torch.float64).numpy()


def oracle_config(spec: WorkloadSpec) -> ref.OracleConfig:
    return ref.OracleConfig(
        d_model=spec.d_model, num_experts=spec.num_experts, top_k=spec.top_k,
        hidden_size=spec.hidden_size, latent_dim=spec.latent_dim,
        up_proj_norm=spec.up_proj_norm, rms_eps=spec.rms_eps,
        gating=GATING_NAMES[spec.gating],
        sigmoid_stability_epsilon=spec.sigmoid_stability_epsilon,
        normalize_expert_weights=spec.normalize_expert_weights,
        restore_weight_scale=spec.restore_weight_scale,
        expert_weight_scale=spec.expert_weight_scale,
        original_top_k=spec.original_top_k,
        router_bias=spec.skew, has_score_bias=spec.score_bias_std > 0)


def oracle_weights(spec: WorkloadSpec, inp) -> ref.OracleWeights:
    h = spec.hidden_size
    w_ug, w_o = inp["w_up_gate"], inp["w_out"]

    def expert(e):
        ug = f64(w_ug[e])
        return ug[:h], ug[h:], f64(w_o[e])

    return ref.OracleWeights(
        w_router=f64(inp["w_router"]), expert=expert, b_router=f64(inp["b_router"]),
        score_bias=f64(inp["score_bias"]), w_down_latent=f64(inp["w_down"]),
        w_up_latent=f64(inp["w_up_latent"]))


def near_tie_tokens(keys: np.ndarray, k: int, gap: float = 1e-5) -> np.ndarray:
    """Tokens whose top-(k+1) sorted keys have a consecutive gap below ``gap``.

    Such a token's choice or order may legitimately differ between float32
    and float64 evaluation.
    """
    T, E = keys.shape
    m = min(k + 1, E)
    part = -np.sort(-keys, axis=1)[:, :m]
    if m < 2:
        return np.zeros(T, bool)
    return (np.diff(-part, axis=1) < gap).any(axis=1)


# Parity bars (layer output against float64; top-k near-tie rule).
REL_L2 = 1e-2
MAX_ABS = 3e-2
TIE_GAP = 1e-5
TIE_FRAC = 1e-3


def output_scale(spec) -> float:
    """The factor by which the configured weight scalings multiply the layer output.

    restore_weight_scale (x top_k), expert_weight_scale (x s) and original_top_k
    (x sqrt(k0 / k)) multiply every routing weight, hence the combined output,
    by one constant; the absolute error scales with it.  The max-abs bar is
    applied to the output divided by this factor (for top_k = 8 the factor is
    2^3, an exact scaling in both implementations).
    """
    s = 1.0
    if spec.restore_weight_scale:
        s *= spec.top_k
    if spec.expert_weight_scale:
        s *= abs(spec.expert_weight_scale)
    if spec.original_top_k and spec.original_top_k != spec.top_k:
        s *= (spec.original_top_k / spec.top_k) ** 0.5
    return s


def assert_close_layer(got, want, what, scale: float = 1.0):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(got - want).max() if got.size else 0.0
    assert rel <= REL_L2 and mx / scale <= MAX_ABS, (
        f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e} (output scale {scale:g}: {mx / scale:.3e})")
    return rel, mx


def check_topk(gpu_idx, oracle_keys, oracle_idx, k):
    """Top-k indices equal except near-ties, which must stay under 0.1% of the tokens."""
    mism = (gpu_idx != oracle_idx).any(axis=1)
    ties = near_tie_tokens(oracle_keys, k, TIE_GAP)
    bad = mism & ~ties
    assert not bad.any(), f"{bad.sum()} top-k mismatches that are not near-ties, e.g. token {np.nonzero(bad)[0][:5]}"
    assert mism.sum() <= TIE_FRAC * len(mism), f"{mism.sum()} near-tie mismatches > 0.1%"
    return mism


def capacity_factor_f32(spec) -> float:
    """The capacity factor as the library sees it (a float32 field)."""
    return float(np.float32(spec.capacity_factor))
