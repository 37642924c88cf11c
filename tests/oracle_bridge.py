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


def half_ulp_bf16(v) -> np.ndarray:
    """Half a bf16 unit in the last place at each value: the largest error of rounding v to bf16.

    bf16 keeps 8 significant bits, so for 2^e <= |v| < 2^(e+1) one step is 2^(e-7).  A bf16 output
    can be no closer to the exact value than this, whatever the computation before the rounding."""
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(a)            # a = m * 2^e, m in [0.5, 1): the leading bit is 2^(e-1)
    return np.where(a > 0, np.ldexp(1.0, e - 9), 0.0)


def assert_close_layer(got, want, what):
    """A bf16 result against the float64 oracle: rel-L2 <= 1e-2 over all values, and every value
    within 3e-2 of the oracle beyond the half-ulp that its own bf16 rounding may cost.

    The raw max-abs is reported beside it.  Above |4| one bf16 step exceeds 3e-2 (0.03125 in
    [4, 8), 0.0625 in [8, 16)), so a raw 3e-2 against either the exact or the bf16-rounded oracle
    would reject correctly rounded outputs; the half-ulp term removes exactly that rounding and
    nothing else."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    d = np.abs(got - want)
    mx = d.max() if got.size else 0.0
    excess = (d - half_ulp_bf16(want)).max() if got.size else 0.0
    assert rel <= REL_L2 and excess <= MAX_ABS, (
        f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e} beyond the bf16 half-ulp={excess:.3e} "
        f"(vs the bf16-rounded oracle: {np.abs(got - ref.round_bf16(want)).max() if got.size else 0.0:.3e})")
    return rel, mx


def assert_close_relative(got, want, what, bound=MAX_ABS):
    """rel-L2 <= 1e-2 and every value within ``bound`` times the largest |want|."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    mx = np.abs(got - want).max() / max(np.abs(want).max(), 1e-30) if got.size else 0.0
    assert rel <= REL_L2 and mx <= bound, f"{what}: rel_l2={rel:.3e} max_abs / max|want| = {mx:.3e}"


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


# Rowwise FP8 scales a row by its largest magnitude after bf16 rounding, so a row whose amax sits
# within computation error of a bf16 rounding midpoint can quantise as a whole either way: every
# code of the row shifts.  Like a near-tie in top-k, both results are correct.  The GPU's fp32
# accumulation is within these relative bands of the float64 value (K up to 7168 for the latent
# projection, 2048 for the experts); the bands are generous.
FP8_EPS_X = 2e-5
FP8_EPS_H = 1e-5


def _amax_ambiguous(rows: np.ndarray, eps: float) -> np.ndarray:
    """Per row: does the bf16-rounded row maximum change under a relative perturbation of eps?"""
    a = np.abs(rows)
    lo = ref.round_bf16(a * (1.0 - eps)).max(axis=1)
    hi = ref.round_bf16(a * (1.0 + eps)).max(axis=1)
    return lo != hi


def fp8_ambiguous_tokens(oc: ref.OracleConfig, ow: ref.OracleWeights, x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Tokens (rows of x, with their expert indices idx) whose FP8 layer output can legitimately
    differ as a whole: the bf16 amax of their routed input row, or of one of their SwiGLU rows H,
    is within the computation-error band of a bf16 rounding midpoint."""
    xr = ref.prepare_routed_input(oc, x, ow.w_down_latent)
    flag = _amax_ambiguous(xr, FP8_EPS_X) if oc.is_latent else np.zeros(len(x), bool)
    xq, xs = ref.quantize_rowwise_e4m3(ref.round_bf16(xr) if oc.is_latent else xr)
    xd = xq * xs.astype(np.float64)[:, None]
    for e in np.unique(idx):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        wu, wg, _ = ref.quantize_expert_fp8(*ow.expert(int(e)))
        rows = xd[toks]
        hrows = ref.silu(rows @ wg.T) * (rows @ wu.T)
        flag[toks] |= _amax_ambiguous(hrows, FP8_EPS_H)
    return flag


# A latent layer feeds the quantiser a bf16 row computed by the down-projection: wherever the
# GPU's fp32-accumulated value and the float64 one fall on either side of a bf16 rounding
# midpoint (a few elements per row), the e4m3 code of that element may differ by one step,
# which moves the token's output by about a percent when the element is large.  The bar for
# that path is therefore the FP8 one: rel-L2 1e-2 over the sample and at most half an e4m3 step
# (2^-4 relative) per token.
FP8_TOKEN_REL = 2.0 ** -4


def assert_close_fp8_layer(got, want, amb, what, latent=False, max_ambiguous_frac=0.1):
    """FP8 layer parity.  Non-latent (exact bf16 expert inputs): the layer bar on tokens with no
    ambiguous row amax; ambiguous ones (a whole row may take the neighbouring scale) must stay few
    and within rel-L2 2e-2 each.  Latent: the FP8 bar above."""
    rels = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
    if latent:
        tot = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert tot <= REL_L2, f"{what}: rel_l2={tot:.3e}"
        assert rels.max() <= FP8_TOKEN_REL, f"{what}: token {int(rels.argmax())} rel_l2={rels.max():.3e}"
        return
    assert amb.mean() <= max_ambiguous_frac, f"{what}: {int(amb.sum())} of {len(amb)} tokens ambiguous"
    if (~amb).any():
        assert_close_layer(got[~amb], want[~amb], what + " (unambiguous tokens)")
    for i in np.nonzero(amb)[0]:
        assert rels[i] <= 2e-2, f"{what}: ambiguous token {i} rel_l2={rels[i]:.3e}"
